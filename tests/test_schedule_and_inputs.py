"""Host logic: the longest-first snake schedule keeps SM-level idle time small
(the single-GPU analogue of DistFlashAttn's load-balancing claim: worker idle
time falls from about half to asymptotically zero), and the seeded input
generators are deterministic and shaped as the workloads say."""

import pytest
import torch

import long_sequence_exact_gb300 as lsx
from long_sequence_exact_gb300.inputs import WORKLOADS, make_inputs


@pytest.fixture(scope="module", autouse=True)
def _built():
    from long_sequence_exact_gb300 import build
    build.build()


@pytest.mark.parametrize("n,workers", [(131072, 152), (32768, 152), (8192, 152), (131072, 148)])
def test_causal_schedule_is_balanced(n, workers):
    makespan, ideal, total = lsx.schedule_stats(1, 32, n, 4096, True, workers)
    assert total == 32 * sum((2 * p + 1) + (2 * p + 2) for p in range(n // 256))
    idle = 1.0 - ideal / makespan
    assert idle < 0.03, f"idle fraction {idle:.3f}"


def test_naive_round_robin_would_be_unbalanced():
    # contrast: contiguous blocks of query tiles per worker (no longest-first
    # dealing) leave most workers idle for a large part of the causal run
    n, h, workers = 131072, 32, 152
    n_pairs = n // 256
    costs = [(2 * p + 1) + (2 * p + 2) for p in range(n_pairs)] * h
    per = -(-len(costs) // workers)
    loads = [sum(costs[i * per:(i + 1) * per]) for i in range(workers)]
    naive_idle = 1.0 - (sum(costs) / workers) / max(loads)
    makespan, ideal, _ = lsx.schedule_stats(1, h, n, 4096, True, workers)
    assert naive_idle > 0.3
    assert 1.0 - ideal / makespan < naive_idle / 10


def test_noncausal_schedule_is_even():
    makespan, ideal, total = lsx.schedule_stats(2, 16, 65536, 4096, False, 152)
    assert total == 2 * 16 * (65536 // 256) * 2 * (65536 // 128)
    assert makespan - ideal <= 2 * (65536 // 128)


def test_generators_are_deterministic_and_shaped():
    w = WORKLOADS["tiny_fp32_causal"]
    a = make_inputs(w)
    b = make_inputs(w)
    for key in ("q", "k", "v", "d_o"):
        assert torch.equal(a[key], b[key])
    assert a["q"].shape == (1, 2, 256, 64) and a["q"].dtype == torch.float32


def test_heavy_tail_rows_are_scaled_by_eight():
    w = WORKLOADS["noncausal_64k_heavytail"].with_(N=2048, B=1, Hq=2, Hkv=2)
    x = make_inputs(w)
    rows = x["heavy_rows"]
    assert rows.shape == (1, 2, int(0.01 * 2048))
    k = x["k"].float()
    for h in range(2):
        heavy = k[0, h, rows[0, h]].abs().mean()
        mask = torch.ones(2048, dtype=torch.bool)
        mask[rows[0, h]] = False
        normal = k[0, h, mask].abs().mean()
        assert 6.0 < float(heavy / normal) < 10.0
    assert x["v"].abs().max() <= 1.0


def test_decode_workload_has_one_query():
    w = WORKLOADS["decode_gqa_1m"].with_(N=4096, B=2)
    x = make_inputs(w, with_grad=False)
    assert x["q"].shape == (2, 32, 1, 128) and x["k"].shape == (2, 8, 4096, 128)
