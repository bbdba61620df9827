"""The device-side record of the balanced causal schedule (lsx_trace_enable):
every persistent tensor-core launch writes one record, every work item is
run by exactly one CTA, and each CTA's times are ordered."""

import pytest
import torch

import bench
import long_sequence_exact_gb300 as lsx
from long_sequence_exact_gb300 import _lib
from long_sequence_exact_gb300.inputs import random_tensor

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("deterministic", [False, True], ids=["fused", "owner_dq"])
def test_trace_records_every_item_once(deterministic):
    # (32 heads: 512 query pairs, enough for the forward not to split rows)
    b, h, n, d = 1, 32, 4096, 128
    q, k, v, d_o = (random_tensor((b, h, n, d), 70 + i, 0.5, device=DEV) for i in range(4))
    lib = _lib.load()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    buf = torch.zeros(1 << 15, dtype=torch.int64, device=DEV)
    lsx.set_deterministic(deterministic)
    try:
        _lib.check(lib.lsx_trace_enable(buf.data_ptr(), buf.numel() * 8), "trace")
        o, lse = lsx.chunked_fwd(q, k, v, 1024, causal=True)
        lsx.chunked_bwd(q, k, v, o, lse, d_o, 1024, causal=True)
        torch.cuda.synchronize()
        used = lib.lsx_trace_used() // 8
    finally:
        lib.lsx_trace_enable(None, 0)
        lsx.set_deterministic(False)
    assert lsx.sync_status() == 0
    words = buf[:used].cpu().tolist()
    recs = bench.parse_trace(words)
    want = ["fwd_tc", "bwd_dkdv_tc", "bwd_dq_tc"] if deterministic else ["fwd_tc", "bwd_fused_tc"]
    assert [r["kernel"] for r in recs] == want
    # items: forward = query-tile pairs x heads, backward = key (or query) tiles x heads
    items = {"fwd_tc": h * (n // 256), "bwd_fused_tc": h * (n // 128),
             "bwd_dkdv_tc": h * (n // 128), "bwd_dq_tc": h * (n // 128)}
    i = 0
    for r in recs:
        assert r["items"] == items[r["kernel"]]
        assert r["ctas"] == min(r["items"], sms)
        assert r["items_run"] == r["items"]
        assert 0.0 <= r["idle_fraction"] < 1.0
        g = r["ctas"]
        for c in range(g):
            start, end = words[i + 3 + 3 * c], words[i + 4 + 3 * c]
            assert 0 < start <= end
        i += 3 + 3 * g
    assert i == used


def test_trace_off_writes_nothing():
    q, k, v = (random_tensor((1, 2, 512, 128), 80 + i, 0.5, device=DEV) for i in range(3))
    lib = _lib.load()
    buf = torch.full((4096,), -1, dtype=torch.int64, device=DEV)
    _lib.check(lib.lsx_trace_enable(buf.data_ptr(), 8 * 2), "trace")  # too small for a record
    try:
        lsx.chunked_fwd(q, k, v, 512, causal=True)
        torch.cuda.synchronize()
        assert lib.lsx_trace_used() == 0
    finally:
        lib.lsx_trace_enable(None, 0)
    lsx.chunked_fwd(q, k, v, 512, causal=True)
    torch.cuda.synchronize()
    assert lsx.sync_status() == 0
    assert bool((buf == -1).all())
