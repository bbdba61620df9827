"""tcgen05 forward (bf16) against the fp64 oracle, through the C ABI."""

import numpy as np
import pytest
import torch

from oracle import attention as A
import long_sequence_exact_gb300 as lsx
from long_sequence_exact_gb300.inputs import WORKLOADS, make_inputs, random_tensor
from helpers import TOL_LSE_BF16, TOL_O_BF16, check_close, check_lse, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def qkv(b, hq, hkv, lq, lk, d, seed, amp=1.0):
    q = random_tensor((b, hq, lq, d), seed, amp, device=DEV)
    k = random_tensor((b, hkv, lk, d), seed + 1, amp, device=DEV)
    v = random_tensor((b, hkv, lk, d), seed + 2, 1.0, device=DEV)
    return q, k, v


CASES = [
    # B, Hq, Hkv, Lq, Lk, D, q_off, kv_off, causal
    (1, 2, 2, 256, 256, 128, 0, 0, True),
    (1, 2, 2, 256, 256, 128, 0, 0, False),
    (1, 2, 2, 256, 256, 64, 0, 0, True),
    (2, 4, 2, 200, 333, 128, 0, 0, False),      # ragged tails, GQA
    (1, 2, 2, 384, 384, 64, 0, 0, True),        # odd number of 128-row tiles
    (1, 2, 2, 300, 500, 64, 200, 0, True),      # causal with offsets
    (1, 3, 1, 130, 700, 128, 1000, 600, True),  # offsets, GQA 3:1
    (1, 2, 2, 128, 256, 128, 0, 64, True),      # first 64 rows see no key
    (1, 1, 1, 1000, 1000, 128, 0, 0, True),     # several items per CTA
    (1, 2, 2, 1, 4096, 128, 4095, 0, True),     # one query row
    (2, 8, 8, 512, 2048, 128, 1536, 0, True),   # a diagonal chunk pair
    (2, 16, 4, 1900, 1900, 64, 0, 0, True),     # d=64: items per CTA > 1, odd tile count
    (2, 32, 8, 1024, 1024, 64, 0, 128, True),   # d=64: pair 0's first tile sees no key
]


@pytest.mark.parametrize("case", CASES)
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("v_copy", [True, False], ids=["v_transposed", "v_as_stored"])
def test_chunk_fwd_matches_oracle(case, out_dtype, v_copy):
    b, hq, hkv, lq, lk, d, q_off, kv_off, causal = case
    q, k, v = qkv(b, hq, hkv, lq, lk, d, seed=11 + lq + lk)
    o, lse = lsx.chunk_fwd(q, k, v, q_off, kv_off, causal, out_dtype=out_dtype,
                           use_workspace=v_copy)
    torch.cuda.synchronize()
    assert lsx.sync_status() == 0
    o_ref, lse_ref = A.attn_fwd(f64(q), f64(k), f64(v), q_off, kv_off, causal)
    check_lse(f64(lse), lse_ref, TOL_LSE_BF16)
    check_close(f64(o), o_ref, TOL_O_BF16)


def test_chunk_fwd_explicit_scale_and_large_scores():
    q, k, v = qkv(1, 2, 2, 256, 512, 128, seed=5, amp=3.0)
    o, lse = lsx.chunk_fwd(q, k, v, 0, 0, False, scale=0.3, out_dtype=torch.float32)
    o_ref, lse_ref = A.attn_fwd(f64(q), f64(k), f64(v), 0, 0, False, 0.3)
    check_lse(f64(lse), lse_ref, TOL_LSE_BF16)
    check_close(f64(o), o_ref, TOL_O_BF16)


def test_accumulate_merges_chunk_pairs_in_ring_order():
    # one query chunk of 512 rows against key chunks 1 then 0 (own chunk first)
    n, c = 1024, 512
    q, k, v = qkv(1, 4, 4, n, n, 128, seed=77)
    qc = q[:, :, c:]
    o = torch.empty((1, 4, c, 128), dtype=torch.float32, device=DEV)
    lse = torch.empty((1, 4, c), dtype=torch.float32, device=DEV)
    lsx.chunk_fwd(qc, k[:, :, c:], v[:, :, c:], c, c, True, out=o, lse=lse)
    lsx.chunk_fwd(qc, k[:, :, :c], v[:, :, :c], c, 0, True, out=o, lse=lse, accumulate=True)
    o_ref, lse_ref = A.attn_fwd(f64(q), f64(k), f64(v), 0, 0, True, rows=np.arange(c, n))
    check_lse(f64(lse), lse_ref, TOL_LSE_BF16)
    check_close(f64(o), o_ref, TOL_O_BF16)


def test_chunked_fwd_whole_sequence():
    n = 2048
    q, k, v = qkv(1, 4, 4, n, n, 128, seed=91, amp=0.5)
    o, lse = lsx.chunked_fwd(q, k, v, chunk_len=512, causal=True)
    o_ref, lse_ref = A.attn_fwd(f64(q), f64(k), f64(v), 0, 0, True)
    check_lse(f64(lse), lse_ref, TOL_LSE_BF16)
    check_close(f64(o), o_ref, TOL_O_BF16)


def test_strided_views_are_honoured():
    # q/k/v as head-interleaved views of a [B, N, H, D] buffer
    b, n, h, d = 1, 384, 4, 128
    base = random_tensor((b, n, 3 * h, d), 3, device=DEV)
    q = base[:, :, :h].transpose(1, 2)
    k = base[:, :, h:2 * h].transpose(1, 2)
    v = base[:, :, 2 * h:].transpose(1, 2)
    o, lse = lsx.chunk_fwd(q, k, v, 0, 0, True)
    o_ref, lse_ref = A.attn_fwd(f64(q), f64(k), f64(v), 0, 0, True)
    check_lse(f64(lse), lse_ref, TOL_LSE_BF16)
    check_close(f64(o), o_ref, TOL_O_BF16)


def test_forward_is_bit_deterministic():
    q, k, v = qkv(1, 8, 8, 1024, 1024, 128, seed=4)
    o1, l1 = lsx.chunk_fwd(q, k, v, 0, 0, True)
    o2, l2 = lsx.chunk_fwd(q, k, v, 0, 0, True)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_empty_key_chunk_gives_identity():
    q = random_tensor((1, 2, 128, 128), 1, device=DEV)
    k = torch.empty((1, 2, 0, 128), dtype=torch.bfloat16, device=DEV)
    o, lse = lsx.chunk_fwd(q, k, k, 0, 0, False, out_dtype=torch.float32)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))


def test_v_layouts_give_the_same_result():
    q, k, v = qkv(2, 4, 2, 700, 900, 128, seed=8)
    a = lsx.chunk_fwd(q, k, v, 200, 0, True, out_dtype=torch.float32, use_workspace=True)
    b = lsx.chunk_fwd(q, k, v, 200, 0, True, out_dtype=torch.float32, use_workspace=False)
    assert float((a[0] - b[0]).abs().max()) <= 1e-5
    assert float((a[1] - b[1]).abs().max()) <= 1e-5


@pytest.mark.parametrize("partial_dtype", [torch.float32, torch.bfloat16])
def test_heavy_tailed_d64_chunk_partials_merged(partial_dtype):
    # The non-causal d = 64 workload's values at N = 4096, computed as 4 x 4
    # chunk pairs: each query chunk visits its key chunks (own first, then
    # the rest), and each new partial is merged into the running one by the
    # forward's fused LSE merge.  Heavy keys (x 8) land in some chunks only,
    # so the running maximum jumps by tens of units between partials: the
    # merge weights span e^-100 .. 1.
    w = WORKLOADS["noncausal_64k_heavytail"].with_(B=1, Hq=2, Hkv=2, N=4096)
    x = make_inputs(w, device=DEV, with_grad=False)
    q, k, v = x["q"], x["k"], x["v"]
    c, nc = 1024, 4
    o = torch.empty(q.shape, dtype=partial_dtype, device=DEV)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=DEV)
    for qc in range(nc):
        qs = slice(qc * c, (qc + 1) * c)
        order = [qc] + [kc for kc in range(nc) if kc != qc]
        for step, kc in enumerate(order):
            ks = slice(kc * c, (kc + 1) * c)
            lsx.chunk_fwd(q[:, :, qs], k[:, :, ks], v[:, :, ks], qc * c, kc * c, False,
                          out=o[:, :, qs], lse=lse[:, :, qs], accumulate=step > 0)
    torch.cuda.synchronize()
    assert lsx.sync_status() == 0
    o_ref, lse_ref = A.attn_fwd(f64(q), f64(k), f64(v), 0, 0, False)
    assert np.max(lse_ref) > 100.0
    check_lse(f64(lse), lse_ref, TOL_LSE_BF16)
    check_close(f64(o), o_ref, TOL_O_BF16)
