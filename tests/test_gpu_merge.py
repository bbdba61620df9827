"""attn_merge / attn_tree_merge / fp32 path / decode against the oracle."""

import math

import numpy as np
import pytest
import torch

from oracle import attention as A
import long_sequence_exact_gb300 as lsx
from long_sequence_exact_gb300.inputs import make_inputs, random_tensor, WORKLOADS
from helpers import (TOL_FP32, TOL_LSE_BF16, TOL_O_BF16, check_close, check_lse, f64,
                     rel_fro)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def partial(shape, seed, dtype=torch.float32, empty_rows=(), lse_amp=20.0):
    o = random_tensor(shape, seed, dtype=dtype, device=DEV)
    lse = random_tensor(shape[:-1], seed + 1000, lse_amp, dtype=torch.float32, device=DEV)
    for r in empty_rows:
        lse[..., r] = -math.inf
        o[..., r, :] = 0
    return o, lse


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dt", [torch.float32, torch.bfloat16])
def test_merge_matches_oracle(d, dt):
    shape = (2, 3, 257, d)
    oa, la = partial(shape, 1, dt, empty_rows=(0, 5))
    ob, lb = partial(shape, 2, dt, empty_rows=(0, 7))
    o, l = lsx.merge(oa, la, ob, lb)
    o_ref, l_ref = A.lse_merge(f64(oa), f64(la), f64(ob), f64(lb))
    tol = TOL_FP32 if dt == torch.float32 else 1e-2
    check_lse(f64(l), l_ref, 1e-5)
    check_close(f64(o), o_ref, tol)


def test_merge_in_place_and_extreme_gaps():
    shape = (1, 2, 64, 128)
    oa, la = partial(shape, 3)
    ob, lb = partial(shape, 4)
    la[..., :8] = 500.0
    lb[..., :8] = -500.0
    la[..., 8:16] = -math.inf
    ref = A.lse_merge(f64(oa), f64(la), f64(ob), f64(lb))
    lsx.merge(oa, la, ob, lb, out=oa, lse_out=la)  # in place into a
    check_lse(f64(la), ref[1], 1e-5)
    check_close(f64(oa), ref[0], TOL_FP32)


def test_merge_dense_and_strided_fp32_forms_agree():
    # contiguous fp32 rows take the elementwise kernel (here with O in place),
    # head-interleaved views the warp-per-row kernel
    shape = (2, 4, 300, 128)
    oa, la = partial(shape, 5, empty_rows=(3,))
    ob, lb = partial(shape, 6, empty_rows=(3, 4))
    ref = A.lse_merge(f64(oa), f64(la), f64(ob), f64(lb))
    sa = oa.transpose(1, 2).contiguous().transpose(1, 2)  # [B, N, H, D] storage
    sb = ob.transpose(1, 2).contiguous().transpose(1, 2)
    o_s, l_s = lsx.merge(sa, la, sb, lb)
    l_d = torch.empty_like(la)
    lsx.merge(oa, la, ob, lb, out=oa, lse_out=l_d)
    for o, l in ((oa, l_d), (o_s, l_s)):
        check_lse(f64(l), ref[1], 1e-5)
        check_close(f64(o), ref[0], TOL_FP32)


@pytest.mark.parametrize("k_parts", [1, 2, 5, 16, 17, 256])
def test_tree_merge_matches_oracle(k_parts):
    shape = (k_parts, 2, 4, 33, 128)
    o_p = random_tensor(shape, 7, device=DEV)
    l_p = random_tensor(shape[:-1], 8, 10.0, device=DEV)
    l_p[:, 0, 0, 0] = -math.inf          # a fully empty row
    l_p[: k_parts // 2, 0, 1, 1] = -math.inf
    o_p = o_p.float()
    o, l = lsx.tree_merge(o_p, l_p.float(), out_dtype=torch.float32)
    o_ref, l_ref = A.tree_merge(f64(o_p), f64(l_p.float()))
    check_lse(f64(l), l_ref, 1e-5)
    check_close(f64(o), o_ref, TOL_FP32)


def test_tree_merge_is_deterministic():
    o_p = random_tensor((64, 1, 8, 1000, 128), 9, device=DEV).float()
    l_p = random_tensor((64, 1, 8, 1000), 10, 5.0, device=DEV).float()
    a = lsx.tree_merge(o_p, l_p)
    b = lsx.tree_merge(o_p, l_p)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_fp32_tiny_workload_chunks_merge_and_backward():
    """The tiny fp32 case: 4 chunks of 64, causal chunk pairs, merge, bwd."""
    w = WORKLOADS["tiny_fp32_causal"]
    x = make_inputs(w, device=DEV)
    q, k, v, d_o = x["q"], x["k"], x["v"], x["d_o"]
    n, c = w.N, w.chunk
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=DEV)
    for qc in range(n // c):
        qs = slice(qc * c, (qc + 1) * c)
        acc = None
        for kc in range(qc, -1, -1):  # own chunk first, as in a ring
            ks = slice(kc * c, (kc + 1) * c)
            part = lsx.chunk_fwd(q[:, :, qs], k[:, :, ks], v[:, :, ks], qc * c, kc * c, True)
            acc = part if acc is None else lsx.merge(*acc, *part)
        o[:, :, qs] = acc[0]
        lse[:, :, qs] = acc[1]
    o_ref, lse_ref = A.attn_fwd(f64(q), f64(k), f64(v), 0, 0, True)
    check_lse(f64(lse), lse_ref, TOL_FP32)
    check_close(f64(o), o_ref, TOL_FP32)
    dq = torch.zeros_like(q)
    dk = torch.zeros_like(k)
    dv = torch.zeros_like(v)
    for qc in range(n // c):
        qs = slice(qc * c, (qc + 1) * c)
        for kc in range(qc + 1):
            ks = slice(kc * c, (kc + 1) * c)
            g = lsx.chunk_bwd(q[:, :, qs], k[:, :, ks], v[:, :, ks], o[:, :, qs], lse[:, :, qs],
                              d_o[:, :, qs], qc * c, kc * c, True,
                              dq=dq[:, :, qs], dk=dk[:, :, ks], dv=dv[:, :, ks], accumulate=True)
    dq_r, dk_r, dv_r = A.attn_bwd(f64(q), f64(k), f64(v), f64(d_o), 0, 0, True)
    check_close(f64(dq), dq_r, TOL_FP32, "dQ")
    check_close(f64(dk), dk_r, TOL_FP32, "dK")
    check_close(f64(dv), dv_r, TOL_FP32, "dV")


@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_decode_matches_oracle(g):
    hkv, n, chunk = 2, 20000, 4096  # ragged last chunk
    q = random_tensor((2, hkv * g, 1, 128), 30, device=DEV)
    kc = random_tensor((2, hkv, n, 128), 31, device=DEV)
    vc = random_tensor((2, hkv, n, 128), 32, device=DEV)
    o, lse = lsx.decode(q, kc, vc, chunk, out_dtype=torch.float32)
    o_ref, lse_ref = A.attn_fwd(f64(q), f64(kc), f64(vc))
    check_lse(f64(lse), lse_ref, 1e-3)
    check_close(f64(o), o_ref, 1e-3)


def test_bounded_wait_reports_timeout_without_fault():
    lsx.set_wait_limit_ns(2_000_000)  # 2 ms
    try:
        assert lsx.sync_status() == 0
        lsx.selftest_bounded_wait()
        assert lsx.sync_status() == -8  # LSX_ERR_TIMEOUT
        assert lsx.sync_status() == 0   # cleared by the read
        # the context is still usable
        o, l = lsx.merge(*partial((1, 1, 4, 64), 1), *partial((1, 1, 4, 64), 2))
        torch.cuda.synchronize()
    finally:
        lsx.set_wait_limit_ns(0)
