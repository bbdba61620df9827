"""The five workloads at their full sizes, on the GPU, in the launch
configuration the bench uses, against the fp64 oracle.

The oracle cannot do every row of a 128K sequence, so these tests:
- recompute sampled query rows one by one (O, LSE, dQ), including rows at
  chunk boundaries;
- check the key rows near the end of a causal sequence exactly (only the
  last query rows see them);
- check identities that hold at any size on every head:
  sum_j dK_j = 0, sum_j dV_j = sum_i dO_i, <Q,dQ> = <K,dK>, <V,dV> = <dO,O>.
Small sizes, where the oracle does every row, are in test_gpu_fwd.py and
test_gpu_bwd.py."""

import numpy as np
import pytest
import torch

from oracle import attention as A
import long_sequence_exact_gb300 as lsx
from long_sequence_exact_gb300.inputs import WORKLOADS, make_inputs
from helpers import (TOL_GRAD_REL, TOL_LSE_BF16, TOL_O_BF16, check_close, check_lse, check_tiles, f64,
                     oracle_bwd_rows, rel_fro)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def sample_rows(n, chunk, extra=24, seed=0):
    rng = np.random.default_rng(seed)
    fixed = {0, 1, chunk - 1, chunk, n // 2 - 1, n // 2, n - 2, n - 1}
    rows = sorted(fixed | set(rng.integers(0, n, size=extra).tolist()))
    return np.array(rows)


def check_identities(q, k, v, o, d_o, dq, dk, dv, heads, causal=True):
    for h in heads:
        Q, K, V, O, dO = (f64(t[0, h]) for t in (q, k, v, o, d_o))
        gQ, gK, gV = f64(dq[0, h]), f64(dk[0, h]), f64(dv[0, h])
        nK, nV = np.linalg.norm(gK), np.linalg.norm(gV)
        assert np.linalg.norm(gK.sum(0)) <= TOL_GRAD_REL * nK
        assert np.linalg.norm(gV.sum(0) - dO.sum(0)) <= TOL_GRAD_REL * nV
        assert abs((Q * gQ).sum() - (K * gK).sum()) <= TOL_GRAD_REL * np.linalg.norm(Q) * np.linalg.norm(gQ)
        assert abs((V * gV).sum() - (dO * O).sum()) <= TOL_GRAD_REL * np.linalg.norm(V) * nV


def test_causal_128k_balanced_full_size():
    w = WORKLOADS["causal_128k_balanced"]
    x = make_inputs(w, device=DEV)
    q, k, v, d_o = x["q"], x["k"], x["v"], x["d_o"]
    o, lse = lsx.chunked_fwd(q, k, v, w.chunk, causal=True)
    dq, dk, dv = lsx.chunked_bwd(q, k, v, o, lse, d_o, w.chunk, causal=True)
    torch.cuda.synchronize()
    assert lsx.sync_status() == 0
    rows = sample_rows(w.N, w.chunk, extra=8)
    for h in (0, 7, 31):
        qh, kh, vh, doh = (f64(t[:, h:h + 1]) for t in (q, k, v, d_o))
        o_ref, lse_ref = A.attn_fwd(qh, kh, vh, 0, 0, True, rows=rows)
        check_lse(f64(lse[:, h:h + 1])[:, :, rows], lse_ref, TOL_LSE_BF16)
        check_close(f64(o[:, h:h + 1])[:, :, rows], o_ref, TOL_O_BF16)
        # the last 2048 key rows are seen only by the last 2048 query rows, so
        # the oracle over those rows gives their dK / dV exactly: 16 key
        # tiles and 16 query tiles compared tile by tile
        tail = np.arange(w.N - 2048, w.N)
        dq_t, dk_t, dv_t = oracle_bwd_rows(qh, kh, vh, doh, 0, 0, True, tail)
        for name, g, r in (("dQ", f64(dq[:, h:h + 1])[:, :, tail], dq_t),
                           ("dK", f64(dk[:, h:h + 1])[:, :, tail], dk_t[:, :, tail]),
                           ("dV", f64(dv[:, h:h + 1])[:, :, tail], dv_t[:, :, tail])):
            assert rel_fro(g, r) <= TOL_GRAD_REL, name
            check_tiles(g, r, name)
        dq_s, _, _ = A.attn_bwd(qh, kh, vh, doh, 0, 0, True, rows=rows[rows < w.N - 2048])
        assert rel_fro(f64(dq[:, h:h + 1])[:, :, rows[rows < w.N - 2048]], dq_s) <= TOL_GRAD_REL
    check_identities(q, k, v, o, d_o, dq, dk, dv, heads=range(0, 32, 3))


def test_causal_32k_ring_order_with_merges():
    """Each query chunk visits key chunks c, c-1, ..., 0 (own first); the
    partials are merged by the forward's fused merge into fp32 (O, LSE); the
    backward runs per chunk pair from the final O/LSE, summing in fp32."""
    w = WORKLOADS["causal_32k_ring"]
    x = make_inputs(w, device=DEV)
    q, k, v, d_o = x["q"], x["k"], x["v"], x["d_o"]
    c, nc = w.chunk, w.N // w.chunk
    o32 = torch.empty(q.shape, dtype=torch.float32, device=DEV)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=DEV)
    for qc in range(nc):
        qs = slice(qc * c, (qc + 1) * c)
        for step, kc in enumerate(range(qc, -1, -1)):
            ks = slice(kc * c, (kc + 1) * c)
            lsx.chunk_fwd(q[:, :, qs], k[:, :, ks], v[:, :, ks], qc * c, kc * c, True,
                          out=o32[:, :, qs], lse=lse[:, :, qs], accumulate=step > 0)
    o = o32.to(torch.bfloat16)
    dq = torch.zeros(q.shape, dtype=torch.float32, device=DEV)
    dk = torch.zeros(k.shape, dtype=torch.float32, device=DEV)
    dv = torch.zeros(v.shape, dtype=torch.float32, device=DEV)
    for qc in range(nc):
        qs = slice(qc * c, (qc + 1) * c)
        for kc in range(qc, -1, -1):
            ks = slice(kc * c, (kc + 1) * c)
            lsx.chunk_bwd(q[:, :, qs], k[:, :, ks], v[:, :, ks], o[:, :, qs], lse[:, :, qs],
                          d_o[:, :, qs], qc * c, kc * c, True, dq=dq[:, :, qs],
                          dk=dk[:, :, ks], dv=dv[:, :, ks], accumulate=True)
    torch.cuda.synchronize()
    assert lsx.sync_status() == 0
    rows = sample_rows(w.N, c)
    for h in (0, 31):
        qh, kh, vh, doh = (f64(t[:, h:h + 1]) for t in (q, k, v, d_o))
        o_ref, lse_ref = A.attn_fwd(qh, kh, vh, 0, 0, True, rows=rows)
        check_lse(f64(lse[:, h:h + 1])[:, :, rows], lse_ref, TOL_LSE_BF16)
        check_close(f64(o32[:, h:h + 1])[:, :, rows], o_ref, TOL_O_BF16)
        dq_r, dk_r, dv_r = A.attn_bwd(qh, kh, vh, doh, 0, 0, True, rows=np.arange(w.N - 512, w.N))
        tail = np.arange(w.N - 512, w.N)
        assert rel_fro(f64(dq[:, h:h + 1])[:, :, tail], dq_r) <= TOL_GRAD_REL
        assert rel_fro(f64(dk[:, h:h + 1])[:, :, tail], dk_r[:, :, tail]) <= TOL_GRAD_REL
        assert rel_fro(f64(dv[:, h:h + 1])[:, :, tail], dv_r[:, :, tail]) <= TOL_GRAD_REL
    # the one-launch chunked path agrees with the ring of chunk pairs
    o2, lse2 = lsx.chunked_fwd(q, k, v, c, causal=True)
    assert float((lse2 - lse).abs().max()) <= 1e-3
    assert float((o2.float() - o32).abs().max()) <= TOL_O_BF16
    check_identities(q, k, v, o, d_o, dq, dk, dv, heads=(0, 15, 31))


def test_noncausal_64k_heavy_tailed_scores():
    w = WORKLOADS["noncausal_64k_heavytail"]
    x = make_inputs(w, device=DEV)
    q, k, v, d_o = x["q"], x["k"], x["v"], x["d_o"]
    o, lse = lsx.chunked_fwd(q, k, v, w.chunk, causal=False)
    dq, dk, dv = lsx.chunked_bwd(q, k, v, o, lse, d_o, w.chunk, causal=False)
    torch.cuda.synchronize()
    assert lsx.sync_status() == 0
    rows = sample_rows(w.N, w.chunk, extra=16)
    for b, h in ((0, 0), (1, 15), (0, 9)):
        qh, kh, vh, doh = (f64(t[b:b + 1, h:h + 1]) for t in (q, k, v, d_o))
        o_ref, lse_ref = A.attn_fwd(qh, kh, vh, 0, 0, False, rows=rows)
        assert np.max(lse_ref) > 40.0  # the heavy rows do dominate some rows
        check_lse(f64(lse[b:b + 1, h:h + 1])[:, :, rows], lse_ref, TOL_LSE_BF16)
        check_close(f64(o[b:b + 1, h:h + 1])[:, :, rows], o_ref, TOL_O_BF16)
        dq_r, _, _ = A.attn_bwd(qh, kh, vh, doh, 0, 0, False, rows=rows)
        assert rel_fro(f64(dq[b:b + 1, h:h + 1])[:, :, rows], dq_r) <= TOL_GRAD_REL
    for b in range(2):
        check_identities(q[b:b + 1], k[b:b + 1], v[b:b + 1], o[b:b + 1], d_o[b:b + 1],
                         dq[b:b + 1], dk[b:b + 1], dv[b:b + 1], heads=(0, 5, 15), causal=False)
    # one whole (b, h) against the oracle over all 65,536 query rows: dK and
    # dV element by element and tile by tile, where the heavy key rows
    # (scores up to ~180) sit among the rest
    b, h = 1, 15
    qh, kh, vh, doh = (f64(t[b:b + 1, h:h + 1]) for t in (q, k, v, d_o))
    _, dk_r, dv_r = oracle_bwd_rows(qh, kh, vh, doh, 0, 0, False, np.arange(w.N))
    for name, g, r in (("dK", f64(dk[b:b + 1, h:h + 1]), dk_r), ("dV", f64(dv[b:b + 1, h:h + 1]), dv_r)):
        assert rel_fro(g, r) <= TOL_GRAD_REL, name
        check_tiles(g, r, name)
    heavy = x["heavy_rows"][b, h].cpu().numpy()
    assert rel_fro(f64(dk[b:b + 1, h:h + 1])[:, :, heavy], dk_r[:, :, heavy]) <= TOL_GRAD_REL


def test_decode_gqa_1m_full_size():
    w = WORKLOADS["decode_gqa_1m"]
    x = make_inputs(w, device=DEV, with_grad=False)
    q, kc, vc = x["q"], x["k"], x["v"]
    o, lse = lsx.decode(q, kc, vc, w.chunk, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert lsx.sync_status() == 0
    g = w.Hq // w.Hkv
    for b, hk in ((0, 0), (3, 5), (7, 7)):
        qh = f64(q[b:b + 1, hk * g:(hk + 1) * g])
        kh, vh = f64(kc[b:b + 1, hk:hk + 1]), f64(vc[b:b + 1, hk:hk + 1])
        o_ref, lse_ref = A.attn_fwd(qh, kh, vh, 0, 0, False)
        check_lse(f64(lse[b:b + 1, hk * g:(hk + 1) * g]), lse_ref, 1e-3)
        check_close(f64(o[b:b + 1, hk * g:(hk + 1) * g]), o_ref, 1e-3)
