"""Seeded random problems for the other entry points, against the fp64
oracle: block-sparse attention (random masks, densities, shapes, GQA, both
head dimensions, causal or not), split-KV decode and shared-prefix tree
decoding (batch, group size, cache and suffix lengths, chunk lengths, output
dtype), and the pairwise and tree merges (shapes, dtypes, empty rows, LSE
gaps, number of partials)."""

import math

import numpy as np
import pytest
import torch

from oracle import attention as A
import long_sequence_exact_gb300 as lsx
from long_sequence_exact_gb300.inputs import random_tensor
from helpers import (TOL_FP32, TOL_GRAD_REL, TOL_LSE_BF16, TOL_O_BF16, bf16_rounding_scales,
                     check_close, check_lse, check_tiles, f64, rel_fro)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("i", range(16))
def test_random_block_sparse(i):
    r = np.random.default_rng(11000 + i)
    d = int(r.choice([64, 128]))
    hkv = int(r.integers(1, 3))
    hq = hkv * int(r.choice([1, 2, 4]))
    b = int(r.integers(1, 3))
    lq = int(r.integers(1, 1300))
    lk = lq if r.integers(0, 2) else int(r.integers(1, 1300))
    causal = bool(r.integers(0, 2))
    density = float(r.choice([0.15, 0.5, 0.9]))
    mask = (r.random((-(-lq // 128), -(-lk // 128))) < density).astype(np.uint8)
    seed = 110 + 7 * i
    q = random_tensor((b, hq, lq, d), seed, 0.7, device=DEV)
    k = random_tensor((b, hkv, lk, d), seed + 1, 0.7, device=DEV)
    v = random_tensor((b, hkv, lk, d), seed + 2, device=DEV)
    d_o = random_tensor((b, hq, lq, d), seed + 3, device=DEV)
    mt = torch.from_numpy(mask)
    o, lse = lsx.block_sparse_fwd(q, k, v, mt, causal)
    grads = lsx.block_sparse_bwd(q, k, v, o, lse, d_o, mt, causal)
    torch.cuda.synchronize()
    assert lsx.sync_status() == 0
    Q, K, V, DO = f64(q), f64(k), f64(v), f64(d_o)
    o_ref, lse_ref = A.attn_fwd(Q, K, V, 0, 0, causal, block_mask=mask)
    check_lse(f64(lse), lse_ref, TOL_LSE_BF16)
    check_close(f64(o), o_ref, TOL_O_BF16)
    ref = A.attn_bwd(Q, K, V, DO, 0, 0, causal, block_mask=mask)
    scales = bf16_rounding_scales(Q, K, V, DO, o_ref, lse_ref, 0, 0, causal, block_mask=mask)
    for name, g, rr, sc in zip(("dQ", "dK", "dV"), grads, ref, scales):
        gg = f64(g)
        assert not np.any(np.isnan(gg)), name
        if not np.any(rr):
            assert not np.any(gg), f"{name} nonzero where no score is visible"
            continue
        assert rel_fro(gg, rr) <= TOL_GRAD_REL, name
        check_tiles(gg, rr, name, round_rows=sc)


@pytest.mark.parametrize("i", range(12))
def test_random_decode(i):
    r = np.random.default_rng(12000 + i)
    b = int(r.integers(1, 5))
    hkv = int(r.choice([1, 2, 4]))
    g = int(r.choice([1, 2, 4, 8]))
    n = int(r.integers(1, 30000))
    chunk = 128 * int(r.choice([1, 4, 32, 64]))
    out_dtype = torch.float32 if r.integers(0, 2) else torch.bfloat16
    seed = 120 + 5 * i
    q = random_tensor((b, hkv * g, 1, 128), seed, device=DEV)
    kc = random_tensor((b, hkv, n, 128), seed + 1, device=DEV)
    vc = random_tensor((b, hkv, n, 128), seed + 2, device=DEV)
    o, lse = lsx.decode(q, kc, vc, chunk, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert lsx.sync_status() == 0
    o_ref, lse_ref = A.attn_fwd(f64(q), f64(kc), f64(vc))
    check_lse(f64(lse), lse_ref, 1e-3)
    check_close(f64(o), o_ref, 1e-3 if out_dtype == torch.float32 else TOL_O_BF16)


@pytest.mark.parametrize("i", range(10))
def test_random_decode_tree(i):
    r = np.random.default_rng(13000 + i)
    branches = int(r.integers(1, 21))
    hkv = int(r.integers(1, 3))
    g = int(r.choice([1, 2, 4, 8]))
    np_ = int(r.integers(1, 12000))
    ns = int(r.choice([0, int(r.integers(1, 1500))]))
    chunk = 128 * int(r.choice([1, 8, 32]))
    seed = 130 + 9 * i
    q = random_tensor((branches, hkv * g, 1, 128), seed, device=DEV)
    pk = random_tensor((1, hkv, np_, 128), seed + 1, device=DEV)
    pv = random_tensor((1, hkv, np_, 128), seed + 2, device=DEV)
    sk = random_tensor((branches, hkv, ns, 128), seed + 3, device=DEV) if ns else None
    sv = random_tensor((branches, hkv, ns, 128), seed + 4, device=DEV) if ns else None
    o, lse = lsx.decode_tree(q, pk, pv, sk, sv, chunk, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert lsx.sync_status() == 0
    qs = f64(q)
    for bi in range(branches):
        kk, vv = f64(pk)[0], f64(pv)[0]
        if ns:
            kk = np.concatenate([kk, f64(sk)[bi]], axis=1)
            vv = np.concatenate([vv, f64(sv)[bi]], axis=1)
        o_ref, l_ref = A.attn_fwd(qs[bi:bi + 1], kk[None], vv[None])
        check_lse(f64(lse[bi:bi + 1]), l_ref, 1e-3)
        check_close(f64(o[bi:bi + 1]), o_ref, 1e-3)


def random_partials(r, k_parts, shape, dtype, seed):
    """k partials [k, B, H, N, D] with LSEs of spread `gap`, some empty rows
    (in some partials, and one row empty in all)."""
    o = random_tensor((k_parts,) + shape, seed, device=DEV).to(dtype)
    gap = float(r.choice([1.0, 20.0, 300.0]))
    lse = random_tensor((k_parts,) + shape[:-1], seed + 1, gap, device=DEV).float()
    n = shape[2]
    for _ in range(int(r.integers(0, 4))):
        p_ = int(r.integers(0, k_parts))
        row = int(r.integers(0, n))
        lse[p_, :, :, row] = -math.inf
        o[p_, :, :, row] = 0
    lse[:, 0, 0, n - 1] = -math.inf
    o[:, 0, 0, n - 1] = 0
    return o, lse


@pytest.mark.parametrize("i", range(16))
def test_random_merges(i):
    r = np.random.default_rng(14000 + i)
    d = int(r.choice([64, 128]))
    shape = (int(r.integers(1, 3)), int(r.integers(1, 6)), int(r.integers(1, 900)), d)
    dt_in = torch.float32 if r.integers(0, 2) else torch.bfloat16
    dt_out = torch.float32 if r.integers(0, 2) else torch.bfloat16

    def tol(ref):
        # fp32 throughout: the fp32 bound; a bf16 output: two half-units in
        # the last place of the largest value (the merge's rounding, then the
        # output's), and at least the bf16 bound of the other tests
        if dt_out == torch.float32:
            return TOL_FP32
        return max(1e-2, 2.0 ** -7 * float(np.max(np.abs(ref))))

    def lse_tol(ref):
        # fp32 LSEs of magnitude up to ~1000 (gaps of 300): a few units in
        # the last place of the largest
        fin = ref[np.isfinite(ref)]
        return max(1e-5, 5e-7 * float(np.max(np.abs(fin)))) if fin.size else 1e-5
    # pairwise
    parts, lses = random_partials(r, 2, shape, dt_in, 140 + 3 * i)
    out = torch.empty(shape, dtype=dt_out, device=DEV)
    o, l_ = lsx.merge(parts[0], lses[0], parts[1], lses[1], out=out)
    o_ref, l_ref = A.lse_merge(f64(parts[0]), f64(lses[0]), f64(parts[1]), f64(lses[1]))
    check_lse(f64(l_), l_ref, lse_tol(l_ref))
    check_close(f64(o), o_ref, tol(o_ref))
    # tree, k partials (fewer rows for many partials: the oracle's fp64 copy)
    k_parts = int(r.choice([1, 3, 16, 33, 257]))
    parts, lses = random_partials(r, k_parts, shape[:2] + (min(shape[2], 10000 // k_parts + 1), d),
                                  dt_in, 150 + 3 * i)
    o, l_ = lsx.tree_merge(parts, lses, out_dtype=dt_out)
    torch.cuda.synchronize()
    assert lsx.sync_status() == 0
    o_ref, l_ref = A.tree_merge(f64(parts), f64(lses))
    check_lse(f64(l_), l_ref, lse_tol(l_ref))
    check_close(f64(o), o_ref, tol(o_ref))


@pytest.mark.parametrize("i", range(12))
def test_random_fp32_chunk_pairs_merged(i):
    """The fp32 path: a random chunk pair split at random key positions into
    up to three key chunks, partials merged pairwise, gradients accumulated
    over the key chunks from the merged O and LSE."""
    r = np.random.default_rng(15000 + i)
    d = int(r.choice([64, 128]))
    hkv = int(r.integers(1, 3))
    hq = hkv * int(r.choice([1, 2]))
    b = int(r.integers(1, 3))
    lq = int(r.integers(1, 300))
    lk = int(r.integers(2, 400))
    causal = bool(r.integers(0, 4) > 0)
    q_off, kv_off = int(r.integers(0, 300)), int(r.integers(0, 300))
    cuts = [0] + sorted(int(c) for c in r.choice(np.arange(1, lk), size=min(2, lk - 1),
                                                  replace=False)) + [lk]
    seed = 160 + 7 * i
    f32 = torch.float32
    q = random_tensor((b, hq, lq, d), seed, dtype=f32, device=DEV)
    k = random_tensor((b, hkv, lk, d), seed + 1, dtype=f32, device=DEV)
    v = random_tensor((b, hkv, lk, d), seed + 2, dtype=f32, device=DEV)
    d_o = random_tensor((b, hq, lq, d), seed + 3, dtype=f32, device=DEV)
    acc = None
    for a, e in zip(cuts[:-1], cuts[1:]):
        part = lsx.chunk_fwd(q, k[:, :, a:e], v[:, :, a:e], q_off, kv_off + a, causal)
        acc = part if acc is None else lsx.merge(*acc, *part)
    o, lse = acc
    dq, dk, dv = torch.zeros_like(q), torch.zeros_like(k), torch.zeros_like(v)
    for a, e in zip(cuts[:-1], cuts[1:]):
        lsx.chunk_bwd(q, k[:, :, a:e], v[:, :, a:e], o, lse, d_o, q_off, kv_off + a, causal,
                      dq=dq, dk=dk[:, :, a:e], dv=dv[:, :, a:e], accumulate=True)
    torch.cuda.synchronize()
    assert lsx.sync_status() == 0
    Q, K, V, DO = f64(q), f64(k), f64(v), f64(d_o)
    o_ref, lse_ref = A.attn_fwd(Q, K, V, q_off, kv_off, causal)
    check_lse(f64(lse), lse_ref, TOL_FP32)
    check_close(f64(o), o_ref, TOL_FP32)
    for name, g, rr in zip(("dQ", "dK", "dV"), (dq, dk, dv),
                           A.attn_bwd(Q, K, V, DO, q_off, kv_off, causal)):
        check_close(f64(g), rr, TOL_FP32, name)
