"""The bf16 rounding model that lets a degenerate gradient tile pass the
per-tile check (tests/helpers.py: bf16_rounding_scales) against a backward
that applies exactly those roundings in fp64: the model must cover the
rounded backward's error on every tile, and stay far below the gradient on
ordinary tiles, so that a wrong tile is still caught.  CPU only."""

import numpy as np
import pytest
import torch

from oracle import attention as A
from long_sequence_exact_gb300.inputs import random_tensor
from helpers import ROUND_MULT, bf16_rounding_scales, f64

# B, Hq, Hkv, Lq, Lk, d, q_off, kv_off, causal, amp; ordinary: every tile
# holds rows that see many keys
CASES = [
    ((1, 8, 2, 226, 487, 64, 309, 533, True, 1.5), False),  # two rows per head see keys
    ((2, 4, 2, 300, 420, 128, 0, 0, True, 1.0), True),
    ((1, 2, 1, 256, 700, 64, 0, 0, False, 1.5), True),
    ((2, 2, 2, 200, 333, 128, 150, 100, True, 0.5), True),
]


def bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).double().numpy()


def rounded_backward(q, k, v, d_o, o, lse, q_off, kv_off, causal):
    """dQ, dK, dV with P, dS and O rounded to bf16 where the tensor-core
    backward rounds them (everything else exact)."""
    b, hq, lq, d = q.shape
    hkv, lk = k.shape[1], k.shape[2]
    scale = 1.0 / np.sqrt(d)
    vis = A.visible(q_off + np.arange(lq), kv_off + np.arange(lk), causal)
    o_b = bf16(o)
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for bi in range(b):
        for h in range(hq):
            g = A.kv_head_of(h, hq, hkv)
            fin = np.isfinite(lse[bi, h])
            s = scale * (q[bi, h] @ k[bi, g].T)
            with np.errstate(over="ignore", invalid="ignore"):
                p = np.where(vis & fin[:, None],
                             np.exp(s - np.where(fin, lse[bi, h], 0.0)[:, None]), 0.0)
            dp = d_o[bi, h] @ v[bi, g].T
            delta = (d_o[bi, h] * o_b[bi, h]).sum(-1)
            ds = bf16(p * (dp - delta[:, None]))
            dq[bi, h] = scale * ds @ k[bi, g]
            dk[bi, g] += scale * ds.T @ q[bi, h]
            dv[bi, g] += bf16(p).T @ d_o[bi, h]
    return dq, dk, dv


def tile_stats(x, rows=128):
    """Frobenius norm of every 128-row tile of [..., N, d] (or of the root
    sum of squares of [..., N] row scales)."""
    if x.ndim == 4:
        n = x.shape[-2]
        x2 = (x ** 2).sum(-1).reshape(-1, n)
    else:
        n = x.shape[-1]
        x2 = (x ** 2).reshape(-1, n)
    return np.array([np.sqrt(x2[a, t0:t0 + rows].sum()) for a in range(x2.shape[0])
                     for t0 in range(0, n, rows)])


@pytest.mark.parametrize("case,ordinary", CASES)
def test_rounding_model_covers_a_rounded_backward(case, ordinary):
    b, hq, hkv, lq, lk, d, q_off, kv_off, causal, amp = case
    q = f64(random_tensor((b, hq, lq, d), 5, amp, device="cpu"))
    k = f64(random_tensor((b, hkv, lk, d), 6, amp, device="cpu"))
    v = f64(random_tensor((b, hkv, lk, d), 7, device="cpu"))
    d_o = f64(random_tensor((b, hq, lq, d), 8, device="cpu"))
    o, lse = A.attn_fwd(q, k, v, q_off, kv_off, causal)
    exact = A.attn_bwd(q, k, v, d_o, q_off, kv_off, causal)
    rounded = rounded_backward(q, k, v, d_o, o, lse, q_off, kv_off, causal)
    scales = bf16_rounding_scales(q, k, v, d_o, o, lse, q_off, kv_off, causal)
    for name, ex, ro, sc in zip(("dQ", "dK", "dV"), exact, rounded, scales):
        err = tile_stats(ro - ex)
        model = tile_stats(sc)
        norm = tile_stats(ex)
        live = norm > 0
        # every tile's rounding error within the model's allowance
        assert np.all(err[live] <= ROUND_MULT * model[live]), name
        # and on ordinary problems the allowance is a small part of the
        # median tile: a lost or doubled contribution (an error of the tile's
        # own size) cannot hide under it
        if ordinary:
            assert np.median(ROUND_MULT * model[live] / norm[live]) < 0.1, name


def test_tile_check_with_the_model_still_catches_a_wrong_tile():
    from helpers import check_tiles
    (b, hq, hkv, lq, lk, d, q_off, kv_off, causal, amp), _ = CASES[1]
    q = f64(random_tensor((b, hq, lq, d), 5, amp, device="cpu"))
    k = f64(random_tensor((b, hkv, lk, d), 6, amp, device="cpu"))
    v = f64(random_tensor((b, hkv, lk, d), 7, device="cpu"))
    d_o = f64(random_tensor((b, hq, lq, d), 8, device="cpu"))
    o, lse = A.attn_fwd(q, k, v, q_off, kv_off, causal)
    exact = A.attn_bwd(q, k, v, d_o, q_off, kv_off, causal)
    scales = bf16_rounding_scales(q, k, v, d_o, o, lse, q_off, kv_off, causal)
    rounded = rounded_backward(q, k, v, d_o, o, lse, q_off, kv_off, causal)
    for ex, ro, sc in zip(exact, rounded, scales):
        check_tiles(ro, ex, round_rows=sc)  # the rounded backward passes
        # one key tile's contribution lost from one tile of rows (a quarter
        # of that tile's value), and one tile doubled
        bad = ro.copy()
        bad[0, 0, 128:256] *= 0.75
        with pytest.raises(AssertionError):
            check_tiles(bad, ex, round_rows=sc)
        bad = ro.copy()
        bad[-1, -1, :128] *= 2.0
        with pytest.raises(AssertionError):
            check_tiles(bad, ex, round_rows=sc)
