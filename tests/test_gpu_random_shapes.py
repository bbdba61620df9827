"""Seeded random problems through the C ABI against the fp64 oracle.

Each case draws its own batch, query/key-value head counts (GQA groups of
1, 2 or 4), chunk lengths (ragged, down to one row), absolute offsets of the
two chunks, masking, head dimension and score amplitude, so that the
combinations the hand-picked cases leave out are met too: causal chunk pairs
whose rows see no key, a query tile pair whose second tile is past the end,
groups split over several items, and the whole-sequence calls on problems
small enough that they split rows or key columns into pieces.  The backward
alternates between the two reduction modes and the two workspace sizes.
"""

import numpy as np
import pytest
import torch

from oracle import attention as A
import long_sequence_exact_gb300 as lsx
from long_sequence_exact_gb300.inputs import random_tensor
from helpers import (TOL_GRAD_REL, TOL_LSE_BF16, TOL_O_BF16, bf16_rounding_scales, check_close,
                     check_lse, check_tiles, f64, rel_fro)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def draw_pair(i):
    """One chunk-pair problem: B, Hq, Hkv, Lq, Lk, d, q_off, kv_off, causal, amp."""
    r = np.random.default_rng(7000 + i)
    d = int(r.choice([64, 128]))
    hkv = int(r.integers(1, 3))
    hq = hkv * int(r.choice([1, 2, 4]))
    b = int(r.integers(1, 3))
    lq = int(r.integers(1, 700))
    lk = int(r.integers(1, 900))
    causal = bool(r.integers(0, 4) > 0)  # mostly causal: the offsets matter there
    q_off = int(r.integers(0, 700))
    kv_off = int(r.integers(0, 700))
    amp = float(r.choice([0.5, 1.0, 1.5]))
    return b, hq, hkv, lq, lk, d, q_off, kv_off, causal, amp


def draw_whole(i):
    """One whole-sequence problem: B, Hq, Hkv, N, d, chunk_len, causal, amp."""
    r = np.random.default_rng(9000 + i)
    d = int(r.choice([64, 128]))
    hkv = int(r.choice([1, 2, 4]))
    hq = hkv * int(r.choice([1, 2, 4]))  # up to 16 heads: some problems fill the SMs unsplit
    b = int(r.integers(1, 3))
    n = int(r.integers(1, 2600))
    chunk = int(r.choice([128, 512, 4096]))
    causal = bool(r.integers(0, 2))
    amp = float(r.choice([0.5, 1.0]))
    return b, hq, hkv, n, d, chunk, causal, amp


def inputs(b, hq, hkv, lq, lk, d, amp, seed):
    q = random_tensor((b, hq, lq, d), seed, amp, device=DEV)
    k = random_tensor((b, hkv, lk, d), seed + 1, amp, device=DEV)
    v = random_tensor((b, hkv, lk, d), seed + 2, device=DEV)
    d_o = random_tensor((b, hq, lq, d), seed + 3, device=DEV)
    return q, k, v, d_o


def check_grads(got, ref, scales):
    """The stated bound on the whole tensor, and every 128-row tile within
    the tile bound or, where its rows see only a few keys, within the bf16
    rounding of the method itself (a per-tile relative bound on such a tile
    would demand digits the rounded P, dS and O do not carry)."""
    for name, g, r, sc in zip(("dQ", "dK", "dV"), got, ref, scales):
        gg = f64(g)
        assert not np.any(np.isnan(gg)), f"{name} has NaN"
        if not np.any(r):
            # nothing visible to these rows / keys: the gradient is exactly zero
            assert not np.any(gg), f"{name} nonzero where no score is visible"
            continue
        e = rel_fro(gg, r)
        assert e <= TOL_GRAD_REL, f"{name} relative Frobenius error {e:.3e}"
        check_tiles(gg, r, name, round_rows=sc)


@pytest.mark.parametrize("i", range(64))
def test_random_chunk_pair(i):
    b, hq, hkv, lq, lk, d, q_off, kv_off, causal, amp = draw_pair(i)
    q, k, v, d_o = inputs(b, hq, hkv, lq, lk, d, amp, seed=70 + 11 * i)
    o, lse = lsx.chunk_fwd(q, k, v, q_off, kv_off, causal, use_workspace=bool(i % 3))
    deterministic = i % 2 == 1
    lsx.set_deterministic(deterministic)
    try:
        grads = lsx.chunk_bwd(q, k, v, o, lse, d_o, q_off, kv_off, causal,
                              use_copies=(i // 2) % 2 == 0)
        torch.cuda.synchronize()
    finally:
        lsx.set_deterministic(False)
    assert lsx.sync_status() == 0
    o_ref, lse_ref = A.attn_fwd(f64(q), f64(k), f64(v), q_off, kv_off, causal)
    check_lse(f64(lse), lse_ref, TOL_LSE_BF16)
    check_close(f64(o), o_ref, TOL_O_BF16)
    # rows without a visible key: O = 0 exactly
    empty = np.isneginf(lse_ref)
    if empty.any():
        assert not np.any(f64(o)[empty]), "O nonzero on a row that sees no key"
    ref = A.attn_bwd(f64(q), f64(k), f64(v), f64(d_o), q_off, kv_off, causal)
    check_grads(grads, ref, bf16_rounding_scales(f64(q), f64(k), f64(v), f64(d_o), o_ref,
                                                 lse_ref, q_off, kv_off, causal))


@pytest.mark.parametrize("i", range(24))
def test_random_whole_sequence(i):
    b, hq, hkv, n, d, chunk, causal, amp = draw_whole(i)
    q, k, v, d_o = inputs(b, hq, hkv, n, n, d, amp, seed=90 + 13 * i)
    o, lse = lsx.chunked_fwd(q, k, v, chunk, causal)
    grads = lsx.chunked_bwd(q, k, v, o, lse, d_o, chunk, causal)
    torch.cuda.synchronize()
    assert lsx.sync_status() == 0
    o_ref, lse_ref = A.attn_fwd(f64(q), f64(k), f64(v), 0, 0, causal)
    check_lse(f64(lse), lse_ref, TOL_LSE_BF16)
    check_close(f64(o), o_ref, TOL_O_BF16)
    ref = A.attn_bwd(f64(q), f64(k), f64(v), f64(d_o), 0, 0, causal)
    check_grads(grads, ref, bf16_rounding_scales(f64(q), f64(k), f64(v), f64(d_o), o_ref,
                                                 lse_ref, 0, 0, causal))
