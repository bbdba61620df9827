"""attn_chunked_fwd / attn_chunked_bwd with rows (key columns) split into
pieces (few heads, long rows): against the fp64 oracle and against the
unsplit launches."""

import ctypes

import numpy as np
import pytest
import torch

from oracle import attention as A
import long_sequence_exact_gb300 as lsx
from long_sequence_exact_gb300 import _lib
from long_sequence_exact_gb300.inputs import random_tensor
from helpers import (TOL_GRAD_REL, TOL_LSE_BF16, TOL_O_BF16, check_close, check_lse, check_tiles,
                     f64, rel_fro)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def qkv(b, hq, hkv, n, d, seed):
    q = random_tensor((b, hq, n, d), seed, 1.0, device=DEV)
    k = random_tensor((b, hkv, n, d), seed + 1, 1.0, device=DEV)
    v = random_tensor((b, hkv, n, d), seed + 2, 1.0, device=DEV)
    return q, k, v


def workspace_sizes(q, k, causal):
    """(attn_chunked_fwd's workspace, the chunk call's: the V copy alone)."""
    lib = _lib.load()
    vq, vk = _lib.view(q), _lib.view(k)
    full = lib.attn_chunked_fwd_workspace_size(ctypes.byref(vq), ctypes.byref(vk), 128,
                                               int(causal))
    base = lib.attn_chunk_fwd_workspace_size(ctypes.byref(vq), ctypes.byref(vk))
    return full, base


def splits(q, k, causal):
    """Whether attn_chunked_fwd plans a split for these shapes (its workspace
    then holds partials beyond the chunk call's V copy)."""
    full, base = workspace_sizes(q, k, causal)
    return full > base


CASES = [
    # B, Hq, Hkv, N, D, causal
    (1, 1, 1, 4096, 128, True),
    (1, 2, 2, 2048, 64, False),
    (1, 4, 2, 3000, 128, True),   # GQA, ragged last tile and pair
    (2, 1, 1, 1408, 64, True),    # odd number of query tiles
]


@pytest.mark.parametrize("case", CASES)
def test_split_rows_match_oracle(case):
    b, hq, hkv, n, d, causal = case
    q, k, v = qkv(b, hq, hkv, n, d, seed=301 + n)
    assert splits(q, k, causal)
    o, lse = lsx.chunked_fwd(q, k, v, 128, causal)
    torch.cuda.synchronize()
    assert lsx.sync_status() == 0
    o_ref, lse_ref = A.attn_fwd(f64(q), f64(k), f64(v), 0, 0, causal)
    check_lse(f64(lse), lse_ref, TOL_LSE_BF16)
    check_close(f64(o), o_ref, TOL_O_BF16)


def test_split_rows_agree_with_the_unsplit_launch_at_32k():
    # one head of 32K causal rows: 64 query pairs for 152 SMs
    q, k, v = qkv(1, 1, 1, 32768, 128, seed=77)
    assert splits(q, k, True)
    o_s, lse_s = lsx.chunked_fwd(q, k, v, 4096, True)
    # a workspace with room for the V copy only: the unsplit launch
    _, base = workspace_sizes(q, k, True)
    small = torch.empty(base, dtype=torch.uint8, device=DEV)
    o_u, lse_u = lsx.chunked_fwd(q, k, v, 4096, True, workspace=small)
    torch.cuda.synchronize()
    assert lsx.sync_status() == 0
    # the same sums in another order: fp32 rounding, then one bf16 rounding
    assert (lse_s - lse_u).abs().max().item() < 1e-4
    assert (o_s.float() - o_u.float()).abs().max().item() < 8e-3
    # and the oracle on sampled rows: the first pair, one in the middle, the last
    for r0 in (0, 16384, 32768 - 256):
        o_ref, lse_ref = A.attn_fwd(f64(q[:, :, r0:r0 + 256]), f64(k), f64(v), r0, 0, True)
        check_lse(f64(lse_s[:, :, r0:r0 + 256]), lse_ref, TOL_LSE_BF16)
        check_close(f64(o_s[:, :, r0:r0 + 256]), o_ref, TOL_O_BF16)


def test_many_heads_do_not_split():
    q, k, v = qkv(1, 32, 32, 4096, 128, seed=9)
    assert not splits(q, k, True)


def bwd_workspace_sizes(q, k, causal):
    """(attn_chunked_bwd's workspace, the chunk call's)."""
    lib = _lib.load()
    vq, vk = _lib.view(q), _lib.view(k)
    full = lib.attn_chunked_bwd_workspace_size(ctypes.byref(vq), ctypes.byref(vk), 128,
                                               int(causal))
    base = lib.attn_chunk_bwd_workspace_size(ctypes.byref(vq), ctypes.byref(vk))
    return full, base


BWD_CASES = [
    # B, Hq, Hkv, N, D, causal: fewer (b, kv head, key tile) items than SMs
    (1, 1, 1, 4096, 128, True),
    (1, 2, 2, 2048, 64, False),
    (1, 4, 2, 3000, 128, True),   # GQA: the pieces cut across the group's heads
    (2, 1, 1, 1408, 64, True),
]


@pytest.mark.parametrize("case", BWD_CASES)
def test_split_backward_matches_oracle(case):
    b, hq, hkv, n, d, causal = case
    q, k, v = qkv(b, hq, hkv, n, d, seed=501 + n)
    d_o = random_tensor((b, hq, n, d), 509 + n, 1.0, device=DEV)
    full, base = bwd_workspace_sizes(q, k, causal)
    assert full > base  # a split is planned
    o, lse = lsx.chunked_fwd(q, k, v, 128, causal)
    dq, dk, dv = lsx.chunked_bwd(q, k, v, o, lse, d_o, 128, causal)
    torch.cuda.synchronize()
    assert lsx.sync_status() == 0
    ref = A.attn_bwd(f64(q), f64(k), f64(v), f64(d_o), 0, 0, causal)
    for got, r, name in zip((dq, dk, dv), ref, ("dQ", "dK", "dV")):
        assert rel_fro(f64(got), r) <= TOL_GRAD_REL, name
        check_tiles(f64(got), r, name)


def test_split_backward_agrees_with_the_unsplit_launch_at_16k():
    # one head of 16K causal rows: 128 key-tile items for 152 SMs
    q, k, v = qkv(1, 1, 1, 16384, 128, seed=71)
    d_o = random_tensor((1, 1, 16384, 128), 79, 1.0, device=DEV)
    full, base = bwd_workspace_sizes(q, k, True)
    assert full > base
    o, lse = lsx.chunked_fwd(q, k, v, 4096, True)
    g_s = lsx.chunked_bwd(q, k, v, o, lse, d_o, 4096, True)
    small = torch.empty(base, dtype=torch.uint8, device=DEV)
    g_u = lsx.chunked_bwd(q, k, v, o, lse, d_o, 4096, True, workspace=small)
    torch.cuda.synchronize()
    assert lsx.sync_status() == 0
    # the same sums in another order (fp32 partials, then one bf16 rounding)
    for a, b_, name in zip(g_s, g_u, ("dQ", "dK", "dV")):
        assert rel_fro(f64(a), f64(b_)) <= 2e-3, name
    # against the oracle on the last 128 rows: their dQ, and dK / dV of the
    # last key tile, which (causal) only those rows see, so that the oracle's
    # row-restricted gradients are exact there
    tail = np.arange(16384 - 128, 16384)
    dq_r, dk_r, dv_r = A.attn_bwd(f64(q), f64(k), f64(v), f64(d_o), 0, 0, True, rows=tail)
    assert rel_fro(f64(g_s[0])[:, :, tail], dq_r) <= TOL_GRAD_REL
    for got, r, name in ((g_s[1], dk_r, "dK"), (g_s[2], dv_r, "dV")):
        assert rel_fro(f64(got)[:, :, tail], r[:, :, tail]) <= TOL_GRAD_REL, name


def test_deterministic_mode_does_not_split_the_backward():
    q, k, v = qkv(1, 1, 1, 4096, 128, seed=9)
    lsx.set_deterministic(True)
    try:
        full, base = bwd_workspace_sizes(q, k, True)
    finally:
        lsx.set_deterministic(False)
    assert full == base
