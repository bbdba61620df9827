"""attn_chunked_fwd with rows split into key pieces (few heads, long rows):
against the fp64 oracle and against the unsplit launch."""

import ctypes

import pytest
import torch

from oracle import attention as A
import long_sequence_exact_gb300 as lsx
from long_sequence_exact_gb300 import _lib
from long_sequence_exact_gb300.inputs import random_tensor
from helpers import TOL_LSE_BF16, TOL_O_BF16, check_close, check_lse, f64

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
