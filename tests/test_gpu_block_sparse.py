"""Block-sparse attention (128 x 128 block mask) through the C ABI against the
fp64 oracle with the same mask, and against the dense chunked path."""

import ctypes

import numpy as np
import pytest
import torch

from oracle import attention as A
import long_sequence_exact_gb300 as lsx
from long_sequence_exact_gb300 import _lib
from long_sequence_exact_gb300.inputs import random_tensor
from helpers import TOL_GRAD_REL, TOL_LSE_BF16, TOL_O_BF16, check_close, check_lse, f64, rel_fro

pytestmark = pytest.mark.gpu
DEV = "cuda"


def make(hq, hkv, n, d, seed):
    q = random_tensor((1, hq, n, d), seed, 0.5, device=DEV)
    k = random_tensor((1, hkv, n, d), seed + 1, 0.5, device=DEV)
    v = random_tensor((1, hkv, n, d), seed + 2, device=DEV)
    d_o = random_tensor((1, hq, n, d), seed + 3, device=DEV)
    return q, k, v, d_o


def random_mask(n, density, seed):
    nb = -(-n // 128)
    m = (np.random.default_rng(seed).random((nb, nb)) < density).astype(np.uint8)
    return m


def check_against_oracle(q, k, v, d_o, mask, causal):
    mt = torch.from_numpy(mask)
    o, lse = lsx.block_sparse_fwd(q, k, v, mt, causal)
    grads = lsx.block_sparse_bwd(q, k, v, o, lse, d_o, mt, causal, dq=torch.empty(q.shape, device=DEV),
                                 dk=torch.empty(k.shape, device=DEV),
                                 dv=torch.empty(v.shape, device=DEV))
    torch.cuda.synchronize()
    assert lsx.sync_status() == 0
    o_ref, l_ref = A.attn_fwd(f64(q), f64(k), f64(v), 0, 0, causal, block_mask=mask)
    check_close(f64(o), o_ref, TOL_O_BF16)
    check_lse(f64(lse), l_ref, TOL_LSE_BF16)
    ref = A.attn_bwd(f64(q), f64(k), f64(v), f64(d_o), 0, 0, causal, block_mask=mask)
    for name, g, r in zip(("dQ", "dK", "dV"), grads, ref):
        e = rel_fro(f64(g), r)
        assert e <= TOL_GRAD_REL, f"{name} relative Frobenius error {e:.3e}"
    return o, lse, grads


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("d", [128, 64])
def test_random_block_mask_matches_oracle(causal, d):
    n = 1000  # ragged last block
    q, k, v, d_o = make(4, 2, n, d, 11 + d)
    mask = random_mask(n, 0.5, 5 + d + causal)
    mask[2, :] = 0  # query rows 256..383 see nothing
    o, lse, grads = check_against_oracle(q, k, v, d_o, mask, causal)
    assert torch.all(o[:, :, 256:384] == 0)
    assert torch.all(torch.isneginf(lse[:, :, 256:384]))
    assert torch.all(grads[0][:, :, 256:384] == 0)


def test_sliding_window_mask_matches_oracle():
    n, w = 4096, 4  # each query block sees itself and the 3 blocks before it
    q, k, v, d_o = make(2, 2, n, 128, 41)
    nb = n // 128
    mask = np.zeros((nb, nb), np.uint8)
    for i in range(nb):
        mask[i, max(0, i - w + 1):i + 1] = 1
    check_against_oracle(q, k, v, d_o, mask, True)


def test_full_mask_equals_dense_chunked_path():
    n = 1536
    q, k, v, d_o = make(4, 4, n, 128, 61)
    nb = n // 128
    full = torch.ones((nb, nb), dtype=torch.uint8)
    # (a workspace with room for the V copy only keeps the chunked forward on
    # its unsplit launch: these 48 query pairs would otherwise be split into
    # key pieces and merged, which rounds differently)
    vq, vk = _lib.view(q), _lib.view(k)
    lib = _lib.load()
    base = lib.attn_chunk_fwd_workspace_size(ctypes.byref(vq), ctypes.byref(vk))
    ws = torch.empty(base, dtype=torch.uint8, device=DEV)
    # (likewise the backward: its 48 key-tile items would be split)
    base_b = lib.attn_chunk_bwd_workspace_size(ctypes.byref(vq), ctypes.byref(vk))
    ws_b = torch.empty(base_b, dtype=torch.uint8, device=DEV)
    for causal in (True, False):
        o1, l1 = lsx.block_sparse_fwd(q, k, v, full, causal)
        o2, l2 = lsx.chunked_fwd(q, k, v, 512, causal, workspace=ws)
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
        g1 = lsx.block_sparse_bwd(q, k, v, o1, l1, d_o, full, causal)
        g2 = lsx.chunked_bwd(q, k, v, o2, l2, d_o, 512, causal, workspace=ws_b)
        # dK, dV identical; dQ's fp32 partial sums land in a varying order
        assert rel_fro(f64(g1[0]), f64(g2[0])) <= 1e-3
        for a, b in zip(g1[1:], g2[1:]):
            assert torch.equal(a, b)
        lsx.set_deterministic(True)
        try:
            g1 = lsx.block_sparse_bwd(q, k, v, o1, l1, d_o, full, causal)
            g2 = lsx.chunked_bwd(q, k, v, o2, l2, d_o, 512, causal)
        finally:
            lsx.set_deterministic(False)
        for a, b in zip(g1, g2):
            assert torch.equal(a, b)


def test_rejects_a_mask_of_the_wrong_shape():
    q, k, v, _ = make(2, 2, 300, 128, 71)
    with pytest.raises(ValueError):
        lsx.block_sparse_fwd(q, k, v, torch.ones((2, 2), dtype=torch.uint8))
