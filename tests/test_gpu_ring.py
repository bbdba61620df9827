"""The ring schedule of ring.py run on the GPU kernels: all ranks' steps in
one process (the one-process drivers), so that the schedule that the gloo
test checks on CPU also drives attn_chunk_fwd / attn_chunk_bwd (accumulate)
and attn_decode / attn_tree_merge; the result must match the fp64 oracle over
the whole sequence (whole cache)."""

import numpy as np
import pytest
import torch

from oracle import attention as A
import long_sequence_exact_gb300 as lsx
from long_sequence_exact_gb300 import ring
from long_sequence_exact_gb300.inputs import random_tensor
from helpers import TOL_GRAD_REL, TOL_LSE_BF16, TOL_O_BF16, check_close, check_lse, check_tiles, f64, rel_fro

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("causal", [True, False])
def test_ring_of_four_ranks_matches_the_whole_sequence(d, causal):
    world, n = 4, 512
    b, hq, hkv = 1, 4, 2
    q = random_tensor((b, hq, world * n, d), 301, 0.5, device=DEV)
    k = random_tensor((b, hkv, world * n, d), 302, 0.5, device=DEV)
    v = random_tensor((b, hkv, world * n, d), 303, device=DEV)
    d_o = random_tensor((b, hq, world * n, d), 304, device=DEV)
    cut = lambda t: [t[:, :, r * n:(r + 1) * n] for r in range(world)]  # noqa: E731
    qs, ks, vs, dos = cut(q), cut(k), cut(v), cut(d_o)
    outs = ring.ring_attention_fwd_sim(qs, ks, vs, causal)
    grads = ring.ring_attention_bwd_sim(qs, ks, vs, [o for o, _ in outs], [l for _, l in outs], dos,
                                        causal)
    torch.cuda.synchronize()
    assert lsx.sync_status() == 0
    o = torch.cat([o_ for o_, _ in outs], dim=2)
    lse = torch.cat([l_ for _, l_ in outs], dim=2)
    o_ref, lse_ref = A.attn_fwd(f64(q), f64(k), f64(v), 0, 0, causal)
    check_lse(f64(lse), lse_ref, TOL_LSE_BF16)
    check_close(f64(o), o_ref, TOL_O_BF16)
    ref = A.attn_bwd(f64(q), f64(k), f64(v), f64(d_o), 0, 0, causal)
    for i, name in enumerate(("dQ", "dK", "dV")):
        g = torch.cat([gr[i] for gr in grads], dim=2)
        assert rel_fro(f64(g), ref[i]) <= TOL_GRAD_REL, name
        check_tiles(f64(g), ref[i], name)


def test_tree_decode_over_four_shards_matches_the_whole_cache():
    shards, ns = 4, 4096
    q = random_tensor((2, 8, 1, 128), 401, device=DEV)
    kc = random_tensor((2, 2, shards * ns, 128), 402, device=DEV)
    vc = random_tensor((2, 2, shards * ns, 128), 403, device=DEV)
    ks = [kc[:, :, s * ns:(s + 1) * ns] for s in range(shards)]
    vs = [vc[:, :, s * ns:(s + 1) * ns] for s in range(shards)]
    o, lse = ring.tree_decode_sim(q, ks, vs, 1024)
    o_one, lse_one = lsx.decode(q, kc, vc, 1024, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert lsx.sync_status() == 0
    o_ref, lse_ref = A.attn_fwd(f64(q), f64(kc), f64(vc), 0, 0, False)
    check_lse(f64(lse), lse_ref, 1e-3)
    check_close(f64(o), o_ref, 1e-3)
    # the same partials as one GPU's own split-KV decode, merged one level up
    assert float((lse - lse_one).abs().max()) <= 1e-5
    assert float((o - o_one).abs().max()) <= 1e-5
