"""Shared-prefix tree decoding (attn_decode_tree) against the fp64 oracle:
each branch's answer is plain attention over the prefix followed by its own
suffix."""

import numpy as np
import pytest
import torch

from oracle import attention as A
import long_sequence_exact_gb300 as lsx
from long_sequence_exact_gb300.inputs import random_tensor
from helpers import check_close, check_lse, f64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def oracle_tree(q, pk, pv, sk, sv):
    qs, out, lse = f64(q), [], []
    for b in range(q.shape[0]):
        k = f64(pk)[0]
        v = f64(pv)[0]
        if sk is not None:
            k = np.concatenate([k, f64(sk)[b]], axis=1)
            v = np.concatenate([v, f64(sv)[b]], axis=1)
        o, l_ = A.attn_fwd(qs[b:b + 1], k[None], v[None])
        out.append(o)
        lse.append(l_)
    return np.concatenate(out), np.concatenate(lse)


@pytest.mark.parametrize("branches,g,np_,ns", [
    (8, 4, 20000, 1000),   # 32 query rows per kv head against the prefix
    (4, 4, 10000, 100),    # 16 rows: one 16-row warp tile, eight key groups
    (3, 4, 5000, 300),     # ragged branch groups (2 + 1)
    (5, 1, 4096, 700),     # MHA, odd branch count
    (16, 8, 9000, 0),      # 128 rows: two groups of 8 branches, no suffixes
    (1, 2, 3000, 129),     # one branch
])
def test_decode_tree_matches_oracle(branches, g, np_, ns):
    hkv = 2
    q = random_tensor((branches, hkv * g, 1, 128), 81, device=DEV)
    pk = random_tensor((1, hkv, np_, 128), 82, device=DEV)
    pv = random_tensor((1, hkv, np_, 128), 83, device=DEV)
    sk = random_tensor((branches, hkv, ns, 128), 84, device=DEV) if ns else None
    sv = random_tensor((branches, hkv, ns, 128), 85, device=DEV) if ns else None
    o, lse = lsx.decode_tree(q, pk, pv, sk, sv, 4096, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert lsx.sync_status() == 0
    o_ref, l_ref = oracle_tree(q, pk, pv, sk, sv)
    check_lse(f64(lse), l_ref, 1e-3)
    check_close(f64(o), o_ref, 1e-3)


def test_decode_tree_equals_plain_decode_on_the_concatenated_cache():
    b, hkv, g, np_, ns = 4, 2, 4, 8192, 512
    q = random_tensor((b, hkv * g, 1, 128), 91, device=DEV)
    pk = random_tensor((1, hkv, np_, 128), 92, device=DEV)
    pv = random_tensor((1, hkv, np_, 128), 93, device=DEV)
    sk = random_tensor((b, hkv, ns, 128), 94, device=DEV)
    sv = random_tensor((b, hkv, ns, 128), 95, device=DEV)
    o, lse = lsx.decode_tree(q, pk, pv, sk, sv, 4096, out_dtype=torch.float32)
    kc = torch.cat([pk.expand(b, -1, -1, -1), sk], dim=2).contiguous()
    vc = torch.cat([pv.expand(b, -1, -1, -1), sv], dim=2).contiguous()
    o2, l2 = lsx.decode(q, kc, vc, 4096, out_dtype=torch.float32)
    # 16 query rows per kv head take the tensor-core prefix kernel, which
    # rounds P to bf16 before the P V product (the plain decode keeps it in
    # f32): O agrees to that rounding, LSE (from the f32 scores) closely
    assert float((o - o2).abs().max()) < 1e-3
    assert float((lse - l2).abs().max()) < 1e-5
