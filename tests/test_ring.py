"""The ring of chunk pairs and the cross-rank decode merge (ring.py) on CPU:
two and three gloo ranks run the real schedule -- which key/value chunk each
rank holds at each step, which pairs the causal mask skips, the merge of the
partials, and the return of dK / dV to their owners -- with the local work
done by a CPU stand-in (the oracle's forward, merged with the oracle's LSE
merge; a chunk-pair backward from the final LSE written out below).  The
result must equal the oracle over the whole sequence.  The same schedule on
the GPU kernels is in test_gpu_ring.py."""

import math
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleOps:
    """CPU stand-in for the library calls the ring makes (float64 numpy)."""

    def __init__(self):
        from oracle import attention as A
        self.A = A
        self.calls = []  # (q_off, kv_off) of every chunk pair computed

    def chunk_fwd(self, q, k, v, q_off, kv_off, causal, scale, o, lse):
        A = self.A
        self.calls.append(("fwd", q_off, kv_off))
        o_c, l_c = A.attn_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), q_off,
                              kv_off, causal, scale)
        o_m, l_m = A.lse_merge(o.double().numpy(), lse.double().numpy(), o_c, l_c)
        o.copy_(torch.from_numpy(o_m))
        lse.copy_(torch.from_numpy(l_m))

    def chunk_bwd(self, q, k, v, o, lse, d_o, q_off, kv_off, causal, scale, dq, dk, dv):
        # one chunk pair's share of the gradients, from the FINAL (merged) O
        # and LSE of the query rows: P = exp(s - LSE), delta = rowsum(dO o O)
        self.calls.append(("bwd", q_off, kv_off))
        f = lambda t: t.double().numpy()  # noqa: E731
        Q, K, V, O, L, dO = f(q), f(k), f(v), f(o), f(lse), f(d_o)
        b, hq, lq, d = Q.shape
        hkv, lk = K.shape[1], K.shape[2]
        sc = 1.0 / math.sqrt(d) if scale is None else scale
        gq, gk, gv = np.zeros_like(Q), np.zeros_like(K), np.zeros_like(V)
        vis = self.A.visible(q_off + np.arange(lq), kv_off + np.arange(lk), causal)
        for bi in range(b):
            for h in range(hq):
                g = self.A.kv_head_of(h, hq, hkv)
                s = sc * Q[bi, h] @ K[bi, g].T
                p = np.where(vis, np.exp(np.where(vis, s, 0.0) - L[bi, h][:, None]), 0.0)
                dp = dO[bi, h] @ V[bi, g].T
                delta = (dO[bi, h] * O[bi, h]).sum(axis=1, keepdims=True)
                ds = p * (dp - delta)
                gv[bi, g] += p.T @ dO[bi, h]
                gq[bi, h] += sc * ds @ K[bi, g]
                gk[bi, g] += sc * ds.T @ Q[bi, h]
        dq += torch.from_numpy(gq).to(dq.dtype)
        dk += torch.from_numpy(gk).to(dk.dtype)
        dv += torch.from_numpy(gv).to(dv.dtype)

    def decode(self, q, kc, vc, chunk_len, scale):
        o, lse = self.A.attn_fwd(q.double().numpy(), kc.double().numpy(), vc.double().numpy(), 0, 0,
                                 False, scale)
        return torch.from_numpy(o), torch.from_numpy(lse)

    def tree_merge(self, o_parts, lse_parts):
        o, lse = self.A.tree_merge(o_parts.numpy(), lse_parts.numpy())
        return torch.from_numpy(o), torch.from_numpy(lse)


def _inputs(seed, b, hq, hkv, n, d):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn((b, hq, n, d), generator=g, dtype=torch.float64)
    k = torch.randn((b, hkv, n, d), generator=g, dtype=torch.float64)
    v = torch.randn((b, hkv, n, d), generator=g, dtype=torch.float64)
    d_o = torch.randn((b, hq, n, d), generator=g, dtype=torch.float64)
    return q, k, v, d_o


def _ring_main(rank, world, port, causal, out):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from long_sequence_exact_gb300 import ring
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        q, k, v, d_o = _inputs(7, 1, 4, 2, 48 * world, 16)
        n = 48
        rows = slice(rank * n, (rank + 1) * n)
        ops = OracleOps()
        o, lse = ring.ring_attention_fwd(q[:, :, rows], k[:, :, rows], v[:, :, rows], causal,
                                         ops=ops)
        dq, dk, dv = ring.ring_attention_bwd(q[:, :, rows], k[:, :, rows], v[:, :, rows], o, lse,
                                             d_o[:, :, rows], causal, ops=ops)
        out[rank] = (o.numpy(), lse.numpy(), dq.numpy(), dk.numpy(), dv.numpy(), ops.calls)
        dist.barrier()
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("causal", [True, False])
def test_ring_over_gloo_ranks_equals_the_whole_sequence(world, causal):
    from oracle import attention as A
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_ring_main, args=(world, port, causal, out), nprocs=world, join=True)
    q, k, v, d_o = (t.numpy() for t in _inputs(7, 1, 4, 2, 48 * world, 16))
    o_ref, lse_ref = A.attn_fwd(q, k, v, 0, 0, causal)
    dq_ref, dk_ref, dv_ref = A.attn_bwd(q, k, v, d_o, 0, 0, causal)
    n = 48
    for r in range(world):
        o, lse, dq, dk, dv, calls = out[r]
        rows = slice(r * n, (r + 1) * n)
        np.testing.assert_allclose(lse, lse_ref[:, :, rows], atol=1e-5)
        np.testing.assert_allclose(o, o_ref[:, :, rows], atol=1e-5)
        np.testing.assert_allclose(dq, dq_ref[:, :, rows], atol=1e-4)
        np.testing.assert_allclose(dk, dk_ref[:, :, rows], atol=1e-4)
        np.testing.assert_allclose(dv, dv_ref[:, :, rows], atol=1e-4)
        # own chunk first, then the previous ranks' (r, r-1, ...); causal
        # skips the chunks after the rank's own
        order = [((r - s) % world) * n for s in range(world)]
        want = [kv for kv in order if not causal or kv <= r * n]
        assert [c[2] for c in calls if c[0] == "fwd"] == want
        assert [c[2] for c in calls if c[0] == "bwd"] == want
        assert all(c[1] == r * n for c in calls)


def _tree_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from long_sequence_exact_gb300 import ring
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        g = torch.Generator().manual_seed(11)
        q = torch.randn((2, 8, 1, 16), generator=g, dtype=torch.float64)
        kc = torch.randn((2, 2, 96 * world, 16), generator=g, dtype=torch.float64)
        vc = torch.randn((2, 2, 96 * world, 16), generator=g, dtype=torch.float64)
        kc[:, :, 5] *= 6.0  # one key dominates the first shard
        rows = slice(rank * 96, (rank + 1) * 96)
        o, lse = ring.tree_decode(q, kc[:, :, rows], vc[:, :, rows], 32, ops=OracleOps())
        out[rank] = (o.numpy(), lse.numpy())
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_tree_decode_over_gloo_ranks_equals_the_whole_cache():
    from oracle import attention as A
    world = 2
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_tree_main, args=(world, port, out), nprocs=world, join=True)
    g = torch.Generator().manual_seed(11)
    q = torch.randn((2, 8, 1, 16), generator=g, dtype=torch.float64)
    kc = torch.randn((2, 2, 96 * world, 16), generator=g, dtype=torch.float64)
    vc = torch.randn((2, 2, 96 * world, 16), generator=g, dtype=torch.float64)
    kc[:, :, 5] *= 6.0
    o_ref, lse_ref = A.attn_fwd(q.numpy(), kc.numpy(), vc.numpy(), 0, 0, False)
    for r in range(world):
        o, lse = out[r]
        np.testing.assert_allclose(lse, lse_ref, atol=1e-12)
        np.testing.assert_allclose(o, o_ref, atol=1e-12)


def test_schedule_helpers():
    from long_sequence_exact_gb300 import ring
    # every rank sees every chunk exactly once over the ring
    for world in (1, 2, 5):
        for r in range(world):
            assert sorted(ring.kv_chunk(r, s, world) for s in range(world)) == list(range(world))
            assert ring.kv_chunk(r, 0, world) == r
    assert ring.visible(3, 3, True) and ring.visible(3, 0, True) and not ring.visible(2, 3, True)
    assert ring.visible(0, 5, False)
