"""Sequence-parallel exact attention across ranks: the ring of chunk pairs and
the cross-rank merge of decode partials.  Host-side schedule only; every step
of the local work is a call into liblsx.

What the pages describe:
  * BurstAttention (method section): the sequence is split into chunks, one
    per device; each device computes the local attention of its query chunk
    against the key/value chunk it currently holds, passes that chunk on
    around a ring, and aggregates the local results into the global ones
    (Ring Attention, on the same page's related work, is the same rotation).
  * DistFlashAttn (core concepts): the backward pass runs from the saved
    output and log-sum-exp, and the key/value gradients travel with their
    chunk until they are back with its owner.
  * Tree Attention (abstract): for decoding, the key/value cache is sharded
    across devices; each computes a partial (O, LSE) and the partials are
    combined by the associative LSE-weighted reduction.

Layout and order (the readings taken where the pages are silent):
  * Rank r holds query, key and value rows [r L, (r + 1) L) of a sequence of
    world * L tokens; causal masking uses those absolute positions.
  * At ring step s rank r holds key/value chunk (r - s) mod world: its own
    chunk first, then the previous ranks' (the order the single-GPU ring
    test of the 32K workload uses).  Chunk pairs the causal mask hides
    entirely (key chunk after the query chunk) are skipped, but the chunk is
    still passed on.
  * The forward keeps an fp32 partial (O, LSE) per rank, starting from the
    merge identity (O = 0, LSE = -inf) and merging every visible pair into it
    with attn_chunk_fwd(accumulate = 1).
  * The backward adds into fp32 dQ (kept) and fp32 dK / dV (travelling with
    the chunk) with attn_chunk_bwd(accumulate = 1); after the last step one
    more pass takes every chunk's dK / dV home.
  * Every received tensor lands in a fresh local buffer before any kernel
    reads it (copy, then compute); nothing is multicast.  Sending the chunk
    held in step s overlaps the compute of step s (both only read it).

Two drivers share the per-step code: ``ring_attention_fwd`` /
``ring_attention_bwd`` / ``tree_decode`` run one rank per process over
``torch.distributed`` point-to-point and all-gather; the ``*_sim`` drivers
run all ranks' steps in one process, passing the tensors by reference, so the
same schedule can be run on one GPU.

The local work goes through an ``ops`` object (default ``LibOps``, the CUDA
library); the schedule is independent of it.
"""

from __future__ import annotations

import math

import torch

from . import attention as _att


# ------------------------------------------------------------- schedule
def kv_chunk(rank: int, step: int, world: int) -> int:
    """Key/value chunk that `rank` holds at ring step `step`."""
    return (rank - step) % world


def visible(q_chunk: int, k_chunk: int, causal: bool) -> bool:
    """Whether any key of chunk k_chunk is visible to a query of q_chunk
    (equal-length chunks, absolute positions)."""
    return (not causal) or k_chunk <= q_chunk


class LibOps:
    """Local work through liblsx (the C ABI): every call is one or two
    kernel launches on the current stream."""

    def chunk_fwd(self, q, k, v, q_off, kv_off, causal, scale, o, lse):
        _att.chunk_fwd(q, k, v, q_off, kv_off, causal, scale, out=o, lse=lse, accumulate=True)

    def chunk_bwd(self, q, k, v, o, lse, d_o, q_off, kv_off, causal, scale, dq, dk, dv):
        _att.chunk_bwd(q, k, v, o, lse, d_o, q_off, kv_off, causal, scale, dq=dq, dk=dk, dv=dv,
                       accumulate=True)

    def decode(self, q, kc, vc, chunk_len, scale):
        return _att.decode(q, kc, vc, chunk_len, scale, out_dtype=torch.float32)

    def tree_merge(self, o_parts, lse_parts):
        return _att.tree_merge(o_parts, lse_parts, out_dtype=torch.float32)


def _partial_identity(q):
    o = torch.zeros(q.shape, dtype=torch.float32, device=q.device)
    lse = torch.full(q.shape[:3], -math.inf, dtype=torch.float32, device=q.device)
    return o, lse


def _fwd_step(ops, rank, step, world, q, held, causal, scale, o, lse):
    c = kv_chunk(rank, step, world)
    if visible(rank, c, causal):
        n = q.shape[2]
        ops.chunk_fwd(q, held[0], held[1], rank * n, c * n, causal, scale, o, lse)


def _bwd_step(ops, rank, step, world, q, o, lse, d_o, held, causal, scale, dq):
    c = kv_chunk(rank, step, world)
    if visible(rank, c, causal):
        n = q.shape[2]
        ops.chunk_bwd(q, held[0], held[1], o, lse, d_o, rank * n, c * n, causal, scale, dq,
                      held[2], held[3])


# ------------------------------------------------- torch.distributed driver
class _P2P:
    """Ring transport: every tensor goes to rank + 1 and the same shapes come
    from rank - 1 into fresh local buffers."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.world = dist.get_world_size(group)
        self.rank = dist.get_rank(group)

        def glob(r):
            return r if group is None else dist.get_global_rank(group, r)
        self.nxt = glob((self.rank + 1) % self.world)
        self.prv = glob((self.rank - 1) % self.world)

    def start(self, tensors):
        d = self.dist
        recv = [torch.empty_like(t) for t in tensors]
        ops = [d.P2POp(d.isend, t.contiguous(), self.nxt, self.group) for t in tensors]
        ops += [d.P2POp(d.irecv, r, self.prv, self.group) for r in recv]
        return d.batch_isend_irecv(ops), recv

    @staticmethod
    def finish(handle):
        reqs, recv = handle
        for r in reqs:
            r.wait()
        return tuple(recv)


def ring_attention_fwd(q, k, v, causal=True, scale=None, group=None, ops=None):
    """Forward of this rank's query chunk over the whole ring.

    q [B, Hq, L, D], k / v [B, Hkv, L, D]: this rank's rows of the sequence.
    Returns the final fp32 (O, LSE) of this rank's query rows: (the LSE
    merge of) every visible chunk pair."""
    ops = ops or LibOps()
    ring = _P2P(group)
    o, lse = _partial_identity(q)
    held = (k, v)
    for step in range(ring.world):
        handle = ring.start(held) if step + 1 < ring.world else None
        _fwd_step(ops, ring.rank, step, ring.world, q, held, causal, scale, o, lse)
        if handle is not None:
            held = ring.finish(handle)
    return o, lse


def ring_attention_bwd(q, k, v, o, lse, d_o, causal=True, scale=None, group=None, ops=None):
    """Backward of the ring from this rank's saved final (O, LSE).

    Returns fp32 (dQ, dK, dV) of this rank's rows: dQ summed over every key
    chunk the rank's queries see, dK / dV summed over every query chunk that
    sees this rank's keys (gathered as the chunk travelled)."""
    ops = ops or LibOps()
    ring = _P2P(group)
    dq = torch.zeros(q.shape, dtype=torch.float32, device=q.device)
    held = (k, v, torch.zeros(k.shape, dtype=torch.float32, device=k.device),
            torch.zeros(v.shape, dtype=torch.float32, device=v.device))
    for step in range(ring.world):
        # the chunk's keys and values move on while this step computes; its
        # gradient accumulators once this step has added to them
        kv = ring.start(held[:2]) if step + 1 < ring.world else None
        _bwd_step(ops, ring.rank, step, ring.world, q, o, lse, d_o, held, causal, scale, dq)
        if ring.world == 1:
            break
        grads = ring.finish(ring.start(held[2:]))
        held = (ring.finish(kv) + grads) if kv is not None else (None, None) + grads
    return dq, held[2], held[3]


def tree_decode(q, k_shard, v_shard, chunk_len, scale=None, group=None, ops=None):
    """One decode step against a key/value cache sharded across ranks.

    Every rank holds the same q [B, Hq, 1, D] and its own shard [B, Hkv, Ns,
    D] of the cache; each computes its partial (split-KV decode and the
    one-pass merge inside the GPU), one all-gather exchanges the partials
    (B Hq (D + 1) fp32 values per rank), and each rank merges them in rank
    order.  Returns fp32 (O, LSE), identical on every rank."""
    import torch.distributed as dist
    ops = ops or LibOps()
    world = dist.get_world_size(group)
    o, lse = ops.decode(q, k_shard, v_shard, chunk_len, scale)
    o_all = [torch.empty_like(o) for _ in range(world)]
    l_all = [torch.empty_like(lse) for _ in range(world)]
    dist.all_gather(o_all, o.contiguous(), group=group)
    dist.all_gather(l_all, lse.contiguous(), group=group)
    return ops.tree_merge(torch.stack(o_all), torch.stack(l_all))


# ------------------------------------------------------ one-process driver
def ring_attention_fwd_sim(qs, ks, vs, causal=True, scale=None, ops=None):
    """All ranks of the ring in one process (lists of per-rank chunks, passed
    on by reference): the same steps as ring_attention_fwd."""
    ops = ops or LibOps()
    world = len(qs)
    outs = [_partial_identity(q) for q in qs]
    held = [(ks[r], vs[r]) for r in range(world)]
    for step in range(world):
        for r in range(world):
            _fwd_step(ops, r, step, world, qs[r], held[r], causal, scale, *outs[r])
        held = [held[(r - 1) % world] for r in range(world)]
    return outs


def ring_attention_bwd_sim(qs, ks, vs, os_, lses, d_os, causal=True, scale=None, ops=None):
    """The steps of ring_attention_bwd for all ranks in one process."""
    ops = ops or LibOps()
    world = len(qs)
    dqs = [torch.zeros(q.shape, dtype=torch.float32, device=q.device) for q in qs]
    held = [(ks[r], vs[r], torch.zeros(ks[r].shape, dtype=torch.float32, device=ks[r].device),
             torch.zeros(vs[r].shape, dtype=torch.float32, device=vs[r].device))
            for r in range(world)]
    for step in range(world):
        for r in range(world):
            _bwd_step(ops, r, step, world, qs[r], os_[r], lses[r], d_os[r], held[r], causal,
                      scale, dqs[r])
        held = [held[(r - 1) % world] for r in range(world)]
    return [(dqs[r], held[r][2], held[r][3]) for r in range(world)]


def tree_decode_sim(q, k_shards, v_shards, chunk_len, scale=None, ops=None):
    """tree_decode's steps for all ranks in one process: one partial per
    shard, merged in shard order."""
    ops = ops or LibOps()
    parts = [ops.decode(q, kc, vc, chunk_len, scale) for kc, vc in zip(k_shards, v_shards)]
    return ops.tree_merge(torch.stack([p_[0] for p_ in parts]), torch.stack([p_[1] for p_ in parts]))
