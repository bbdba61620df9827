"""Python face of liblsx: the same entry points as include/lsx.h on torch tensors.

Shapes: q/o/d_o/dq are [B, H_q, N_q, D]; k/v/dk/dv are [B, H_kv, N_k, D]; an
LSE is [B, H, N] float32 (natural log).  All tensors live on the current CUDA
device; calls are enqueued on the current stream.  Outputs are allocated here
when not supplied (PyTorch is the allocator; the library itself never
allocates).
"""

from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import check, load, stream_handle, view


def _scale(scale):
    return -1.0 if scale is None else float(scale)


def _ws(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


def chunk_fwd(q, k, v, q_off=0, kv_off=0, causal=False, scale=None, out=None,
              lse=None, accumulate=False, out_dtype=None, workspace=None,
              use_workspace=True):
    """Partial (O, LSE) of one query chunk against one key/value chunk.

    With accumulate=True, ``out``/``lse`` must hold a partial over other keys
    and receive the merged result.  use_workspace=False reads V as stored
    (no scratch); otherwise a workspace for the key-contiguous V copy is
    allocated here unless one is given.
    """
    lib = load()
    b, h, n, d = q.shape
    if out is None:
        out = torch.empty((b, h, n, d), dtype=out_dtype or q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((b, h, n), dtype=torch.float32, device=q.device)
    vq, vk, vv, vo, vl = view(q), view(k), view(v), view(out), view(lse)
    ws_ptr, ws_n = None, 0
    if use_workspace:
        need = lib.attn_chunk_fwd_workspace_size(ctypes.byref(vq), ctypes.byref(vk))
        if need:
            if workspace is None:
                workspace = _ws(need, q.device)
            ws_ptr, ws_n = workspace.data_ptr(), workspace.numel()
    check(lib.attn_chunk_fwd(ctypes.byref(vq), ctypes.byref(vk), ctypes.byref(vv),
                             int(q_off), int(kv_off), int(bool(causal)), _scale(scale),
                             ctypes.byref(vo), ctypes.byref(vl), int(bool(accumulate)),
                             ws_ptr, ws_n, stream_handle()), "attn_chunk_fwd")
    return out, lse


def merge(o_a, lse_a, o_b, lse_b, out=None, lse_out=None):
    """LSE-weighted merge of two partials; out may be o_a (in place)."""
    lib = load()
    if out is None:
        out = torch.empty_like(o_a)
    if lse_out is None:
        lse_out = torch.empty_like(lse_a)
    va, la, vb, lb, vo, lo = (view(t) for t in (o_a, lse_a, o_b, lse_b, out, lse_out))
    check(lib.attn_merge(ctypes.byref(va), ctypes.byref(la), ctypes.byref(vb),
                         ctypes.byref(lb), ctypes.byref(vo), ctypes.byref(lo),
                         stream_handle()), "attn_merge")
    return out, lse_out


def tree_merge(o_parts, lse_parts, out=None, lse_out=None, out_dtype=None):
    """One-pass merge of k partials: o_parts [k, B, H, N, D], lse_parts [k, B, H, N]."""
    lib = load()
    k_parts = o_parts.shape[0]
    if out is None:
        out = torch.empty(o_parts.shape[1:], dtype=out_dtype or o_parts.dtype,
                          device=o_parts.device)
    if lse_out is None:
        lse_out = torch.empty(lse_parts.shape[1:], dtype=torch.float32, device=o_parts.device)
    vp, lp = view(o_parts[0]), view(lse_parts[0])
    vo, lo = view(out), view(lse_out)
    check(lib.attn_tree_merge(ctypes.byref(vp), int(o_parts.stride(0)), ctypes.byref(lp),
                              int(lse_parts.stride(0)), int(k_parts), ctypes.byref(vo),
                              ctypes.byref(lo), stream_handle()), "attn_tree_merge")
    return out, lse_out


def chunk_bwd(q, k, v, o, lse, d_o, q_off=0, kv_off=0, causal=False, scale=None,
              dq=None, dk=None, dv=None, accumulate=False, grad_dtype=None,
              workspace=None, use_copies=True):
    """dQ, dK, dV of one chunk pair from the saved final O and LSE.

    use_copies=False sizes the workspace at the minimum (delta rows only),
    which makes the kernels read Q, dO, K as stored."""
    lib = load()
    gd = grad_dtype or q.dtype
    dq = torch.empty(q.shape, dtype=gd, device=q.device) if dq is None else dq
    dk = torch.empty(k.shape, dtype=gd, device=q.device) if dk is None else dk
    dv = torch.empty(v.shape, dtype=gd, device=q.device) if dv is None else dv
    vs = [view(t) for t in (q, k, v, o, lse, d_o, dq, dk, dv)]
    size_fn = lib.attn_chunk_bwd_workspace_size if use_copies else \
        lib.attn_chunk_bwd_min_workspace_size
    need = size_fn(ctypes.byref(vs[0]), ctypes.byref(vs[1]))
    if workspace is None:
        workspace = _ws(need, q.device)
    check(lib.attn_chunk_bwd(*(ctypes.byref(x) for x in vs[:6]), int(q_off), int(kv_off),
                             int(bool(causal)), _scale(scale),
                             *(ctypes.byref(x) for x in vs[6:]), int(bool(accumulate)),
                             workspace.data_ptr(), workspace.numel(), stream_handle()),
          "attn_chunk_bwd")
    return dq, dk, dv


def chunked_fwd(q, k, v, chunk_len, causal=True, scale=None, out=None, lse=None,
                workspace=None):
    """Whole-sequence forward over chunk pairs in one persistent launch."""
    lib = load()
    b, h, n, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((b, h, n), dtype=torch.float32, device=q.device)
    vq, vk, vv, vo, vl = view(q), view(k), view(v), view(out), view(lse)
    need = lib.attn_chunked_fwd_workspace_size(ctypes.byref(vq), ctypes.byref(vk),
                                               int(chunk_len), int(bool(causal)))
    ws = workspace if workspace is not None else (_ws(need, q.device) if need else None)
    check(lib.attn_chunked_fwd(ctypes.byref(vq), ctypes.byref(vk), ctypes.byref(vv),
                               int(chunk_len), int(bool(causal)), _scale(scale),
                               ctypes.byref(vo), ctypes.byref(vl),
                               ws.data_ptr() if ws is not None else None,
                               ws.numel() if ws is not None else 0, stream_handle()),
          "attn_chunked_fwd")
    return out, lse


def chunked_bwd(q, k, v, o, lse, d_o, chunk_len, causal=True, scale=None,
                dq=None, dk=None, dv=None, workspace=None):
    """Whole-sequence backward from the saved O and LSE."""
    lib = load()
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    vs = [view(t) for t in (q, k, v, o, lse, d_o, dq, dk, dv)]
    need = lib.attn_chunked_bwd_workspace_size(ctypes.byref(vs[0]), ctypes.byref(vs[1]),
                                               int(chunk_len), int(bool(causal)))
    if workspace is None:
        workspace = _ws(need, q.device)
    check(lib.attn_chunked_bwd(*(ctypes.byref(x) for x in vs[:6]), int(chunk_len),
                               int(bool(causal)), _scale(scale),
                               *(ctypes.byref(x) for x in vs[6:]),
                               workspace.data_ptr(), workspace.numel(), stream_handle()),
          "attn_chunked_bwd")
    return dq, dk, dv


def _block_mask(mask, q, k):
    """uint8 [ceil(Lq/128), ceil(Lk/128)] contiguous on q's device."""
    nq, nk = -(-q.shape[2] // 128), -(-k.shape[2] // 128)
    if tuple(mask.shape) != (nq, nk):
        raise ValueError(f"block mask must be [{nq}, {nk}] (128 x 128 blocks)")
    return mask.to(device=q.device, dtype=torch.uint8).contiguous()


def block_sparse_fwd(q, k, v, block_mask, causal=False, scale=None, out=None, lse=None,
                     workspace=None):
    """Whole-sequence forward restricted to a 128 x 128 block mask."""
    lib = load()
    b, h, n, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((b, h, n), dtype=torch.float32, device=q.device)
    m = _block_mask(block_mask, q, k)
    vq, vk, vv, vo, vl = view(q), view(k), view(v), view(out), view(lse)
    need = lib.attn_block_sparse_fwd_workspace_size(ctypes.byref(vq), ctypes.byref(vk))
    ws = workspace if workspace is not None else _ws(need, q.device)
    check(lib.attn_block_sparse_fwd(ctypes.byref(vq), ctypes.byref(vk), ctypes.byref(vv),
                                    m.data_ptr(), int(bool(causal)), _scale(scale),
                                    ctypes.byref(vo), ctypes.byref(vl), ws.data_ptr(), ws.numel(),
                                    stream_handle()), "attn_block_sparse_fwd")
    return out, lse


def block_sparse_bwd(q, k, v, o, lse, d_o, block_mask, causal=False, scale=None,
                     dq=None, dk=None, dv=None, workspace=None):
    """Whole-sequence backward restricted to a 128 x 128 block mask."""
    lib = load()
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    m = _block_mask(block_mask, q, k)
    vs = [view(t) for t in (q, k, v, o, lse, d_o, dq, dk, dv)]
    need = lib.attn_block_sparse_bwd_workspace_size(ctypes.byref(vs[0]), ctypes.byref(vs[1]))
    ws = workspace if workspace is not None else _ws(need, q.device)
    check(lib.attn_block_sparse_bwd(*(ctypes.byref(x) for x in vs[:6]), m.data_ptr(),
                                    int(bool(causal)), _scale(scale),
                                    *(ctypes.byref(x) for x in vs[6:]), ws.data_ptr(),
                                    ws.numel(), stream_handle()), "attn_block_sparse_bwd")
    return dq, dk, dv


def decode_workspace_size(q, kc, chunk_len) -> int:
    lib = load()
    vq, vk = view(q), view(kc)
    return int(lib.attn_decode_workspace_size(ctypes.byref(vq), ctypes.byref(vk), int(chunk_len)))


def decode(q, kc, vc, chunk_len, scale=None, out=None, lse=None, workspace=None,
           out_dtype=None):
    """One query token per sequence against a key/value cache: split + tree merge."""
    lib = load()
    b, h, n, d = q.shape
    if out is None:
        out = torch.empty((b, h, n, d), dtype=out_dtype or q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((b, h, n), dtype=torch.float32, device=q.device)
    vq, vk, vv, vo, vl = view(q), view(kc), view(vc), view(out), view(lse)
    need = lib.attn_decode_workspace_size(ctypes.byref(vq), ctypes.byref(vk), int(chunk_len))
    if workspace is None:
        workspace = _ws(need, q.device)
    check(lib.attn_decode(ctypes.byref(vq), ctypes.byref(vk), ctypes.byref(vv), int(chunk_len),
                          _scale(scale), ctypes.byref(vo), ctypes.byref(vl),
                          workspace.data_ptr(), workspace.numel(), stream_handle()),
          "attn_decode")
    return out, lse


def decode_tree(q, pk, pv, sk, sv, chunk_len, scale=None, out=None, lse=None, workspace=None,
                out_dtype=None):
    """One decode step of B branches sharing the prefix cache (pk, pv
    [1, Hkv, Np, D]); sk, sv [B, Hkv, Ns, D] are the branches' own suffixes
    (None when there are none).  The prefix is read once per branch group."""
    lib = load()
    b, h, n, d = q.shape
    if out is None:
        out = torch.empty((b, h, n, d), dtype=out_dtype or q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((b, h, n), dtype=torch.float32, device=q.device)
    vq, vpk, vpv, vo, vl = view(q), view(pk), view(pv), view(out), view(lse)
    vsk = view(sk) if sk is not None else None
    vsv = view(sv) if sv is not None else None
    rs = (lambda t: ctypes.byref(t) if t is not None else None)
    need = lib.attn_decode_tree_workspace_size(ctypes.byref(vq), ctypes.byref(vpk), rs(vsk),
                                               int(chunk_len))
    if workspace is None:
        workspace = _ws(need, q.device)
    check(lib.attn_decode_tree(ctypes.byref(vq), ctypes.byref(vpk), ctypes.byref(vpv), rs(vsk),
                               rs(vsv), int(chunk_len), _scale(scale), ctypes.byref(vo),
                               ctypes.byref(vl), workspace.data_ptr(), workspace.numel(),
                               stream_handle()), "attn_decode_tree")
    return out, lse


def sync_status(stream=None) -> int:
    """Synchronise, return and clear the device status word (0 = ok)."""
    return int(load().lsx_sync_status(stream_handle(stream)))


def set_wait_limit_ns(ns: int) -> None:
    load().lsx_set_wait_limit_ns(int(ns))


def set_deterministic(on: bool) -> None:
    """Select the backward's dQ reduction order (lsx_set_deterministic):
    False (default) = fused dK/dV/dQ kernel adding dQ with fp32 reduce-adds,
    True = owner-computes dQ kernel, bitwise repeatable."""
    load().lsx_set_deterministic(1 if on else 0)


def selftest_bounded_wait() -> None:
    check(load().lsx_selftest_bounded_wait(stream_handle()), "lsx_selftest_bounded_wait")


def schedule_stats(B, H, N, chunk_len, causal, n_workers):
    """(makespan, ideal, total) in key tiles of the forward schedule (host only)."""
    out = (ctypes.c_int64 * 3)()
    check(load().lsx_schedule_stats(int(B), int(H), int(N), int(chunk_len), int(bool(causal)),
                                    int(n_workers), out), "lsx_schedule_stats")
    return int(out[0]), int(out[1]), int(out[2])


def status_string(code: int) -> str:
    return load().lsx_status_string(int(code)).decode()


def version() -> str:
    return load().lsx_version().decode()
