"""attn_chunk_bwd_noalloc: the backward for callers that cannot allocate
device memory at the call (an extension inside a host application that owns
the memory pool, a loop that forbids allocation after start-up).  It must give
the same gradients as attn_chunk_bwd, whose workspace the caller provides,
call after call, although every call reuses one fixed array in the library.

Collected last on purpose (file name), so a failure here comes after every
other test has run; it also passes alone in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

import long_sequence_exact_gb300 as lsx
from long_sequence_exact_gb300 import _lib
from long_sequence_exact_gb300.inputs import random_tensor
from helpers import TOL_FP32, TOL_GRAD_REL, f64, rel_fro

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _noalloc(q, k, v, o, lse, d_o, q_off, kv_off, causal, grad_dtype):
    lib = _lib.load()
    dq = torch.full(q.shape, float("nan"), dtype=grad_dtype, device=DEV)
    dk = torch.full(k.shape, float("nan"), dtype=grad_dtype, device=DEV)
    dv = torch.full(v.shape, float("nan"), dtype=grad_dtype, device=DEV)
    vs = [_lib.view(t) for t in (q, k, v, o, lse, d_o, dq, dk, dv)]
    rc = lib.attn_chunk_bwd_noalloc(*(ctypes.byref(x) for x in vs[:6]), q_off, kv_off,
                                    int(causal), -1.0, *(ctypes.byref(x) for x in vs[6:]),
                                    0, _lib.stream_handle())
    assert rc == 0, _lib.STATUS.get(rc, rc)
    return dq, dk, dv


CASES = [
    # B, Hq, Hkv, Lq, Lk, D, q_off, kv_off, causal, dtype
    (1, 4, 2, 640, 640, 128, 0, 0, True, torch.bfloat16),
    (2, 2, 2, 300, 500, 64, 200, 0, True, torch.bfloat16),
    (1, 2, 2, 256, 256, 64, 0, 0, False, torch.float32),
]


def _problem(case, seed):
    b, hq, hkv, lq, lk, d, q_off, kv_off, causal, dt = case
    amp = 0.5
    q = random_tensor((b, hq, lq, d), seed, amp, dtype=dt, device=DEV)
    k = random_tensor((b, hkv, lk, d), seed + 1, amp, dtype=dt, device=DEV)
    v = random_tensor((b, hkv, lk, d), seed + 2, dtype=dt, device=DEV)
    d_o = random_tensor((b, hq, lq, d), seed + 3, dtype=dt, device=DEV)
    o, lse = lsx.chunk_fwd(q, k, v, q_off, kv_off, causal)
    return (q, k, v, o, lse, d_o, q_off, kv_off, causal), dt


def test_noalloc_matches_workspace_backward_on_consecutive_calls():
    # several calls in a row, different shapes, each checked against the
    # entry point with a caller workspace
    for rep in range(2):
        for n, case in enumerate(CASES):
            args, dt = _problem(case, seed=100 * rep + 10 * n)
            got = _noalloc(*args, grad_dtype=dt)
            ref = lsx.chunk_bwd(*args, grad_dtype=dt)
            torch.cuda.synchronize()
            assert lsx.sync_status() == 0
            for g, r in zip(got, ref):
                gg, rr = f64(g), f64(r)
                assert not np.any(np.isnan(gg))
                if dt == torch.float32:
                    assert np.max(np.abs(gg - rr)) <= TOL_FP32
                else:
                    assert rel_fro(gg, rr) <= TOL_GRAD_REL


def test_noalloc_rejects_problems_beyond_its_array():
    lib = _lib.load()
    cap = lib.attn_chunk_bwd_noalloc_max_bytes()
    assert cap == 16 << 20
    rows = cap // 4 + 1024  # more query rows than the array holds
    q = _lib.LsxTensor()
    q.data, q.dtype, q.B, q.H, q.N, q.D = 0x1000, 0, 1, 1, rows, 128
    q.stride_b, q.stride_h, q.stride_n = rows * 128, rows * 128, 128
    z = _lib.LsxTensor()
    rc = lib.attn_chunk_bwd_noalloc(ctypes.byref(q), ctypes.byref(q), ctypes.byref(q),
                                    ctypes.byref(q), ctypes.byref(z), ctypes.byref(q), 0, 0, 1,
                                    -1.0, ctypes.byref(q), ctypes.byref(q), ctypes.byref(q), 0,
                                    None)
    assert rc == -6  # LSX_ERR_WORKSPACE, nothing launched
