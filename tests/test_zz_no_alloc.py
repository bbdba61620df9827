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
from helpers import TOL_FP32, TOL_GRAD_REL, check_tiles, f64, oracle_bwd_rows, rel_fro

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


@pytest.mark.parametrize("grad_dtype", [torch.bfloat16, torch.float32])
def test_noalloc_delta_only_branch_matches_oracle(grad_dtype):
    # 65,536 query rows at d = 128: the row sums fit the fixed array (256 KiB)
    # but the fp32 dQ accumulator and the operand copies (32 MiB) do not, so
    # the call runs the backward without them: the two owner kernels for a
    # bf16 dq, the fused kernel adding straight into an f32 dq.  Two calls
    # in a row (different inputs), each against the oracle over every row
    # and against the workspace entry point given the same minimum size.
    lib = _lib.load()
    b, hq, hkv, n, d = 1, 4, 2, 16384, 128
    q0 = torch.empty((b, hq, n, d), dtype=torch.bfloat16, device=DEV)
    k0 = torch.empty((b, hkv, n, d), dtype=torch.bfloat16, device=DEV)
    vq, vk = _lib.view(q0), _lib.view(k0)
    cap = lib.attn_chunk_bwd_noalloc_max_bytes()
    assert lib.attn_chunk_bwd_min_workspace_size(ctypes.byref(vq), ctypes.byref(vk)) <= cap
    assert lib.attn_chunk_bwd_workspace_size(ctypes.byref(vq), ctypes.byref(vk)) > cap
    for rep in range(2):
        seed = 900 + 10 * rep
        q = random_tensor((b, hq, n, d), seed, 0.5, device=DEV)
        k = random_tensor((b, hkv, n, d), seed + 1, 0.5, device=DEV)
        v = random_tensor((b, hkv, n, d), seed + 2, device=DEV)
        d_o = random_tensor((b, hq, n, d), seed + 3, device=DEV)
        o, lse = lsx.chunk_fwd(q, k, v, 0, 0, True)
        got = _noalloc(q, k, v, o, lse, d_o, 0, 0, True, grad_dtype)
        ws = lsx.chunk_bwd(q, k, v, o, lse, d_o, 0, 0, True, grad_dtype=grad_dtype,
                           use_copies=False)
        torch.cuda.synchronize()
        assert lsx.sync_status() == 0
        ref = oracle_bwd_rows(f64(q), f64(k), f64(v), f64(d_o), 0, 0, True, np.arange(n))
        for name, g, w_, r in zip(("dQ", "dK", "dV"), got, ws, ref):
            gg = f64(g)
            assert not np.any(np.isnan(gg)), name
            assert rel_fro(gg, r) <= TOL_GRAD_REL, name
            check_tiles(gg, r, name)
            # same kernels as the workspace call; dQ's fp32 adds land in run order
            assert rel_fro(gg, f64(w_)) <= (2e-3 if name == "dQ" else 1e-6), name


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
