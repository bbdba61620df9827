"""ctypes binding of liblsx (include/lsx.h): argument marshalling only.

Every computation happens in the CUDA library; this module turns torch
tensors into ``lsx_tensor`` views, passes the current CUDA stream, and raises
``LsxError`` on a non-zero status.  There is no fallback: if the library is
missing the first call raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblsx.so")

LSX_BF16 = 0
LSX_F32 = 1

STATUS = {
    0: "LSX_OK", -1: "LSX_ERR_NULL", -2: "LSX_ERR_SHAPE", -3: "LSX_ERR_DTYPE",
    -4: "LSX_ERR_ALIGN", -5: "LSX_ERR_UNSUPPORTED", -6: "LSX_ERR_WORKSPACE",
    -7: "LSX_ERR_LAUNCH", -8: "LSX_ERR_TIMEOUT", -9: "LSX_ERR_DEVICE",
}


class LsxError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)} ({code})")


class LsxTensor(ctypes.Structure):
    _fields_ = [
        ("data", ctypes.c_void_p),
        ("dtype", ctypes.c_int32),
        ("reserved", ctypes.c_int32),
        ("B", ctypes.c_int64), ("H", ctypes.c_int64),
        ("N", ctypes.c_int64), ("D", ctypes.c_int64),
        ("stride_b", ctypes.c_int64), ("stride_h", ctypes.c_int64),
        ("stride_n", ctypes.c_int64),
    ]


_P = ctypes.POINTER(LsxTensor)
_VP = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int
_SZ = ctypes.c_size_t

# name -> (restype, argtypes), mirroring include/lsx.h
SIGNATURES = {
    "attn_chunk_fwd_workspace_size": (_SZ, [_P, _P]),
    "attn_chunk_fwd": (_INT, [_P, _P, _P, _I64, _I64, _INT, ctypes.c_float, _P, _P, _INT, _VP, _SZ, _VP]),
    "attn_merge": (_INT, [_P, _P, _P, _P, _P, _P, _VP]),
    "attn_tree_merge": (_INT, [_P, _I64, _P, _I64, _INT, _P, _P, _VP]),
    "attn_chunk_bwd_min_workspace_size": (_SZ, [_P, _P]),
    "attn_decode_tree_workspace_size": (_SZ, [_P, _P, _P, _I64]),
    "attn_decode_tree": (_INT, [_P, _P, _P, _P, _P, _I64, ctypes.c_float, _P, _P, _VP, _SZ, _VP]),
    "attn_block_sparse_fwd_workspace_size": (_SZ, [_P, _P]),
    "attn_block_sparse_fwd": (_INT, [_P, _P, _P, _VP, _INT, ctypes.c_float, _P, _P, _VP, _SZ, _VP]),
    "attn_block_sparse_bwd_workspace_size": (_SZ, [_P, _P]),
    "attn_block_sparse_bwd": (_INT, [_P, _P, _P, _P, _P, _P, _VP, _INT, ctypes.c_float, _P, _P, _P,
                                     _VP, _SZ, _VP]),
    "attn_chunk_bwd_workspace_size": (_SZ, [_P, _P]),
    "attn_chunk_bwd": (_INT, [_P, _P, _P, _P, _P, _P, _I64, _I64, _INT, ctypes.c_float,
                              _P, _P, _P, _INT, _VP, _SZ, _VP]),
    "attn_chunk_bwd_noalloc_max_bytes": (_SZ, []),
    "attn_chunk_bwd_noalloc": (_INT, [_P, _P, _P, _P, _P, _P, _I64, _I64, _INT, ctypes.c_float,
                                      _P, _P, _P, _INT, _VP]),
    "attn_chunked_fwd_workspace_size": (_SZ, [_P, _P, _I64, _INT]),
    "attn_chunked_fwd": (_INT, [_P, _P, _P, _I64, _INT, ctypes.c_float, _P, _P, _VP, _SZ, _VP]),
    "attn_chunked_bwd_workspace_size": (_SZ, [_P, _P, _I64, _INT]),
    "attn_chunked_bwd": (_INT, [_P, _P, _P, _P, _P, _P, _I64, _INT, ctypes.c_float,
                                _P, _P, _P, _VP, _SZ, _VP]),
    "attn_decode_workspace_size": (_SZ, [_P, _P, _I64]),
    "attn_decode": (_INT, [_P, _P, _P, _I64, ctypes.c_float, _P, _P, _VP, _SZ, _VP]),
    "lsx_sync_status": (_INT, [_VP]),
    "lsx_status_string": (ctypes.c_char_p, [_INT]),
    "lsx_set_wait_limit_ns": (None, [ctypes.c_uint64]),
    "lsx_set_deterministic": (None, [_INT]),
    "lsx_selftest_bounded_wait": (_INT, [_VP]),
    "lsx_schedule_stats": (_INT, [_I64, _I64, _I64, _I64, _INT, _INT, ctypes.POINTER(_I64)]),
    "lsx_trace_enable": (_INT, [_VP, _SZ]),
    "lsx_trace_used": (_SZ, []),
    "lsx_version": (ctypes.c_char_p, []),
    "lsx_timing_enable": (_INT, [_INT]),
    "lsx_timing_report": (_INT, [ctypes.c_char_p, _SZ]),
    "lsx_timing_reset": (_INT, []),
}

_lib = None


def load(path: str = LIB_PATH):
    """Load liblsx.so (built by build.py); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'` "
                "(there is no CPU fallback)")
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return LSX_BF16
    if t.dtype == torch.float32:
        return LSX_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def view(t: torch.Tensor | None) -> LsxTensor:
    """[B, H, N, D] tensor (D contiguous) or [B, H, N] LSE -> lsx_tensor."""
    v = LsxTensor()
    if t is None:
        return v
    if t.dim() == 3:
        b, h, n = t.shape
        sb, sh, sn = t.stride()
        d = 1
    elif t.dim() == 4:
        b, h, n, d = t.shape
        sb, sh, sn, sd = t.stride()
        if sd != 1 and d > 1:
            raise ValueError("the last dimension must be contiguous")
    else:
        raise ValueError("expected a [B, H, N, D] or [B, H, N] tensor")
    v.data = t.data_ptr()
    v.dtype = _dtype_code(t)
    v.B, v.H, v.N, v.D = b, h, n, d
    v.stride_b, v.stride_h, v.stride_n = sb, sh, sn
    return v


def stream_handle(stream: torch.cuda.Stream | None = None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def check(code: int, where: str) -> None:
    if code != 0:
        raise LsxError(code, where)
