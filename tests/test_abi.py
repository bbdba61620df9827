"""CPU-side checks of the C ABI: the library loads, exports every symbol that
include/lsx.h declares, and rejects bad arguments before touching a device.
No call here launches a kernel."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lsx.h")


@pytest.fixture(scope="module")
def lib():
    from long_sequence_exact_gb300 import build, _lib
    build.build()
    return _lib.load()


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[\w\*\s]+?\b((?:attn|lsx)_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("attn_chunk_fwd", "attn_merge", "attn_tree_merge", "attn_chunk_bwd",
                 "attn_chunked_fwd", "attn_chunked_bwd", "attn_decode", "lsx_sync_status"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"liblsx.so does not export {name}"


def test_binding_covers_every_declared_symbol():
    from long_sequence_exact_gb300 import _lib
    assert set(declared_functions()) <= set(_lib.SIGNATURES)


def test_status_strings_and_version(lib):
    assert lib.lsx_version().decode().startswith("lsx")
    for code in range(0, -10, -1):
        assert lib.lsx_status_string(code)
    assert lib.lsx_status_string(-8).decode() == "device-side bounded wait ran out"


def _t(b=1, h=2, n=128, d=128, dtype=0, ptr=0x10000, strides=None):
    from long_sequence_exact_gb300._lib import LsxTensor
    t = LsxTensor()
    t.data = ptr
    t.dtype = dtype
    t.B, t.H, t.N, t.D = b, h, n, d
    sb, sh, sn = strides or (h * n * d, n * d, d)
    t.stride_b, t.stride_h, t.stride_n = sb, sh, sn
    return t


def _lse(b=1, h=2, n=128, ptr=0x20000):
    return _t(b, h, n, 1, 1, ptr, (h * n, n, 1))


R = ctypes.byref


def test_fwd_rejects_bad_arguments_before_any_launch(lib):
    q, k, v, o, l = _t(), _t(), _t(), _t(), _lse()
    fwd = lambda *a: lib.attn_chunk_fwd(*a, 0, 0, 1, -1.0, R(o), R(l), 0, None, 0, None)  # noqa
    assert lib.attn_chunk_fwd(None, R(k), R(v), 0, 0, 1, -1.0, R(o), R(l), 0, None, 0, None) == -1
    assert fwd(R(_t(d=96)), R(_t(d=96)), R(_t(d=96))) in (-5, -2)
    assert fwd(R(q), R(_t(d=64)), R(v)) == -2               # D mismatch
    assert fwd(R(_t(h=3)), R(k), R(v)) == -2                # Hq % Hkv != 0
    assert fwd(R(q), R(_t(dtype=1)), R(v)) == -3            # mixed dtypes
    assert fwd(R(_t(ptr=0x10008)), R(k), R(v)) == -4        # misaligned base
    assert fwd(R(_t(strides=(128 * 130, 130 * 128, 130 + 2))), R(k), R(v)) == -4
    bad_l = _lse()
    bad_l.dtype = 0
    assert lib.attn_chunk_fwd(R(q), R(k), R(v), 0, 0, 1, -1.0, R(o), R(bad_l), 0, None, 0,
                              None) == -3
    assert lib.attn_chunk_fwd(R(q), R(k), R(v), -1, 0, 1, -1.0, R(o), R(l), 0, None, 0,
                              None) == -2


def test_bwd_requires_workspace(lib):
    q, k, v, o, l, do, dq, dk, dv = (_t(), _t(), _t(), _t(), _lse(), _t(), _t(), _t(), _t())
    need = lib.attn_chunk_bwd_min_workspace_size(R(q), R(k))
    assert need >= 2 * 128 * 4
    # the full size adds the key-contiguous copy of K (2 heads x 128 x 128 bf16)
    assert lib.attn_chunk_bwd_workspace_size(R(q), R(k)) >= need + 2 * 128 * 128 * 2
    rc = lib.attn_chunk_bwd(R(q), R(k), R(v), R(o), R(l), R(do), 0, 0, 1, -1.0, R(dq), R(dk),
                            R(dv), 0, None, 0, None)
    assert rc == -6
    rc = lib.attn_chunk_bwd(R(q), R(k), R(v), R(o), R(l), R(do), 0, 0, 1, -1.0, R(dq), R(dk),
                            R(dv), 0, ctypes.c_void_p(0x40000), need - 1, None)
    assert rc == -6


def test_merge_and_tree_merge_validation(lib):
    a, b, o = _t(dtype=1), _t(dtype=1), _t(dtype=1)
    la, lb, lo = _lse(), _lse(), _lse()
    assert lib.attn_merge(R(a), R(la), R(_t(n=64, dtype=1)), R(lb), R(o), R(lo), None) == -2
    assert lib.attn_merge(R(a), R(_lse(n=64)), R(b), R(lb), R(o), R(lo), None) == -2
    assert lib.attn_tree_merge(R(a), 0, R(la), 0, 0, R(o), R(lo), None) == -5
    assert lib.attn_tree_merge(R(a), 0, R(la), 0, 5000, R(o), R(lo), None) == -5


def test_decode_validation(lib):
    q = _t(b=2, h=8, n=1)
    kc = _t(b=2, h=1, n=4096)
    o, l = _t(b=2, h=8, n=1), _lse(b=2, h=8, n=1)
    assert lib.attn_decode(R(_t(b=2, h=16, n=1)), R(kc), R(kc), 4096, -1.0, R(_t(b=2, h=16, n=1)),
                           R(_lse(b=2, h=16, n=1)), None, 0, None) == -5   # group of 16
    assert lib.attn_decode(R(q), R(kc), R(kc), 100, -1.0, R(o), R(l), None, 0, None) == -5
    assert lib.attn_decode(R(q), R(kc), R(kc), 4096, -1.0, R(o), R(l), None, 0, None) == -6


def test_trace_buffer_validation(lib):
    # host-side bookkeeping only: nothing is launched
    assert lib.lsx_trace_enable(ctypes.c_void_p(0x10004), 4096) == -4  # not 8-byte aligned
    assert lib.lsx_trace_enable(None, 0) == 0
    assert lib.lsx_trace_used() == 0
