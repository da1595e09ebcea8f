"""Host-side checks of the C ABI (no GPU needed): the library builds and
loads, exports every function include/bitdelta.h declares, and its argument
checks return the documented status before touching any device memory."""
import ctypes
import os
import re

import pytest
import torch

from bit_weight_delta_bd_gb300 import bitdelta as bd

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "bitdelta.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    __graft_entry__.build()
    return bd.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bd_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(bd.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(11):
        s = bd.status_string(code)
        assert s.startswith("BD_")
    assert bd.status_string(999) == "BD_ERR_UNKNOWN"
    assert bd.bd_version() == 10000


def test_bounds_checked_build_exports_every_declared_symbol(lib):
    """The bounds-checked variant (-DBD_DEBUG_BOUNDS) builds, exports the
    same functions and says it is that variant; the normal library says it is
    not."""
    from bit_weight_delta_bd_gb300 import build

    path = build.build(debug_bounds=True)
    blib = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(blib, name), name
    assert blib.bd_debug_bounds_enabled() == 1
    assert lib.bd_debug_bounds_enabled() == 0


def test_cuda_error_names(lib):
    assert lib.bd_cuda_error_string(0).decode() == "cudaSuccess"
    assert lib.bd_cuda_error_string(1).decode() == "cudaErrorInvalidValue"
    assert lib.bd_cuda_error_string(2).decode() == "cudaErrorMemoryAllocation"


@pytest.mark.skipif(torch.cuda.is_available(), reason="needs a machine without a usable GPU")
def test_failed_cuda_call_keeps_its_code(lib):
    """A call that passes every host check reaches the CUDA runtime, which
    fails here (no GPU): the status is BD_ERR_CUDA and the runtime's own code
    is kept for the thread and named in the Python error."""
    st = _linear(lib)
    assert st == bd.BD_ERR_CUDA
    code = lib.bd_last_cuda_error()
    assert code != 0 and lib.bd_cuda_error_string(code).decode().startswith("cudaError")
    with pytest.raises(bd.BitDeltaError) as e:
        bd._check(st, "bd_linear")
    assert e.value.cuda_error == code and lib.bd_cuda_error_string(code).decode() in str(e.value)


def test_workspace_sizes(lib):
    assert bd.bd_linear_workspace_size(4, 100, 256) >= 256
    # multi: error word + x of one token group sorted by variant
    assert bd.bd_linear_multi_workspace_size(64, 14, 8192, 8192) >= 1024 + 64 * 8192 * 2
    assert bd.bd_route_workspace_size(100, 14) >= 256
    pm = bd.bd_compress_workspace_size(28672, 8192, bd.BD_ALPHA_PER_MATRIX)
    pr = bd.bd_compress_workspace_size(28672, 8192, bd.BD_ALPHA_PER_ROW)
    assert pm >= 256 + 8 * (28672 // 8) and pr >= 256 and pm % 256 == 0


# Fake, never-dereferenced device addresses: every call below must be
# rejected by the host-side checks.
A = 1 << 40


def _linear(lib, x=A, T=4, w=A + (1 << 30), s=A + (2 << 30), a=A + (3 << 30), mode=1, d_out=16, d_in=256,
            y=A + (4 << 30), out=1, ws=A + (5 << 30), ws_bytes=4096):
    return lib.bd_linear(x, T, w, s, a, mode, d_out, d_in, y, out, ws, ws_bytes, None)


def test_linear_argument_checks(lib):
    assert _linear(lib, d_in=96) == bd.BD_ERR_UNSUPPORTED_SHAPE
    assert _linear(lib, d_in=0) == bd.BD_ERR_UNSUPPORTED_SHAPE
    assert _linear(lib, T=-1) == bd.BD_ERR_UNSUPPORTED_SHAPE
    assert _linear(lib, mode=3) == bd.BD_ERR_INVALID_ARG
    assert _linear(lib, out=5) == bd.BD_ERR_INVALID_ARG
    assert _linear(lib, x=A + 8) == bd.BD_ERR_MISALIGNED
    assert _linear(lib, y=A + 4) == bd.BD_ERR_MISALIGNED
    assert _linear(lib, ws=A + (5 << 30) + 64) == bd.BD_ERR_MISALIGNED
    assert _linear(lib, ws_bytes=8) == bd.BD_ERR_WORKSPACE
    assert _linear(lib, ws=0) == bd.BD_ERR_WORKSPACE
    assert _linear(lib, y=A) == bd.BD_ERR_INVALID_ARG  # y overlaps x
    assert _linear(lib, s=0) == bd.BD_ERR_INVALID_ARG
    assert _linear(lib, T=0) == bd.BD_OK  # empty batch: nothing to do
    assert _linear(lib, d_out=0) == bd.BD_OK


def test_compress_argument_checks(lib):
    ws = A + (5 << 30)
    c = lambda **k: lib.bd_compress(k.get("w", A), k.get("f", A + (1 << 30)), k.get("d_out", 8),  # noqa: E731
                                    k.get("d_in", 256), k.get("mode", 1), k.get("s", A + (2 << 30)),
                                    k.get("a", A + (3 << 30)), k.get("ws", ws), k.get("wsb", 4096), None)
    assert c(d_in=100) == bd.BD_ERR_UNSUPPORTED_SHAPE
    assert c(d_out=-1) == bd.BD_ERR_UNSUPPORTED_SHAPE
    assert c(mode=2) == bd.BD_ERR_INVALID_ARG
    assert c(w=A + 2) == bd.BD_ERR_MISALIGNED
    assert c(a=A + (3 << 30) + 2) == bd.BD_ERR_MISALIGNED
    assert c(s=A) == bd.BD_ERR_INVALID_ARG  # signs overlap w_base
    assert c(wsb=16) == bd.BD_ERR_WORKSPACE
    assert c(d_out=0) == bd.BD_OK


def test_multi_and_route_argument_checks(lib):
    tab = (ctypes.c_void_p * 2)(A + (2 << 30), A + (6 << 30))
    atab = (ctypes.c_void_p * 2)(A + (3 << 30), A + (7 << 30))
    m = lambda V=2, vid=A + (8 << 30), t=tab: lib.bd_linear_multi(  # noqa: E731
        A, 4, vid, V, ctypes.addressof(t), ctypes.addressof(atab), 1, A + (1 << 30), 16, 256, A + (4 << 30), 1,
        A + (5 << 30), 1 << 29, None)
    assert m(V=0) == bd.BD_ERR_INVALID_ARG
    assert m(V=65) == bd.BD_ERR_INVALID_ARG
    assert m(vid=A + (8 << 30) + 2) == bd.BD_ERR_MISALIGNED
    bad = (ctypes.c_void_p * 2)(A + (2 << 30) + 4, A + (6 << 30))
    assert m(t=bad) == bd.BD_ERR_MISALIGNED
    assert lib.bd_route(A, 10, -1, A + (1 << 30), A + (2 << 30), A + (5 << 30), 4096, None) == bd.BD_ERR_INVALID_ARG
    assert lib.bd_route(A, 10, 3, A, A + (2 << 30), A + (5 << 30), 4096, None) == bd.BD_ERR_INVALID_ARG  # perm = vid
    assert lib.bd_check_async(0, None) == bd.BD_ERR_WORKSPACE


def test_monosoup_argument_checks(lib):
    tab = (ctypes.c_void_p * 2)(A + (1 << 30), A + (2 << 30))
    ws = A + (5 << 30)
    need = lib.bd_monosoup_workspace_size(16, 256, 2, 4, 8)
    assert need >= 256 + 16 * 8 * 4 + 256 * 8 * 4

    def m(k=2, d_out=16, d_in=256, rank=4, l=8, q=1, om=A + (3 << 30), out=A + (4 << 30), t=tab, wsb=need,
          dtype=0):
        return lib.bd_monosoup_merge(A, ctypes.addressof(t), k, d_out, d_in, rank, l, q, om, out, dtype, ws, wsb,
                                     None)

    assert m(k=0) == bd.BD_ERR_INVALID_ARG
    assert m(l=65) == bd.BD_ERR_INVALID_ARG
    assert m(l=6) == bd.BD_ERR_INVALID_ARG  # l must be a multiple of 4
    assert m(om=A + (3 << 30) + 4) == bd.BD_ERR_MISALIGNED  # omega 16-byte aligned
    assert m(rank=9) == bd.BD_ERR_INVALID_ARG  # rank > l
    assert m(rank=-1) == bd.BD_ERR_INVALID_ARG
    assert m(q=17) == bd.BD_ERR_INVALID_ARG
    assert m(dtype=3) == bd.BD_ERR_INVALID_ARG
    assert m(d_in=100) == bd.BD_ERR_UNSUPPORTED_SHAPE
    assert m(d_out=-1) == bd.BD_ERR_UNSUPPORTED_SHAPE
    assert m(om=0) == bd.BD_ERR_INVALID_ARG  # rank > 0 needs the test matrix
    assert m(out=A + (4 << 30) + 8) == bd.BD_ERR_MISALIGNED
    bad = (ctypes.c_void_p * 2)(A + (1 << 30), A + (2 << 30) + 2)
    assert m(t=bad) == bd.BD_ERR_MISALIGNED
    assert m(out=A + (2 << 30)) == bd.BD_ERR_INVALID_ARG  # output overlaps a checkpoint
    assert m(wsb=need - 1) == bd.BD_ERR_WORKSPACE
    assert m(d_out=0) == bd.BD_OK
