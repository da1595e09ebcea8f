"""Thin ctypes binding of libbitdelta.so (include/bitdelta.h).

Argument marshalling only: every function here checks that its torch tensors
live on the current CUDA device with the expected dtype and layout, passes
their device pointers and the current CUDA stream to the C entry point of the
same name, and raises ``BitDeltaError`` on a non-OK status.  All arithmetic
runs in the library's sm_103a kernels; there is no fallback path, so a missing
or unloadable library raises instead of computing anything.

PyTorch is used for device memory and streams only.  bf16 buffers may be
passed as ``torch.bfloat16`` or as their ``torch.uint16``/``torch.int16`` bit
patterns.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# BD_LIBRARY selects another build of the library (the bounds-checked one,
# libbitdelta_bounds.so, in its test)
LIB_PATH = os.environ.get("BD_LIBRARY") or os.path.join(_HERE, "libbitdelta.so")

BD_OK = 0
BD_ERR_INVALID_ARG = 1
BD_ERR_UNSUPPORTED_SHAPE = 2
BD_ERR_MISALIGNED = 3
BD_ERR_BAD_VARIANT = 4
BD_ERR_NONFINITE = 5
BD_ERR_CUDA = 6
BD_ERR_TIMEOUT = 7
BD_ERR_WORKSPACE = 8
BD_ERR_DEVICE = 9
BD_ERR_BOUNDS = 10

BD_ALPHA_PER_MATRIX = 0
BD_ALPHA_PER_ROW = 1
BD_OUT_BF16 = 0
BD_OUT_F32 = 1
BD_MAX_VARIANTS = 64
BD_NOALLOC_MAX_ROWS = 262144

# Every symbol include/bitdelta.h declares.
EXPORTS = (
    "bd_version", "bd_status_string", "bd_last_cuda_error", "bd_cuda_error_string",
    "bd_compress_workspace_size", "bd_compress",
    "bd_linear_workspace_size", "bd_linear",
    "bd_linear_multi_workspace_size", "bd_linear_multi",
    "bd_route_workspace_size", "bd_route",
    "bd_debug_reconstruct", "bd_check_async", "bd_compress_noalloc", "bd_debug_bounds_check",
    "bd_debug_bounds_enabled",
    "bd_cache_create", "bd_cache_destroy", "bd_cache_set_source", "bd_cache_step", "bd_cache_release",
    "bd_cache_get_stats", "bd_cache_query", "bd_cache_debug_fail_load", "bd_materialize",
    "bd_monosoup_workspace_size", "bd_monosoup_merge",
)
BD_CACHE_SERVED = 0
BD_CACHE_BASE = 1
BD_CACHE_QUEUED = 2


class CacheStats(ctypes.Structure):
    """bd_cache_stats (include/bitdelta.h)."""
    _fields_ = [("steps", ctypes.c_int64), ("requests", ctypes.c_int64), ("hits", ctypes.c_int64),
                ("misses", ctypes.c_int64), ("queued", ctypes.c_int64), ("loads", ctypes.c_int64),
                ("evictions", ctypes.c_int64), ("bytes_loaded", ctypes.c_int64), ("slots", ctypes.c_int32),
                ("resident", ctypes.c_int32), ("pinned", ctypes.c_int32)]


class BitDeltaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        self.cuda_error = 0
        msg = f"{where}: {status_string(status)}"
        if self.status == BD_ERR_CUDA and _lib is not None:
            self.cuda_error = int(_lib.bd_last_cuda_error())
            msg += f" ({_lib.bd_cuda_error_string(self.cuda_error).decode()}, code {self.cuda_error})"
        super().__init__(msg)


_lib = None
_lock = threading.Lock()
_i64, _i32, _vp, _sz, _int = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libbitdelta.so (built by ``bit_weight_delta_bd_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"libbitdelta.so is not built ({path}); run __graft_entry__.build() first")
        lib = ctypes.CDLL(path)
        sig = {
            "bd_version": ([], _int),
            "bd_status_string": ([_int], ctypes.c_char_p),
            "bd_last_cuda_error": ([], _int),
            "bd_cuda_error_string": ([_int], ctypes.c_char_p),
            "bd_compress_workspace_size": ([_i64, _i64, _int], _sz),
            "bd_compress": ([_vp, _vp, _i64, _i64, _int, _vp, _vp, _vp, _sz, _vp], _int),
            "bd_linear_workspace_size": ([_i64, _i64, _i64], _sz),
            "bd_linear": ([_vp, _i64, _vp, _vp, _vp, _int, _i64, _i64, _vp, _int, _vp, _sz, _vp], _int),
            "bd_linear_multi_workspace_size": ([_i64, _i32, _i64, _i64], _sz),
            "bd_linear_multi": ([_vp, _i64, _vp, _i32, _vp, _vp, _int, _vp, _i64, _i64, _vp, _int, _vp, _sz, _vp],
                                _int),
            "bd_route_workspace_size": ([_i64, _i32], _sz),
            "bd_route": ([_vp, _i64, _i32, _vp, _vp, _vp, _sz, _vp], _int),
            "bd_debug_reconstruct": ([_vp, _vp, _vp, _int, _i64, _i64, _vp, _vp], _int),
            "bd_check_async": ([_vp, _vp], _int),
            "bd_debug_bounds_check": ([_vp], _int),
            "bd_debug_bounds_enabled": ([], _int),
            "bd_compress_noalloc": ([_vp, _vp, _i64, _i64, _int, _vp, _vp, _vp], _int),
            "bd_materialize": ([_vp, _vp, _vp, _int, _i64, _i64, _vp, _vp], _int),
            "bd_monosoup_workspace_size": ([_i64, _i64, _i32, _i32, _i32], _sz),
            "bd_monosoup_merge": ([_vp, _vp, _i32, _i64, _i64, _i32, _i32, _i32, _vp, _vp, _int, _vp, _sz, _vp],
                                  _int),
            "bd_cache_create": ([_vp, _sz, _sz, _i32, ctypes.c_double, _vp, ctypes.POINTER(_vp)], _int),
            "bd_cache_destroy": ([_vp], None),
            "bd_cache_set_source": ([_vp, _i32, _vp, _sz], _int),
            "bd_cache_step": ([_vp, _vp, _i64, _vp, _vp, _vp], _int),
            "bd_cache_release": ([_vp, _vp], _int),
            "bd_cache_get_stats": ([_vp, ctypes.POINTER(CacheStats)], _int),
            "bd_cache_debug_fail_load": ([_vp, _i64], _int),
            "bd_cache_query": ([_vp, _i32, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32),
                                ctypes.POINTER(ctypes.c_double)], _int),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
        return lib


def status_string(status: int) -> str:
    try:
        return load().bd_status_string(int(status)).decode()
    except RuntimeError:
        return f"status {status}"


def _check(status: int, where: str) -> None:
    if status != BD_OK:
        raise BitDeltaError(status, where)


_BF16_LIKE = (torch.bfloat16, torch.uint16, torch.int16)


def _ptr(t: torch.Tensor | None, name: str, dtypes=None, allow_none: bool = False) -> int | None:
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, not the current device")
    if dtypes is not None and t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _ws(ws: torch.Tensor) -> tuple[int, int]:
    if ws.dtype != torch.uint8:
        raise ValueError("workspace must be a torch.uint8 tensor")
    return _ptr(ws, "ws"), ws.numel()


def new_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zero-filled workspace (the library requires zeros before first use)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


# ------------------------------------------------------------------------------- sizes

def bd_version() -> int:
    return int(load().bd_version())


def bd_compress_workspace_size(d_out: int, d_in: int, alpha_mode: int) -> int:
    return int(load().bd_compress_workspace_size(d_out, d_in, alpha_mode))


def bd_linear_workspace_size(T: int, d_out: int, d_in: int) -> int:
    return int(load().bd_linear_workspace_size(T, d_out, d_in))


def bd_linear_multi_workspace_size(T: int, V: int, d_out: int, d_in: int) -> int:
    return int(load().bd_linear_multi_workspace_size(T, V, d_out, d_in))


def bd_route_workspace_size(T: int, V: int) -> int:
    return int(load().bd_route_workspace_size(T, V))


# ------------------------------------------------------------------------------- calls

def bd_compress(w_base, w_ft, alpha_mode, signs, alpha, ws, stream=None) -> None:
    d_out, d_in = w_base.shape
    if tuple(w_ft.shape) != (d_out, d_in):
        raise ValueError("w_ft shape differs from w_base")
    wsp, wsn = _ws(ws)
    _check(load().bd_compress(_ptr(w_base, "w_base", _BF16_LIKE), _ptr(w_ft, "w_ft", _BF16_LIKE), d_out, d_in,
                              int(alpha_mode), _ptr(signs, "signs", (torch.int32, torch.uint32)),
                              _ptr(alpha, "alpha", (torch.float32,)), wsp, wsn, _stream(stream)), "bd_compress")


def bd_compress_noalloc(w_base, w_ft, alpha_mode, signs, alpha, stream=None) -> None:
    """bd_compress without a workspace, for callers that cannot allocate
    device memory; the library keeps the scratch in a fixed device array
    (at most BD_NOALLOC_MAX_ROWS rows; calls that overlap on the GPU race)."""
    d_out, d_in = w_base.shape
    if tuple(w_ft.shape) != (d_out, d_in):
        raise ValueError("w_ft shape differs from w_base")
    _check(load().bd_compress_noalloc(_ptr(w_base, "w_base", _BF16_LIKE), _ptr(w_ft, "w_ft", _BF16_LIKE), d_out,
                                      d_in, int(alpha_mode), _ptr(signs, "signs", (torch.int32, torch.uint32)),
                                      _ptr(alpha, "alpha", (torch.float32,)), _stream(stream)),
           "bd_compress_noalloc")


def bd_linear(x, w_base, signs, alpha, alpha_mode, y, ws, stream=None) -> None:
    T, d_in = x.shape
    d_out = w_base.shape[0]
    out_dtype = BD_OUT_F32 if y.dtype == torch.float32 else BD_OUT_BF16
    wsp, wsn = _ws(ws)
    _check(load().bd_linear(_ptr(x, "x", _BF16_LIKE), T, _ptr(w_base, "w_base", _BF16_LIKE),
                            _ptr(signs, "signs", (torch.int32, torch.uint32)), _ptr(alpha, "alpha", (torch.float32,)),
                            int(alpha_mode), d_out, d_in, _ptr(y, "y", (torch.float32, torch.bfloat16)), out_dtype,
                            wsp, wsn, _stream(stream)), "bd_linear")


def bd_linear_multi(x, vid, signs_list, alpha_list, alpha_mode, w_base, y, ws, stream=None) -> None:
    T, d_in = x.shape
    d_out = w_base.shape[0]
    V = len(signs_list)
    if len(alpha_list) != V:
        raise ValueError("signs_list and alpha_list differ in length")
    s_tab = (ctypes.c_void_p * max(V, 1))(*[_ptr(s, "signs", (torch.int32, torch.uint32)) for s in signs_list])
    a_tab = (ctypes.c_void_p * max(V, 1))(*[_ptr(a, "alpha", (torch.float32,)) for a in alpha_list])
    out_dtype = BD_OUT_F32 if y.dtype == torch.float32 else BD_OUT_BF16
    wsp, wsn = _ws(ws)
    _check(load().bd_linear_multi(_ptr(x, "x", _BF16_LIKE), T, _ptr(vid, "vid", (torch.int32,)), V,
                                  ctypes.addressof(s_tab), ctypes.addressof(a_tab), int(alpha_mode),
                                  _ptr(w_base, "w_base", _BF16_LIKE), d_out, d_in,
                                  _ptr(y, "y", (torch.float32, torch.bfloat16)), out_dtype, wsp, wsn,
                                  _stream(stream)), "bd_linear_multi")


def bd_materialize(w_base, signs, alpha, alpha_mode, w_eff, stream=None) -> None:
    d_out, d_in = w_base.shape
    _check(load().bd_materialize(_ptr(w_base, "w_base", _BF16_LIKE), _ptr(signs, "signs", (torch.int32, torch.uint32)),
                                 _ptr(alpha, "alpha", (torch.float32,)), int(alpha_mode), d_out, d_in,
                                 _ptr(w_eff, "w_eff", _BF16_LIKE), _stream(stream)), "bd_materialize")


def bd_monosoup_workspace_size(d_out: int, d_in: int, k: int, rank: int, l: int) -> int:
    return int(load().bd_monosoup_workspace_size(d_out, d_in, k, rank, l))


def bd_monosoup_merge(w_base, w_ft_list, rank, l, power_iters, omega, w_merged, ws, stream=None) -> None:
    """W_merged = W_base + (1/k) sum_i truncated_SVD_rank(W_i - W_base); omega [d_in][l] fp32 Gaussian."""
    d_out, d_in = w_base.shape
    k = len(w_ft_list)
    tab = (ctypes.c_void_p * max(k, 1))(*[_ptr(w, "w_ft", _BF16_LIKE) for w in w_ft_list])
    out_dtype = BD_OUT_F32 if w_merged.dtype == torch.float32 else BD_OUT_BF16
    wsp, wsn = _ws(ws)
    _check(load().bd_monosoup_merge(_ptr(w_base, "w_base", _BF16_LIKE), ctypes.addressof(tab), k, d_out, d_in,
                                    int(rank), int(l), int(power_iters),
                                    _ptr(omega, "omega", (torch.float32,), allow_none=True),
                                    _ptr(w_merged, "w_merged", _BF16_LIKE + (torch.float32,)), out_dtype, wsp, wsn,
                                    _stream(stream)), "bd_monosoup_merge")


def bd_route(vid, V, perm, seg_off, ws, stream=None) -> None:
    T = vid.numel()
    wsp, wsn = _ws(ws)
    _check(load().bd_route(_ptr(vid, "vid", (torch.int32,)), T, int(V), _ptr(perm, "perm", (torch.int32,)),
                           _ptr(seg_off, "seg_off", (torch.int32,)), wsp, wsn, _stream(stream)), "bd_route")


def bd_debug_reconstruct(w_base, signs, alpha, alpha_mode, w_eff, stream=None) -> None:
    d_out, d_in = w_base.shape
    _check(load().bd_debug_reconstruct(_ptr(w_base, "w_base", _BF16_LIKE),
                                       _ptr(signs, "signs", (torch.int32, torch.uint32)),
                                       _ptr(alpha, "alpha", (torch.float32,)), int(alpha_mode), d_out, d_in,
                                       _ptr(w_eff, "w_eff", (torch.float32,)), _stream(stream)),
           "bd_debug_reconstruct")


def bd_debug_bounds_check() -> tuple[int, int]:
    """(status, kernel bits): BD_ERR_BOUNDS if a kernel of a bounds-checked
    build met an index outside its buffer since the last call; synchronises
    the device."""
    bits = ctypes.c_uint32(0)
    st = int(load().bd_debug_bounds_check(ctypes.byref(bits)))
    return st, int(bits.value)


def bd_debug_bounds_enabled() -> bool:
    return bool(load().bd_debug_bounds_enabled())


def bd_check_async(ws, stream=None) -> int:
    """Waits for the stream and returns (and clears) the asynchronous status."""
    wsp, _ = _ws(ws)
    return int(load().bd_check_async(wsp, _stream(stream)))


class DeltaCache:
    """The bd_cache_* entry points (delta cache of section "Altyapı ayrıntıları").

    ``arena`` is a torch.uint8 CUDA tensor the cache divides into slots of
    ``slot_bytes``; ``arena=None`` with ``n_slots`` runs the policy without
    any CUDA call (steps then report slot offsets).  Host sources are CPU
    tensors (page-locked for asynchronous copies); they are kept referenced
    here for as long as the cache lives."""

    def __init__(self, arena, slot_bytes: int, n_pinned: int, rate_decay: float = 1.0, copy_stream=None,
                 n_slots: int | None = None):
        lib = load()
        if arena is None:
            if n_slots is None:
                raise ValueError("a dry-run cache needs n_slots")
            ptr, nbytes, cs = None, int(n_slots) * int(slot_bytes), None
        else:
            if arena.dtype != torch.uint8:
                raise ValueError("arena must be a torch.uint8 tensor")
            ptr, nbytes = _ptr(arena, "arena"), arena.numel()
            cs = (copy_stream or torch.cuda.current_stream()).cuda_stream
        h = _vp()
        _check(lib.bd_cache_create(ptr, nbytes, int(slot_bytes), int(n_pinned), float(rate_decay), cs,
                                   ctypes.byref(h)), "bd_cache_create")
        self._h, self._lib, self.dry = h, lib, arena is None
        self._arena, self._sources = arena, {}

    def set_source(self, variant: int, host: torch.Tensor) -> None:
        if host.is_cuda or not host.is_contiguous():
            raise ValueError("a source is a contiguous CPU tensor")
        _check(self._lib.bd_cache_set_source(self._h, int(variant), host.data_ptr(),
                                             host.numel() * host.element_size()), "bd_cache_set_source")
        self._sources[int(variant)] = host

    def step(self, vids, stream=None):
        """Per request: (device address or slot offset, or None; state)."""
        import numpy as np

        v = np.ascontiguousarray(np.asarray(vids, dtype=np.int32))
        n = v.size
        delta = (_vp * max(n, 1))()
        state = np.zeros(max(n, 1), np.int32)
        st = None if self.dry else _stream(stream)
        _check(self._lib.bd_cache_step(self._h, v.ctypes.data, n, st, delta, state.ctypes.data), "bd_cache_step")
        # a served request's slot offset 0 (dry run) reads back from ctypes as None
        return [(delta[i] or 0) if state[i] == BD_CACHE_SERVED else None for i in range(n)], state[:n].copy()

    def release(self, stream=None) -> None:
        _check(self._lib.bd_cache_release(self._h, None if self.dry else _stream(stream)), "bd_cache_release")

    def stats(self) -> dict:
        out = CacheStats()
        _check(self._lib.bd_cache_get_stats(self._h, ctypes.byref(out)), "bd_cache_get_stats")
        return {name: getattr(out, name) for name, _ in CacheStats._fields_}

    def query(self, variant: int):
        r, pn, rate = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_double()
        _check(self._lib.bd_cache_query(self._h, int(variant), ctypes.byref(r), ctypes.byref(pn), ctypes.byref(rate)),
               "bd_cache_query")
        return bool(r.value), bool(pn.value), rate.value

    def debug_fail_load(self, n: int) -> None:
        """Test aid: the n-th load from now fails like a failed copy (bd_cache_debug_fail_load)."""
        _check(self._lib.bd_cache_debug_fail_load(self._h, int(n)), "bd_cache_debug_fail_load")

    def close(self) -> None:
        if self._h:
            self._lib.bd_cache_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
