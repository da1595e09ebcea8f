"""BitDelta CPU oracle -- TEST INFRASTRUCTURE ONLY.

A plain fp64 C implementation (``bitdelta_oracle.c``) of what the fused
BitDelta path computes, plus this numpy shim.  Only ``tests/``, the smoke
check and the benchmark's CPU-baseline leg may import it; the product package
never does, and the two share no code.

What it follows: "BitDelta: Tek bir GPU kumesinden 14 Zen modeli sunmak"
(Hanzo blog, 2026-02-28), sections "Matematiksel temel" (eqs. (1)-(3)),
"Sunum mimarisi" (the conceptual fused_bitdelta_linear listing and the serving
pipeline) and "Altyapi ayrintilari" (the packed int8 sign storage and float32
alpha per output dimension), and section "MonoSoup" (the rank-r truncated-SVD
merge of several fine-tuned checkpoints of one base).

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(closed forms, brute force, hand-built bit patterns, special cases that reduce
to a numpy routine, and the page's printed sizes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bitdelta_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_vp = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP) into oracle/_build/liboracle.so."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "bitdelta_oracle.h")))
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall", "-Wextra",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_set_threads.argtypes = [ctypes.c_int]
            lib.oracle_set_threads.restype = ctypes.c_int
            lib.oracle_compress.argtypes = [_vp, _vp, _i64, _i64, ctypes.c_int, _vp, _vp]
            lib.oracle_compress.restype = ctypes.c_int
            lib.oracle_compress_rows.argtypes = [_vp, _vp, _i64, _i64, _vp, _i64, _vp, _vp]
            lib.oracle_compress_rows.restype = ctypes.c_int
            lib.oracle_unpack_signs.argtypes = [_vp, _i64, _i64, _vp]
            lib.oracle_unpack_signs.restype = ctypes.c_int
            lib.oracle_pack_signs.argtypes = [_vp, _i64, _i64, _vp]
            lib.oracle_pack_signs.restype = ctypes.c_int
            lib.oracle_reconstruct.argtypes = [_vp, _vp, _vp, ctypes.c_int, _i64, _i64, _vp]
            lib.oracle_reconstruct.restype = ctypes.c_int
            lib.oracle_linear_rows.argtypes = [_vp, _i64, _vp, _vp, _vp, ctypes.c_int, _i64, _i64, _vp, _i64,
                                               _vp]
            lib.oracle_linear_rows.restype = ctypes.c_int
            lib.oracle_route.argtypes = [_vp, _i64, _i32, _vp, _vp]
            lib.oracle_route.restype = _i64
            lib.oracle_linear_multi_rows.argtypes = [_vp, _i64, _vp, _i32, _vp, _vp, ctypes.c_int, _vp, _i64,
                                                     _i64, _vp, _i64, _vp]
            lib.oracle_linear_multi_rows.restype = ctypes.c_int
            lib.oracle_compressed_bytes.argtypes = [_i64, _i64, _i64]
            lib.oracle_compressed_bytes.restype = _i64
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def set_threads(n: int = 0) -> int:
    """Set the OpenMP thread count (0 keeps the default); returns the count in use."""
    return int(_load().oracle_set_threads(int(n)))


def compress(w_base_bits: np.ndarray, w_ft_bits: np.ndarray, per_row: bool):
    """(signs uint32 [d_out][d_in/32], alpha float32 [d_out] or [1])."""
    wb = _c(w_base_bits, np.uint16)
    wf = _c(w_ft_bits, np.uint16)
    d_out, d_in = wb.shape
    signs = np.zeros((d_out, d_in // 32), np.uint32)
    alpha = np.zeros(d_out if per_row else 1, np.float32)
    rc = _load().oracle_compress(_ptr(wb), _ptr(wf), d_out, d_in, int(per_row), _ptr(signs), _ptr(alpha))
    if rc != 0:
        raise ValueError("oracle_compress: bad arguments")
    return signs, alpha


def compress_rows(w_base_bits: np.ndarray, w_ft_bits: np.ndarray, rows: np.ndarray):
    """Per-row compression of the listed rows only: (signs [n][d_in/32], alpha [n])."""
    wb = _c(w_base_bits, np.uint16)
    wf = _c(w_ft_bits, np.uint16)
    d_out, d_in = wb.shape
    r = _c(rows, np.int64)
    signs = np.zeros((len(r), d_in // 32), np.uint32)
    alpha = np.zeros(len(r), np.float32)
    rc = _load().oracle_compress_rows(_ptr(wb), _ptr(wf), d_out, d_in, _ptr(r), len(r), _ptr(signs),
                                      _ptr(alpha))
    if rc != 0:
        raise ValueError("oracle_compress_rows: bad arguments")
    return signs, alpha


def unpack_signs(signs: np.ndarray, d_in: int) -> np.ndarray:
    s = _c(signs, np.uint32)
    d_out = s.shape[0]
    out = np.zeros((d_out, d_in), np.int8)
    if _load().oracle_unpack_signs(_ptr(s), d_out, d_in, _ptr(out)) != 0:
        raise ValueError("oracle_unpack_signs: bad arguments")
    return out


def pack_signs(s: np.ndarray) -> np.ndarray:
    a = _c(s, np.int8)
    d_out, d_in = a.shape
    out = np.zeros((d_out, d_in // 32), np.uint32)
    if _load().oracle_pack_signs(_ptr(a), d_out, d_in, _ptr(out)) != 0:
        raise ValueError("oracle_pack_signs: bad arguments")
    return out


def reconstruct(w_base_bits, signs, alpha, per_row: bool) -> np.ndarray:
    wb = _c(w_base_bits, np.uint16)
    d_out, d_in = wb.shape
    s = _c(signs, np.uint32)
    a = _c(alpha, np.float32)
    out = np.zeros((d_out, d_in), np.float64)
    if _load().oracle_reconstruct(_ptr(wb), _ptr(s), _ptr(a), int(per_row), d_out, d_in, _ptr(out)) != 0:
        raise ValueError("oracle_reconstruct: bad arguments")
    return out


def round_to_bf16(v: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of fp64 values rounded to nearest, ties to even, in
    one rounding.  bf16 keeps 8 significant bits down to 2^-126 and a fixed
    spacing of 2^-133 below it (its subnormals), so the rounding quantum of
    v = m 2^e (0.5 <= |m| < 1) is q = 2^max(e - 8, -133) and the result is
    rint(v / q) q (numpy's rint rounds halves to even; both steps are exact
    in fp64).  That value is a bf16 number, hence exact in fp32, whose upper
    16 bits are its pattern; magnitudes past the largest bf16 become inf
    through the same fp32 read-back."""
    v = np.asarray(v, np.float64)
    _, e = np.frexp(v)
    q = np.ldexp(1.0, np.maximum(e - 8, -133))
    r = np.rint(v / q) * q
    with np.errstate(over="ignore"):
        f = r.astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def materialize(w_base_bits, signs, alpha, per_row: bool) -> np.ndarray:
    """The variant's dense weights as bf16 bits: W_eff = W_base + alpha * s
    (section "Matematiksel temel", eq. (2)) in fp64, rounded once to bf16 --
    the weights a non-fused server would build before a standard matmul."""
    return round_to_bf16(reconstruct(w_base_bits, signs, alpha, per_row))


def linear(x_bits, w_base_bits, signs, alpha, per_row: bool, rows=None) -> np.ndarray:
    """fp64 y [T][len(rows)] (all rows when rows is None); the rows' signs
    and alpha are indexed by absolute row number."""
    x = _c(x_bits, np.uint16)
    wb = _c(w_base_bits, np.uint16)
    s = _c(signs, np.uint32)
    a = _c(alpha, np.float32)
    T = x.shape[0]
    d_out, d_in = wb.shape
    r = None if rows is None else _c(rows, np.int64)
    n = d_out if r is None else len(r)
    y = np.zeros((T, n), np.float64)
    rc = _load().oracle_linear_rows(_ptr(x), T, _ptr(wb), _ptr(s), _ptr(a), int(per_row), d_out, d_in,
                                    None if r is None else _ptr(r), n, _ptr(y))
    if rc != 0:
        raise ValueError("oracle_linear_rows: bad arguments")
    return y


def route(vid: np.ndarray, V: int):
    """(perm int32 [T], seg_off int32 [V+2], number of out-of-range ids)."""
    v = _c(vid, np.int32)
    T = len(v)
    perm = np.zeros(T, np.int32)
    seg = np.zeros(V + 2, np.int32)
    n_bad = _load().oracle_route(_ptr(v), T, V, _ptr(perm), _ptr(seg))
    if n_bad < 0:
        raise ValueError("oracle_route: bad arguments")
    return perm, seg, int(n_bad)


def linear_multi(x_bits, vid, signs_list, alpha_list, per_row: bool, w_base_bits, rows=None) -> np.ndarray:
    x = _c(x_bits, np.uint16)
    v = _c(vid, np.int32)
    wb = _c(w_base_bits, np.uint16)
    d_out, d_in = wb.shape
    V = len(signs_list)
    s_arrs = [_c(s, np.uint32) for s in signs_list]
    a_arrs = [_c(a, np.float32) for a in alpha_list]
    s_tab = (ctypes.c_void_p * max(V, 1))(*[_ptr(s) for s in s_arrs])
    a_tab = (ctypes.c_void_p * max(V, 1))(*[_ptr(a) for a in a_arrs])
    T = x.shape[0]
    r = None if rows is None else _c(rows, np.int64)
    n = d_out if r is None else len(r)
    y = np.zeros((T, n), np.float64)
    rc = _load().oracle_linear_multi_rows(_ptr(x), T, _ptr(v), V, ctypes.addressof(s_tab),
                                          ctypes.addressof(a_tab), int(per_row), _ptr(wb), d_out, d_in,
                                          None if r is None else _ptr(r), n, _ptr(y))
    if rc != 0:
        raise ValueError("oracle_linear_multi_rows: bad arguments")
    return y


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """fp64 values of bf16 bit patterns (the upper 16 bits of an fp32)."""
    return (np.ascontiguousarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def monosoup_merge_f64(w_base: np.ndarray, w_ft_list, rank: int) -> np.ndarray:
    """MonoSoup merge, section "MonoSoup" of the BitDelta post, in fp64: for
    each checkpoint the task vector Delta_i = W_i - W_base, its rank-`rank`
    truncated SVD tau_i = U_i[:, :r] diag(S_i[:r]) Vh_i[:r] (numpy's SVD as
    the library step), and W_merged = W_base + (1/k) * sum_i tau_i."""
    w_base = np.asarray(w_base, np.float64)
    acc = np.zeros_like(w_base)
    for w in w_ft_list:
        d = np.asarray(w, np.float64) - w_base
        if rank > 0:
            u, sv, vh = np.linalg.svd(d, full_matrices=False)
            acc += (u[:, :rank] * sv[:rank]) @ vh[:rank]
    return w_base + acc / len(w_ft_list)


def monosoup_merge(w_base_bits: np.ndarray, w_ft_bits_list, rank: int) -> np.ndarray:
    """``monosoup_merge_f64`` on bf16 weights (Delta_i is exact in fp64)."""
    return monosoup_merge_f64(bf16_to_f64(w_base_bits), [bf16_to_f64(w) for w in w_ft_bits_list], rank)


def compressed_bytes(d_out: int, d_in: int, n_alpha: int) -> int:
    return int(_load().oracle_compressed_bytes(d_out, d_in, n_alpha))
