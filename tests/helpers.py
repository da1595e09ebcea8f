"""Shared test helpers: device transfer of bf16 bit patterns and the
tolerance checks of the linear outputs.

Tolerances (from the BitDelta serving targets): linear outputs against the
fp64 oracle must have relative Frobenius error <= 5e-3 and max abs error
<= 2e-2.  For bf16 outputs the elementwise bound is 2e-2 + half a bf16 ulp of
the exact value, because rounding the exact result to bf16 alone already
reaches ~2e-2 when |y| ~ 8.  fp32 outputs must in addition meet the fp32
dot-product bound (n + 4) * 2^-22 * sum_j |x_j| (|w_j| + alpha): fp32
accumulation in any order keeps the error under (n + 4) * 2^-24 times that
sum when every addition rounds to nearest; the factor 4 of slack covers
tensor-core accumulators that truncate instead of rounding.  The prefill path
(T > 64) rounds W_eff to bf16 before its contraction, which adds up to
2^-9 * |x_j| * (|w_j| + alpha) per term to that bound.  The multi-variant
kernel computes sum_j x_j s_j as 2 sum_j x_j v_j - C with |v_j| <= 9 and
C = sum_j x_j c_j, 0 <= c_j <= 17, itself an fp32 sum (an exact recoding of
the sign operand), so its bound weighs alpha by 2 * 9 + 17 / 4 + 1 < 24
instead of 1.
"""
from __future__ import annotations

import numpy as np
import torch

from bit_weight_delta_bd_gb300 import synth

REL_FRO = 5e-3
MAX_ABS = 2e-2


def to_dev(a: np.ndarray, dev) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev)
    if a.dtype == np.uint32:
        return torch.from_numpy(a.view(np.int32)).to(dev)
    return torch.from_numpy(a).to(dev)


def u32(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint32)


def bf16_half_ulp(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1e-30)))
    return np.where(a > 0, 2.0 ** (e - 8), 0.0)


def y_host(y: torch.Tensor) -> np.ndarray:
    return y.float().cpu().numpy().astype(np.float64)


def check_linear(y_gpu: np.ndarray, y_ref: np.ndarray, bf16_out: bool, bound: np.ndarray | None = None,
                 what: str = ""):
    assert y_gpu.shape == y_ref.shape, (y_gpu.shape, y_ref.shape)
    assert np.all(np.isfinite(y_gpu)), what
    err = y_gpu - y_ref
    fro = np.linalg.norm(err) / max(np.linalg.norm(y_ref), 1e-30)
    assert fro <= REL_FRO, f"{what}: relative Frobenius {fro:.3e}"
    if bf16_out:
        lim = MAX_ABS + bf16_half_ulp(y_ref)
        bad = np.abs(err) > lim
        assert not bad.any(), f"{what}: {bad.sum()} elements above 2e-2 + ulp/2 (max {np.abs(err).max():.3e})"
    else:
        m = np.abs(err).max() if err.size else 0.0
        assert m <= MAX_ABS, f"{what}: max abs {m:.3e}"
        if bound is not None:
            over = np.abs(err) > bound
            assert not over.any(), f"{what}: {over.sum()} elements above the fp32 accumulation bound"
    return fro


PREFILL_MIN_T = 65  # bd_linear runs the tensor-core prefill GEMM from this many tokens on


def fp32_bound(x_bits, wb_bits, alpha, per_row: bool, rows=None, weff_bf16: bool = False) -> np.ndarray:
    """(n + 4) * 2^-22 * sum_j |x_j| (|w_j| + alpha) for the listed rows
    (plus 2^-9 times the same sum when W_eff is rounded to bf16)."""
    x = np.abs(synth.bf16_bits_to_f32(x_bits).astype(np.float64))
    wb = wb_bits if rows is None else wb_bits[rows]
    w = np.abs(synth.bf16_bits_to_f32(wb).astype(np.float64))
    a = np.asarray(alpha, np.float64)
    if per_row:
        a = a if rows is None else a[rows]
        a = np.broadcast_to(a, (w.shape[0],))
    else:
        a = np.full(w.shape[0], float(a[0]))
    s = x @ w.T + x.sum(axis=1)[:, None] * a[None, :]
    n = wb.shape[1]
    return ((n + 4) * 2.0 ** -22 + (2.0 ** -9 if weff_bf16 else 0.0)) * s + 1e-30


def fp32_bound_multi(x_bits, wb_bits, alphas, vid, rows, sign_weight: float = 24.0) -> np.ndarray:
    """Per-token form of fp32_bound for the multi-variant kernel:
    (n + 4) * 2^-22 * sum_j |x_j| (|w_j| + sign_weight * alpha_v(t)), alpha_v of
    the token's variant (0 for base-model tokens); alphas[v] holds the
    per-row alpha of the listed rows."""
    x = np.abs(synth.bf16_bits_to_f32(x_bits).astype(np.float64))
    w = np.abs(synth.bf16_bits_to_f32(wb_bits[rows]).astype(np.float64))
    a = np.zeros((x.shape[0], len(rows)))
    for t, v in enumerate(np.asarray(vid)):
        if 0 <= v < len(alphas):
            a[t] = np.asarray(alphas[v], np.float64)
    s = x @ w.T + sign_weight * x.sum(axis=1)[:, None] * a
    return (wb_bits.shape[1] + 4) * 2.0 ** -22 * s + 1e-30
