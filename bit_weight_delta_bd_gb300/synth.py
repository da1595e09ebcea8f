"""Seeded synthetic inputs for the BitDelta path (shared by tests and bench).

This module only draws random numbers and rounds them to bf16; it holds none
of the method's arithmetic (no Delta, sign, alpha, packing or linear), so both
the CPU oracle and the CUDA path can take their inputs from it without sharing
any computation.

Distributions follow the BitDelta post ("BitDelta: Tek bir GPU kumesinden 14
Zen modeli sunmak", section "Matematiksel temel", the Laplace model
Delta_ij ~ Laplace(0, b)) and the workload shapes of the serving setup:

* ``W_base`` ~ N(0, 0.02) drawn in fp32, rounded to bf16 (RNE);
* ``Delta`` ~ Laplace(0, b) drawn in fp64; ``W_ft = bf16(W_base + Delta)``;
* ``x`` ~ N(0, 1) drawn in fp32, rounded to bf16;
* variant ids ~ Zipf(s = 1.1) over ranks 1..V, id = rank - 1, drawn by inverse
  CDF from uniforms (``searchsorted(..., side="right")``).

Draw order within one generator is W_base, Delta, x (then variant ids).
bf16 tensors are returned as their uint16 bit patterns.
"""
from __future__ import annotations

import numpy as np


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 (or fp64 via fp32) to bf16 with round-to-nearest-even."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def base_weight(rng: np.random.Generator, d_out: int, d_in: int, std: float = 0.02) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal((d_out, d_in), dtype=np.float32) * np.float32(std))


def finetuned_weight(rng: np.random.Generator, w_base_bits: np.ndarray, b: float) -> np.ndarray:
    """bf16(W_base + Laplace(0, b)) with the Laplace draw in fp64."""
    delta = rng.laplace(0.0, b, size=w_base_bits.shape)
    return f32_to_bf16_bits(bf16_bits_to_f32(w_base_bits).astype(np.float64) + delta)


def activations(rng: np.random.Generator, T: int, d_in: int) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal((T, d_in), dtype=np.float32))


def zipf_variant_ids(rng: np.random.Generator, T: int, V: int, s: float = 1.1) -> np.ndarray:
    ranks = np.arange(1, V + 1, dtype=np.float64)
    p = ranks ** (-s)
    cdf = np.cumsum(p / p.sum())
    cdf[-1] = 1.0
    u = rng.random(T)
    return np.minimum(np.searchsorted(cdf, u, side="right"), V - 1).astype(np.int32)


def single_problem(seed: int, d_out: int, d_in: int, T: int, b: float = 1e-3):
    """(W_base, W_ft, x) bf16 bit patterns for one linear; draw order W_base, Delta, x."""
    rng = np.random.default_rng(seed)
    wb = base_weight(rng, d_out, d_in)
    wf = finetuned_weight(rng, wb, b)
    x = activations(rng, T, d_in)
    return wb, wf, x


def multi_problem(seed: int, d_out: int, d_in: int, T: int, V: int, b_lo: float = 5e-4, b_hi: float = 2e-3):
    """(W_base, [W_ft_v], x, vid, b) for V variants sharing one W_base.

    The per-variant Laplace scales b_v ~ U[b_lo, b_hi] are drawn first, then
    W_base, then each variant's Delta in order, then x, then the Zipf ids.
    """
    rng = np.random.default_rng(seed)
    b = rng.uniform(b_lo, b_hi, size=V)
    wb = base_weight(rng, d_out, d_in)
    wfs = [finetuned_weight(rng, wb, float(b[v])) for v in range(V)]
    x = activations(rng, T, d_in)
    vid = zipf_variant_ids(rng, T, V)
    return wb, wfs, x, vid, b


def sample_rows(seed: int, d_out: int, n: int) -> np.ndarray:
    """A sorted seeded subset of row indices that always includes the first
    and the last row (so tile edges and the ragged tail are covered)."""
    rng = np.random.default_rng(seed + 7919)
    n = min(n, d_out)
    pick = rng.choice(d_out, size=n, replace=False)
    pick[0] = 0
    if n > 1:
        pick[1] = d_out - 1
    return np.unique(pick).astype(np.int64)


# ------------------------------------------------------------------------------------------
# On-device draws for workloads too large to draw on the host (the 8-layer slice).  Same
# distributions as above; torch's seeded CUDA generator; the Laplace draw is the inverse CDF
# of a uniform draw, in fp32.  Still no method arithmetic.

# (name, d_out, d_in) of the seven linears of one 70B-shaped decoder layer
SLICE_LINEARS = (("q", 8192, 8192), ("k", 1024, 8192), ("v", 1024, 8192), ("o", 8192, 8192),
                 ("gate", 28672, 8192), ("up", 28672, 8192), ("down", 8192, 28672))


def slice_seed(seed: int, layer: int, matrix: int, variant: int = -1) -> int:
    """Seed of one matrix's W_base (variant = -1) or of one variant's delta."""
    return seed * 1_000_003 + layer * 1009 + matrix * 101 + (variant + 1) * 7_919_993


def device_generator(seed: int, device):
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def device_base_weight(seed: int, d_out: int, d_in: int, device, std: float = 0.02):
    """bf16 W_base ~ N(0, std) drawn on `device` (fp32 draw, RNE to bf16)."""
    import torch

    g = device_generator(seed, device)
    return (torch.randn(d_out, d_in, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)


def device_finetuned_weight(seed: int, w_base, b: float):
    """bf16(W_base + Laplace(0, b)) drawn on W_base's device."""
    import torch

    g = device_generator(seed, w_base.device)
    # uniform on the open interval (0, 1): rand() may return 0, whose inverse CDF is infinite
    u = torch.rand(w_base.shape, generator=g, device=w_base.device, dtype=torch.float32)
    u = u * (1.0 - 2.0 ** -23) + 2.0 ** -24 - 0.5
    delta = -b * torch.sign(u) * torch.log1p(-2.0 * u.abs())
    return (w_base.float() + delta).to(torch.bfloat16)


def slice_variant_scales(seed: int, V: int, b_lo: float = 5e-4, b_hi: float = 2e-3) -> np.ndarray:
    return np.random.default_rng(seed).uniform(b_lo, b_hi, size=V)


def monosoup_checkpoints(seed: int, d_out: int, d_in: int, k: int, rank_signal: int,
                         sigma_hi: float = 4.0, sigma_lo: float = 1.0):
    """Inputs of a MonoSoup merge (section "MonoSoup" of the BitDelta post):
    W_base as ``base_weight`` and k fine-tuned checkpoints
    W_i = bf16(W_base + U_i diag(s) V_i^T), U_i [d_out][rank_signal] and
    V_i [d_in][rank_signal] standard normal scaled by 1/sqrt(rows) (nearly
    orthonormal columns), s log-spaced from sigma_hi down to sigma_lo: the
    few high-variance directions the post says fine-tuning moves a weight
    along, plus the bf16 rounding of W_i as the small remainder.  Draw order:
    W_base, then U_i, V_i per checkpoint.  Returns (w_base_bits, [w_i_bits])."""
    rng = np.random.default_rng(seed)
    wb = base_weight(rng, d_out, d_in)
    s = np.geomspace(sigma_hi, sigma_lo, rank_signal) if rank_signal > 0 else np.zeros(0)
    wb64 = bf16_bits_to_f32(wb).astype(np.float64)
    out = []
    for _ in range(k):
        u = rng.standard_normal((d_out, rank_signal)) / np.sqrt(d_out)
        v = rng.standard_normal((d_in, rank_signal)) / np.sqrt(d_in)
        out.append(f32_to_bf16_bits((wb64 + (u * s) @ v.T).astype(np.float32)))
    return wb, out


def monosoup_noisy_checkpoints(seed: int, d_out: int, d_in: int, k: int, rank_signal: int, b: float = 1e-3,
                               sigma_hi: float = 4.0, sigma_lo: float = 1.0):
    """MonoSoup inputs whose task vectors carry a noise floor of real size:
    W_i = bf16(W_base + U_i diag(s) V_i^T + L_i), the low-rank part as in
    ``monosoup_checkpoints`` and L_i ~ Laplace(0, b) elementwise (the delta
    model of section "Matematiksel temel"), which the post's truncation is
    meant to remove as noise.  Draw order: W_base, then U_i, V_i, L_i per
    checkpoint.  Returns (w_base_bits, [w_i_bits])."""
    rng = np.random.default_rng(seed)
    wb = base_weight(rng, d_out, d_in)
    s = np.geomspace(sigma_hi, sigma_lo, rank_signal) if rank_signal > 0 else np.zeros(0)
    wb64 = bf16_bits_to_f32(wb).astype(np.float64)
    out = []
    for _ in range(k):
        u = rng.standard_normal((d_out, rank_signal)) / np.sqrt(d_out)
        v = rng.standard_normal((d_in, rank_signal)) / np.sqrt(d_in)
        noise = rng.laplace(0.0, b, size=(d_out, d_in))
        out.append(f32_to_bf16_bits((wb64 + (u * s) @ v.T + noise).astype(np.float32)))
    return wb, out


def monosoup_spectrum_checkpoints(seed: int, d_out: int, d_in: int, k: int, s):
    """MonoSoup inputs with a prescribed spectrum: W_i = bf16(W_base + U_i
    diag(s) V_i^T) with U_i [d_out][len(s)] and V_i [d_in][len(s)] exactly
    orthonormal (the Q factors of standard normal matrices), so that the
    singular values of W_i - W_base are s up to the bf16 rounding of W_i
    (repeated values stay repeated to that level).  Draw order: W_base, then
    the two normal matrices per checkpoint.  Returns (w_base_bits,
    [w_i_bits])."""
    rng = np.random.default_rng(seed)
    wb = base_weight(rng, d_out, d_in)
    s = np.asarray(s, dtype=np.float64)
    wb64 = bf16_bits_to_f32(wb).astype(np.float64)
    out = []
    for _ in range(k):
        u, _r = np.linalg.qr(rng.standard_normal((d_out, len(s))))
        v, _r = np.linalg.qr(rng.standard_normal((d_in, len(s))))
        out.append(f32_to_bf16_bits((wb64 + (u * s) @ v.T).astype(np.float32)))
    return wb, out


def gaussian_test_matrix(seed: int, d_in: int, l: int) -> np.ndarray:
    """Standard normal fp32 [d_in][l]: the random test matrix a randomized
    range finder draws (here an input, so both sides see the same one)."""
    return np.random.default_rng(seed).standard_normal((d_in, l), dtype=np.float32)
