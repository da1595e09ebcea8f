"""Pins of the CPU oracle to what the BitDelta post and the mathematics fix.

Nothing here compares the oracle with itself: every check is a closed form, a
brute-force search, an exact rational computation, a hand-built bit pattern, a
value the post prints, or a special case that reduces to a numpy routine.
Source: "BitDelta: Tek bir GPU kumesinden 14 Zen modeli sunmak" (Hanzo blog,
2026-02-28), sections "Matematiksel temel", "Sunum mimarisi" and
"Altyapi ayrintilari".
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from bit_weight_delta_bd_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bits(values) -> np.ndarray:
    """Exact bf16 bit patterns of values that bf16 represents exactly."""
    f = np.asarray(values, dtype=np.float32)
    b = synth.f32_to_bf16_bits(f)
    assert np.array_equal(synth.bf16_bits_to_f32(b), f), "test value not exact in bf16"
    return b


def _delta(wb_bits, wf_bits):
    return synth.bf16_bits_to_f32(wf_bits).astype(np.float64) - synth.bf16_bits_to_f32(wb_bits).astype(np.float64)


# --------------------------------------------------------------------------------------------
# eq. (3): alpha = mean|Delta| is the L2-optimal scale for the sign code (brute-force search)
# --------------------------------------------------------------------------------------------

def _argmin_scale(delta: np.ndarray, s: np.ndarray) -> float:
    """Brute force: grid of 10^4 points over [0, 2 max|Delta|], then golden-section refinement."""
    top = 2.0 * float(np.max(np.abs(delta))) if delta.size else 0.0
    if top == 0.0:
        return 0.0
    grid = np.linspace(0.0, top, 10001)
    err = ((delta[None, :] - grid[:, None] * s[None, :]) ** 2).sum(axis=1)
    k = int(np.argmin(err))
    lo, hi = grid[max(k - 1, 0)], grid[min(k + 1, len(grid) - 1)]

    def f(a):
        return float(((delta - a * s) ** 2).sum())

    g = (math.sqrt(5.0) - 1.0) / 2.0
    a, b = lo, hi
    c, d = b - g * (b - a), a + g * (b - a)
    for _ in range(200):
        if f(c) < f(d):
            b = d
        else:
            a = c
        c, d = b - g * (b - a), a + g * (b - a)
    return 0.5 * (a + b)


def _tiny_cases():
    rng = np.random.default_rng(11)
    cases = []
    for d_out, d_in in [(4, 32), (8, 32), (3, 64)]:
        wb = synth.base_weight(rng, d_out, d_in)
        wf = synth.finetuned_weight(rng, wb, 1e-3)
        cases.append((wb, wf))
    # an all-zero-delta row and a single-nonzero row
    wb = synth.base_weight(rng, 4, 32)
    wf = wb.copy()
    wf[1, 7] = synth.f32_to_bf16_bits(np.array([0.5], np.float32))[0]
    wf[2] = synth.finetuned_weight(rng, wb[2:3], 2e-3)[0]
    cases.append((wb, wf))
    return cases


@pytest.mark.parametrize("case", range(4))
def test_alpha_is_l2_optimal_per_row(case):
    wb, wf = _tiny_cases()[case]
    signs, alpha = oracle.compress(wb, wf, per_row=True)
    s = oracle.unpack_signs(signs, wb.shape[1]).astype(np.float64)
    delta = _delta(wb, wf)
    for i in range(wb.shape[0]):
        a_star = _argmin_scale(delta[i], s[i])
        assert alpha[i] == pytest.approx(a_star, rel=1e-6, abs=1e-12), (i, alpha[i], a_star)


@pytest.mark.parametrize("case", range(4))
def test_alpha_is_l2_optimal_per_matrix(case):
    wb, wf = _tiny_cases()[case]
    signs, alpha = oracle.compress(wb, wf, per_row=False)
    assert alpha.shape == (1,)
    s = oracle.unpack_signs(signs, wb.shape[1]).astype(np.float64).ravel()
    a_star = _argmin_scale(_delta(wb, wf).ravel(), s)
    assert alpha[0] == pytest.approx(a_star, rel=1e-6, abs=1e-12)


def test_alpha_all_zero_delta_is_zero():
    wb = synth.base_weight(np.random.default_rng(3), 5, 64)
    for per_row in (True, False):
        signs, alpha = oracle.compress(wb, wb, per_row=per_row)
        assert np.all(alpha == 0.0)
        assert np.all(signs == 0xFFFFFFFF)  # sign(0) := +1 everywhere


# --------------------------------------------------------------------------------------------
# bit layout: hand-built rows (tests/golden/hand_bits.txt)
# --------------------------------------------------------------------------------------------

def _hand_rows():
    rows = []
    with open(os.path.join(GOLDEN, "hand_bits.txt")) as fh:
        for line in fh:
            if not line.strip() or line.startswith("#"):
                continue
            name, cols, words = [p.strip() for p in line.split("|")]
            wf = np.full(64, -1.0, np.float32)
            if cols:
                for item in cols.split(","):
                    c, v = item.split("=")
                    wf[int(c)] = np.float32(float(v))
            rows.append((name, wf, [int(w, 16) for w in words.split()]))
    return rows


def test_hand_built_bit_patterns():
    rows = _hand_rows()
    assert len(rows) >= 8
    wf = np.stack([r[1] for r in rows])
    wb = np.zeros_like(wf)
    signs, _ = oracle.compress(_bits(wb), _bits(wf), per_row=True)
    for k, (name, _, words) in enumerate(rows):
        assert [int(w) for w in signs[k]] == words, name


def test_byte_view_is_int8_rows_of_d_in_over_8():
    """Little-endian byte view = int8 [d_out][d_in/8], bit k of byte c <-> column 8c+k."""
    rng = np.random.default_rng(5)
    s = np.where(rng.random((6, 96)) < 0.5, -1, 1).astype(np.int8)
    packed = oracle.pack_signs(s)
    as_bytes = packed.view(np.uint8)
    assert as_bytes.shape == (6, 96 // 8)
    expect = np.packbits((s > 0).astype(np.uint8), axis=1, bitorder="little")
    assert np.array_equal(as_bytes, expect)


def test_pack_unpack_round_trips():
    rng = np.random.default_rng(6)
    s = np.where(rng.random((9, 128)) < 0.3, -1, 1).astype(np.int8)
    assert np.array_equal(oracle.unpack_signs(oracle.pack_signs(s), 128), s)
    bits = rng.integers(0, 2**32, size=(7, 4), dtype=np.uint64).astype(np.uint32)
    assert np.array_equal(oracle.pack_signs(oracle.unpack_signs(bits, 128)), bits)


def test_compress_rejects_d_in_not_multiple_of_32():
    wb = np.zeros((2, 48), np.uint16)
    with pytest.raises(ValueError):
        oracle.compress(wb, wb, per_row=True)


# --------------------------------------------------------------------------------------------
# sizes the page prints
# --------------------------------------------------------------------------------------------

def test_page_sizes():
    n = 0
    with open(os.path.join(GOLDEN, "page_sizes.txt")) as fh:
        for line in fh:
            if not line.strip() or line.startswith("#"):
                continue
            name, d_out, d_in, n_alpha, expect = line.split("--")[0].split()
            assert oracle.compressed_bytes(int(d_out), int(d_in), int(n_alpha)) == int(expect), name
            n += 1
    assert n == 2
    # per-row alpha adds 4 bytes per output row (float32, one per output dimension)
    assert oracle.compressed_bytes(4096, 4096, 4096) == 4096 * 512 + 4 * 4096


def test_page_memory_arithmetic():
    vals = {}
    with open(os.path.join(GOLDEN, "page_memory.txt")) as fh:
        for line in fh:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                vals[k] = float(v)
    params, nv = int(vals["params"]), int(vals["variants"])
    base_bytes = 2 * params  # bf16
    assert base_bytes / 1e9 == vals["base_gb"]
    assert nv * base_bytes / 1e12 == pytest.approx(vals["naive_tb"])
    delta_bytes = oracle.compressed_bytes(params, 1, 0)
    total = base_bytes + nv * delta_bytes
    assert total / 1e9 == pytest.approx(vals["bitdelta_gb_approx"], abs=1.0)
    assert 100 * (1 - total / (nv * base_bytes)) == pytest.approx(vals["reduction_pct_approx"], abs=0.5)


# --------------------------------------------------------------------------------------------
# eq. (2) and the listing: reconstruction invariants
# --------------------------------------------------------------------------------------------

@pytest.mark.parametrize("per_row", [True, False])
def test_reconstruction_invariants(per_row):
    wb, wf, _ = synth.single_problem(21, 24, 96, 1)
    signs, alpha = oracle.compress(wb, wf, per_row=per_row)
    weff = oracle.reconstruct(wb, signs, alpha, per_row)
    base = synth.bf16_bits_to_f32(wb).astype(np.float64)
    a = alpha.astype(np.float64)[:, None] if per_row else np.float64(alpha[0])
    diff = weff - base
    assert np.array_equal(np.abs(diff), np.broadcast_to(a, diff.shape))
    delta = _delta(wb, wf)
    code = np.where(delta < 0, -1.0, 1.0)
    assert np.array_equal(np.sign(diff), code)
    assert (delta == 0).any(), "fixture should exercise sign(0)"


# --------------------------------------------------------------------------------------------
# the linear: special cases that reduce to numpy, and exact rational arithmetic
# --------------------------------------------------------------------------------------------

@pytest.mark.parametrize("per_row", [True, False])
def test_zero_delta_is_plain_gemm(per_row):
    rng = np.random.default_rng(8)
    wb = synth.base_weight(rng, 40, 96)
    x = synth.activations(rng, 5, 96)
    signs, alpha = oracle.compress(wb, wb, per_row=per_row)
    y = oracle.linear(x, wb, signs, alpha, per_row)
    ref = synth.bf16_bits_to_f32(x).astype(np.float64) @ synth.bf16_bits_to_f32(wb).astype(np.float64).T
    assert y.shape == (5, 40)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("direction", [+1.0, -1.0])
def test_zero_base_is_alpha_times_token_sum(direction):
    rng = np.random.default_rng(9)
    mags = rng.integers(1, 9, size=(12, 64)).astype(np.float32) / 64.0
    wb = np.zeros((12, 64), np.float32)
    wf = direction * mags
    signs, alpha = oracle.compress(_bits(wb), _bits(wf), per_row=True)
    x = synth.activations(rng, 3, 64)
    y = oracle.linear(x, _bits(wb), signs, alpha, True)
    xs = synth.bf16_bits_to_f32(x).astype(np.float64).sum(axis=1)
    ref = direction * xs[:, None] * mags.astype(np.float64).mean(axis=1)[None, :]
    np.testing.assert_allclose(y, ref, rtol=1e-6, atol=0)


def test_linear_exact_rationals():
    """Dyadic inputs: the exact result, computed with Fractions, must be reproduced exactly."""
    rng = np.random.default_rng(10)
    d_out, d_in, T = 6, 64, 3
    wb = rng.integers(-8, 9, size=(d_out, d_in)).astype(np.float32) / 64.0
    e = rng.integers(5, 9, size=d_out)
    s = np.where(rng.random((d_out, d_in)) < 0.5, -1.0, 1.0).astype(np.float32)
    wf = wb + s * (2.0 ** (-e.astype(np.float32)))[:, None]
    x = rng.integers(-4, 5, size=(T, d_in)).astype(np.float32)
    signs, alpha = oracle.compress(_bits(wb), _bits(wf), per_row=True)
    assert np.array_equal(alpha, (2.0 ** -e).astype(np.float32))
    y = oracle.linear(_bits(x), _bits(wb), signs, alpha, True)
    for t in range(T):
        for i in range(d_out):
            exact = sum(Fraction(float(x[t, j])) * (Fraction(float(wb[i, j])) +
                                                     Fraction(1, 2 ** int(e[i])) * int(s[i, j]))
                        for j in range(d_in))
            assert Fraction(y[t, i]) == exact


def test_linear_rows_subset_matches_listed_rows():
    wb, wf, x = synth.single_problem(12, 33, 64, 2)
    signs, alpha = oracle.compress(wb, wf, per_row=True)
    y_all = oracle.linear(x, wb, signs, alpha, True)
    rows = np.array([0, 5, 32], np.int64)
    y_sub = oracle.linear(x, wb, signs, alpha, True, rows=rows)
    assert np.array_equal(y_sub, y_all[:, rows])
    s2, a2 = oracle.compress_rows(wb, wf, rows)
    assert np.array_equal(s2, signs[rows]) and np.array_equal(a2, alpha[rows])


# --------------------------------------------------------------------------------------------
# the Laplace model of section "Matematiksel temel"
# --------------------------------------------------------------------------------------------

def test_laplace_statistics():
    """For Delta ~ Laplace(0, b): E|Delta| = b, and E(Delta - alpha s)^2 / E Delta^2 -> 1/2."""
    b = 1e-3
    wb, wf, _ = synth.single_problem(13, 256, 4096, 1, b=b)
    signs, alpha = oracle.compress(wb, wf, per_row=False)
    assert alpha[0] == pytest.approx(b, rel=0.01)
    delta = _delta(wb, wf)
    s = oracle.unpack_signs(signs, 4096).astype(np.float64)
    ratio = np.linalg.norm(delta - alpha[0] * s) / np.linalg.norm(delta)
    assert ratio == pytest.approx(1 / math.sqrt(2), rel=0.01)
    # about 4% of the deltas are exactly zero after bf16 rounding; they all got +1
    zero = delta == 0
    assert 0.02 < zero.mean() < 0.08
    assert np.all(s[zero] == 1)


# --------------------------------------------------------------------------------------------
# the router (section "Sunum mimarisi", serving steps 1-3)
# --------------------------------------------------------------------------------------------

@pytest.mark.parametrize("T,V", [(0, 3), (1, 1), (64, 14), (257, 5), (1000, 64)])
def test_route_is_stable_sort_by_key(T, V):
    rng = np.random.default_rng(T + V)
    vid = rng.integers(-1, V, size=T).astype(np.int32)
    if T > 4:
        vid[::7] = V + 3  # out of range: routed as base and counted
        vid[1] = -5
    perm, seg, n_bad = oracle.route(vid, V)
    key = np.where((vid >= -1) & (vid < V), vid + 1, 0)
    assert n_bad == int(((vid < -1) | (vid >= V)).sum())
    assert np.array_equal(perm, np.argsort(key, kind="stable"))
    counts = np.bincount(key, minlength=V + 1)
    assert np.array_equal(seg, np.concatenate([[0], np.cumsum(counts)]).astype(np.int32))


def test_multi_routes_each_token_to_its_variant():
    """W_base = 0 and all-plus signs: y[t][i] = alpha_{vid[t]}[i] * sum_j x[t][j] (0 for base tokens)."""
    rng = np.random.default_rng(14)
    V, d_out, d_in, T = 4, 8, 64, 9
    wb = np.zeros((d_out, d_in), np.float32)
    signs_l, alpha_l = [], []
    for v in range(V):
        wf = np.full((d_out, d_in), 2.0 ** -(v + 3), np.float32) * (1 + np.arange(d_out))[:, None]
        s, a = oracle.compress(_bits(wb), _bits(wf), per_row=True)
        signs_l.append(s)
        alpha_l.append(a)
    vid = np.array([0, 3, -1, 2, 2, 1, 0, -1, 3], np.int32)
    x = synth.activations(rng, T, d_in)
    y = oracle.linear_multi(x, vid, signs_l, alpha_l, True, _bits(wb))
    xs = synth.bf16_bits_to_f32(x).astype(np.float64).sum(axis=1)
    for t in range(T):
        expect = np.zeros(d_out) if vid[t] < 0 else 2.0 ** -(vid[t] + 3) * (1 + np.arange(d_out)) * xs[t]
        np.testing.assert_allclose(y[t], expect, rtol=1e-12, atol=1e-15)


def test_multi_out_of_range_ids_are_base_model_tokens():
    """The reading for ids outside [-1, V): such a token is computed with
    W_base alone.  With W_base = 0 its output is exactly 0; with a random
    W_base it equals numpy's fp64 product x W_base^T (the Delta = 0 GEMM),
    while the in-range tokens keep their variant's alpha * sum_j x_j."""
    rng = np.random.default_rng(15)
    V, d_out, d_in, T = 3, 6, 64, 10
    signs_l, alpha_l = [], []
    wb0 = np.zeros((d_out, d_in), np.float32)
    for v in range(V):
        wf = np.full((d_out, d_in), 2.0 ** -(v + 2), np.float32)
        s, a = oracle.compress(_bits(wb0), _bits(wf), per_row=True)
        signs_l.append(s)
        alpha_l.append(a)
    vid = np.array([V, 0, -2, 2, V + 7, -1, 1, -9, 0, 2 ** 30], np.int32)
    bad = (vid < -1) | (vid >= V)
    x = synth.activations(rng, T, d_in)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    y = oracle.linear_multi(x, vid, signs_l, alpha_l, True, _bits(wb0))
    assert np.all(y[bad] == 0.0) and np.all(y[vid == -1] == 0.0)
    for t in np.flatnonzero((vid >= 0) & (vid < V)):
        np.testing.assert_allclose(y[t], 2.0 ** -(vid[t] + 2) * xf[t].sum(), rtol=1e-12)
    wb = synth.base_weight(rng, d_out, d_in)
    y2 = oracle.linear_multi(x, vid, signs_l, alpha_l, True, wb)
    gemm = xf @ synth.bf16_bits_to_f32(wb).astype(np.float64).T
    np.testing.assert_allclose(y2[bad], gemm[bad], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(y2[vid == -1], gemm[vid == -1], rtol=1e-12, atol=1e-15)
    _, _, n_bad = oracle.route(vid, V)
    assert n_bad == int(bad.sum())


def test_synth_zipf_ids_in_range_and_skewed():
    rng = np.random.default_rng(0)
    vid = synth.zipf_variant_ids(rng, 20000, 14)
    assert vid.min() >= 0 and vid.max() <= 13
    counts = np.bincount(vid, minlength=14) / 20000
    p = np.arange(1, 15, dtype=np.float64) ** -1.1
    np.testing.assert_allclose(counts, p / p.sum(), atol=0.01)


# ---------------------------------------------------------------- bf16 rounding of the materialised weights

def test_round_to_bf16_hand_cases():
    """Ties go to the even significand, both signs; a value just above a tie
    rounds up even though fp32 could not hold it (one rounding, not two)."""
    one = np.float64(1.0)
    cases = {
        one: 0x3F80,
        one + 2.0**-8: 0x3F80,               # tie between 1 and 1 + 2^-7: even (1)
        one + 3 * 2.0**-8: 0x3F82,           # tie between 1 + 2^-7 and 1 + 2^-6: even (mantissa 2)
        one + 2.0**-8 + 2.0**-30: 0x3F81,    # above the tie: up
        one + 2.0**-8 - 2.0**-30: 0x3F80,    # below the tie: down
        -(one + 3 * 2.0**-8): 0xBF82,
        -(one + 2.0**-8 + 2.0**-30): 0xBF81,
        0.0: 0x0000,
    }
    got = oracle.round_to_bf16(np.array(list(cases.keys())))
    assert [int(g) for g in got] == list(cases.values())


def test_round_to_bf16_matches_the_fp32_rounding_of_the_input_module():
    """For values exactly representable in fp32 the one rounding to bf16 is
    the fp32 -> bf16 rounding that synth implements independently."""
    rng = np.random.default_rng(3)
    v = (rng.standard_normal(20000) * 2.0 ** rng.integers(-20, 20, 20000)).astype(np.float32)
    assert np.array_equal(oracle.round_to_bf16(v.astype(np.float64)), synth.f32_to_bf16_bits(v))


def _all_finite_bf16():
    """(values, patterns) of every finite non-negative bf16 number, ascending."""
    pats = np.arange(0, 0x7F80, dtype=np.uint16)
    return synth.bf16_bits_to_f32(pats).astype(np.float64), pats


def _nearest_bf16_brute_force(v: np.ndarray) -> np.ndarray:
    """The definition of round-to-nearest-even, by search over every finite
    bf16 value: the closest one, the one with an even last significand bit
    on a tie; the sign is carried over (so -0.0 stays -0.0)."""
    vals, pats = _all_finite_bf16()
    out = np.zeros(v.shape, np.uint16)
    for i, x in enumerate(v):
        a = abs(float(x))
        k = int(np.searchsorted(vals, a))  # vals[k-1] < a <= vals[k]
        cand = [j for j in (k - 1, k) if 0 <= j < len(vals)]
        d = [abs(vals[j] - a) for j in cand]
        best = min(d)
        ties = [cand[n] for n in range(len(cand)) if d[n] == best]
        j = ties[0] if len(ties) == 1 else next(t for t in ties if int(pats[t]) % 2 == 0)
        out[i] = int(pats[j]) | (0x8000 if math.copysign(1.0, float(x)) < 0 else 0)
    return out


def test_round_to_bf16_brute_force_normal_and_subnormal():
    """Against the brute-force nearest-even search: random values from bf16's
    subnormal range (below 2^-126, spacing 2^-133) up through its normal
    range, the exact midpoints between neighbouring bf16 values (ties) and a
    hair either side of them, both signs, zeros."""
    rng = np.random.default_rng(41)
    vals, _ = _all_finite_bf16()
    sub = rng.uniform(0, 2.0 ** -126, 400)
    normal = rng.standard_normal(400) * 2.0 ** rng.integers(-126, 120, 400)
    k = rng.integers(0, len(vals) - 1, 400)
    mid = (vals[k] + vals[k + 1]) / 2
    near = np.concatenate([mid, mid * (1 + 2.0 ** -40), mid * (1 - 2.0 ** -40)])
    v = np.concatenate([sub, -sub[:100], normal, near, -near[:200], [0.0, -0.0, 2.0 ** -134, 3 * 2.0 ** -134]])
    assert np.array_equal(oracle.round_to_bf16(v), _nearest_bf16_brute_force(v))


def test_materialize_is_the_rounded_reconstruction():
    """W_eff bits are the bf16 rounding of W_base + alpha s, and decoding them
    is within half a bf16 ulp of the fp64 reconstruction."""
    wb, wf, _ = synth.single_problem(7, 16, 64, 1)
    s, a = oracle.compress(wb, wf, per_row=True)
    bits = oracle.materialize(wb, s, a, True)
    exact = oracle.reconstruct(wb, s, a, True)
    dec = synth.bf16_bits_to_f32(bits).astype(np.float64)
    ulp = 2.0 ** (np.floor(np.log2(np.abs(exact))) - 7)
    assert np.all(np.abs(dec - exact) <= ulp / 2)


# ---------------------------------------------------------------- MonoSoup
# Section "MonoSoup" of the BitDelta post: tau_i = rank-r truncated SVD of
# Delta_i = W_i - W_base, W_merged = W_base + (1/k) sum_i tau_i.


def _orthonormal(rng, n, m):
    q, _ = np.linalg.qr(rng.standard_normal((n, m)))
    return q


def test_monosoup_truncation_closed_form():
    """Delta_i = U diag(s) V^T built from orthonormal U, V and decreasing s
    without any SVD: the rank-r truncation keeps exactly the r leading terms,
    so the merge is W_base + mean_i U_i[:, :r] diag(s_i[:r]) V_i[:, :r]^T.
    A dropped 1/k, an off-by-one rank, a transposed factor or a sign slip all
    fail this (non-square, k = 3)."""
    rng = np.random.default_rng(0)
    d_out, d_in, k, r = 24, 40, 3, 4
    wb = rng.standard_normal((d_out, d_in))
    ws, expect = [], np.zeros((d_out, d_in))
    for _ in range(k):
        u, v = _orthonormal(rng, d_out, 10), _orthonormal(rng, d_in, 10)
        s = np.sort(rng.uniform(0.5, 5.0, 10))[::-1]
        ws.append(wb + (u * s) @ v.T)
        expect += (u[:, :r] * s[:r]) @ v[:, :r].T
    got = oracle.monosoup_merge_f64(wb, ws, r)
    np.testing.assert_allclose(got, wb + expect / k, rtol=0, atol=1e-12)


def test_monosoup_truncation_repeated_singular_values():
    """Singular values that repeat inside the kept rank (a cluster of three
    and a pair, then a gap): the SVD may return any basis of a repeated
    singular subspace, but the rank-r truncation is still unique and equals
    the sum of the r leading terms U diag(s) V^T built without any SVD."""
    rng = np.random.default_rng(5)
    d_out, d_in, r = 20, 28, 5
    s = np.array([3.0, 3.0, 3.0, 2.0, 2.0, 0.5, 0.25, 0.1])
    u, v = _orthonormal(rng, d_out, len(s)), _orthonormal(rng, d_in, len(s))
    wb = rng.standard_normal((d_out, d_in))
    got = oracle.monosoup_merge_f64(wb, [wb + (u * s) @ v.T], r)
    np.testing.assert_allclose(got, wb + (u[:, :r] * s[:r]) @ v[:, :r].T, rtol=0, atol=1e-12)


def test_monosoup_special_cases():
    rng = np.random.default_rng(1)
    wb = rng.standard_normal((12, 16))
    w1, w2 = wb + rng.standard_normal((12, 16)), wb + rng.standard_normal((12, 16))
    # rank 0: the base itself
    np.testing.assert_array_equal(oracle.monosoup_merge_f64(wb, [w1, w2], 0), wb)
    # full rank, one checkpoint: the checkpoint itself
    np.testing.assert_allclose(oracle.monosoup_merge_f64(wb, [w1], 12), w1, atol=1e-12)
    # full rank, several: the plain average of the checkpoints
    np.testing.assert_allclose(oracle.monosoup_merge_f64(wb, [w1, w2], 12), (w1 + w2) / 2, atol=1e-12)
    # k copies of one checkpoint merge like that checkpoint alone
    np.testing.assert_allclose(oracle.monosoup_merge_f64(wb, [w1, w1, w1], 5),
                               oracle.monosoup_merge_f64(wb, [w1], 5), atol=1e-12)


def test_monosoup_eckart_young():
    """The truncation error ||Delta - tau||_F^2 equals the sum of the
    eigenvalues of Delta^T Delta past the r largest (eigvalsh, a different
    routine from the SVD the oracle calls), and projecting Delta on random
    r-dimensional subspaces never does better (rank-r optimality)."""
    rng = np.random.default_rng(2)
    d = rng.standard_normal((30, 20))
    r = 6
    tau = oracle.monosoup_merge_f64(np.zeros_like(d), [d], r)
    assert np.linalg.matrix_rank(tau) == r
    err = np.sum((d - tau) ** 2)
    lam = np.sort(np.linalg.eigvalsh(d.T @ d))[::-1]
    assert abs(err - lam[r:].sum()) <= 1e-9 * lam.sum()
    for _ in range(20):
        q = _orthonormal(rng, 30, r)
        assert np.sum((d - q @ (q.T @ d)) ** 2) >= err * (1 - 1e-12)


def test_bf16_to_f64_patterns():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x3C23, 0x7F7F], np.uint16)
    got = oracle.bf16_to_f64(bits)
    assert got[0] == 1.0 and got[1] == -2.0 and got[2] == 0.0 and np.signbit(got[3])
    assert got[4] == float.fromhex("0x1.46p-7") and got[5] == float.fromhex("0x1.FEp127")
