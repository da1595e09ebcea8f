"""GPU parity of libbitdelta.so against the fp64 CPU oracle, through the C ABI.

Packed signs and routing must match bit for bit, alpha to 1e-6 relative, and
linear outputs within the tolerances of tests/helpers.py.  Workloads follow
the BitDelta serving setup: a 256x256 tiny linear, the 28672x8192 FFN-shaped
decode GEMV (T = 1, 4, 16), and the 8192x8192 multi-tenant decode with 14
variants and 64 Zipf-routed tokens; plus ragged shapes, exact dyadic inputs
(where any summation order is exact, so results must be bit-identical), row
sharding, canary guards, determinism and argument errors.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

import oracle
from bit_weight_delta_bd_gb300 import bitdelta as bd
from bit_weight_delta_bd_gb300 import synth
from helpers import (PREFILL_MIN_T, bf16_half_ulp, check_linear, fp32_bound, fp32_bound_multi,  # noqa: F401
                     to_dev, u32, y_host)

pytestmark = pytest.mark.gpu

PR, PM = bd.BD_ALPHA_PER_ROW, bd.BD_ALPHA_PER_MATRIX


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def gpu_compress(wb_d, wf_d, mode, dev):
    d_out, d_in = wb_d.shape
    signs = torch.empty((d_out, d_in // 32), dtype=torch.int32, device=dev)
    alpha = torch.empty(d_out if mode == PR else 1, dtype=torch.float32, device=dev)
    ws = bd.new_workspace(bd.bd_compress_workspace_size(d_out, d_in, mode), dev)
    bd.bd_compress(wb_d, wf_d, mode, signs, alpha, ws)
    assert bd.bd_check_async(ws) == bd.BD_OK
    return signs, alpha


def gpu_linear(x_d, wb_d, signs, alpha, mode, dev, f32=True):
    T, d_out = x_d.shape[0], wb_d.shape[0]
    y = torch.empty((T, d_out), dtype=torch.float32 if f32 else torch.bfloat16, device=dev)
    ws = bd.new_workspace(bd.bd_linear_workspace_size(T, d_out, wb_d.shape[1]), dev)
    bd.bd_linear(x_d, wb_d, signs, alpha, mode, y, ws)
    assert bd.bd_check_async(ws) == bd.BD_OK
    return y


def assert_alpha(a_gpu, a_ref):
    a_gpu = np.asarray(a_gpu, np.float64)
    a_ref = np.asarray(a_ref, np.float64)
    np.testing.assert_allclose(a_gpu, a_ref, rtol=1e-6, atol=0)


# ============================================================================ compress

def test_compress_tiny_per_matrix(dev):
    wb, wf, _ = synth.single_problem(0, 256, 256, 4)
    s_ref, a_ref = oracle.compress(wb, wf, per_row=False)
    s, a = gpu_compress(to_dev(wb, dev), to_dev(wf, dev), PM, dev)
    assert np.array_equal(u32(s), s_ref)
    assert_alpha(a.cpu().numpy(), a_ref)


@pytest.mark.parametrize("mode", [PR, PM])
@pytest.mark.parametrize("d_out,d_in", [(1, 128), (17, 384), (33, 1024), (100, 256), (8, 8192 + 128)])
def test_compress_shapes(dev, mode, d_out, d_in):
    wb, wf, _ = synth.single_problem(d_out * 7 + d_in, d_out, d_in, 1)
    s_ref, a_ref = oracle.compress(wb, wf, per_row=mode == PR)
    s, a = gpu_compress(to_dev(wb, dev), to_dev(wf, dev), mode, dev)
    assert np.array_equal(u32(s), s_ref)
    assert_alpha(a.cpu().numpy(), a_ref)


@pytest.fixture(scope="module")
def decode_problem():
    """The 28672 x 8192 FFN-shaped matrix of the decode workload, seed 0."""
    wb, wf, _ = synth.single_problem(0, 28672, 8192, 1)
    return wb, wf


def test_compress_ffn_full_and_deterministic(dev, decode_problem):
    wb, wf = decode_problem
    s_ref, a_ref = oracle.compress(wb, wf, per_row=True)
    wb_d, wf_d = to_dev(wb, dev), to_dev(wf, dev)
    s1, a1 = gpu_compress(wb_d, wf_d, PR, dev)
    assert np.array_equal(u32(s1), s_ref)
    assert_alpha(a1.cpu().numpy(), a_ref)
    s2, a2 = gpu_compress(wb_d, wf_d, PR, dev)
    assert torch.equal(s1, s2) and torch.equal(a1, a2)
    # per-matrix alpha on the same data (same bits)
    s3, a3 = gpu_compress(wb_d, wf_d, PM, dev)
    _, am_ref = oracle.compress(wb, wf, per_row=False)
    assert torch.equal(s3, s1)
    assert_alpha(a3.cpu().numpy(), am_ref)


def test_compress_nonfinite_is_flagged(dev):
    wb, wf, _ = synth.single_problem(3, 16, 256, 1)
    wf = wf.copy()
    wf[5, 17] = 0x7F80  # +inf
    d = to_dev(wb, dev), to_dev(wf, dev)
    signs = torch.empty((16, 8), dtype=torch.int32, device=dev)
    alpha = torch.empty(16, dtype=torch.float32, device=dev)
    ws = bd.new_workspace(bd.bd_compress_workspace_size(16, 256, PR), dev)
    bd.bd_compress(d[0], d[1], PR, signs, alpha, ws)
    assert bd.bd_check_async(ws) == bd.BD_ERR_NONFINITE
    assert bd.bd_check_async(ws) == bd.BD_OK  # cleared
    s_ref, _ = oracle.compress(wb, wf, per_row=True)
    assert np.array_equal(u32(signs), s_ref)  # bits still written


def _golden_hand_rows():
    """Rows of tests/golden/hand_bits.txt: (name, W_ft values [64], expected words [2]).
    W_base = 0 everywhere; W_ft = -1.0 except the listed columns."""
    rows = []
    with open(os.path.join(os.path.dirname(__file__), "golden", "hand_bits.txt")) as fh:
        for line in fh:
            if not line.strip() or line.startswith("#"):
                continue
            name, cols, words = [p.strip() for p in line.split("|")]
            wf = np.full(64, -1.0, np.float32)
            for item in filter(None, cols.split(",")):
                c, v = item.split("=")
                wf[int(c)] = np.float32(float(v))
            rows.append((name, wf, [int(w, 16) for w in words.split()]))
    return rows


@pytest.mark.parametrize("mode", [PR, PM])
def test_compress_golden_hand_rows_on_device(dev, mode):
    """The hand-built sign rows (sign(0) = +1 for +0.0 and -0.0, the bit of
    each column at its place) through bd_compress, checked against the words
    the golden file prints, not against the oracle.  Each 64-column pattern
    is placed at every 64-column offset of a 1024-column row and at several
    row positions of a 37-row matrix (different lanes, warps and CTAs); the
    rest of the matrix is -1.0 (all bits 0)."""
    rows = _golden_hand_rows()
    assert any(r[0] == "negzero_col9" for r in rows) and any(r[0] == "zero_col5" for r in rows)
    d_out, d_in = 37, 1024
    wf = np.full((d_out, d_in), -1.0, np.float32)
    expect = np.zeros((d_out, d_in // 32), np.uint32)
    placed = 0
    for k, (name, pat, words) in enumerate(rows):
        for r in (k, k + 8, k + 29) if k + 29 < d_out else (k, k + 8):
            off = 64 * ((r * 5 + k) % (d_in // 64))
            wf[r, off:off + 64] = pat
            expect[r, off // 32:off // 32 + 2] = words
            placed += 1
    assert placed >= 16
    wb = np.zeros_like(wf)
    wf_bits = synth.f32_to_bf16_bits(wf)
    assert np.any(wf_bits == 0x8000), "-0.0 must reach the device as its own bit pattern"
    s, a = gpu_compress(to_dev(synth.f32_to_bf16_bits(wb), dev), to_dev(wf_bits, dev), mode, dev)
    got = u32(s)
    for r in range(d_out):
        assert np.array_equal(got[r], expect[r]), f"row {r}: {[hex(w) for w in got[r]]}"
    absd = np.abs(wf.astype(np.float64))  # |Delta| = |W_ft| with W_base = 0
    a_ref = absd.mean(axis=1) if mode == PR else np.array([absd.mean()])
    assert_alpha(a.cpu().numpy(), a_ref.astype(np.float32))


def test_compress_row_blocks_per_matrix_alpha(dev):
    """Row sharding of a per-matrix alpha through the library: bd_compress on
    pointer-offset row blocks (one of them empty, whose alpha buffer keeps
    its NaN), alphas combined with the fp64 row weighting of the sharded
    all-reduce, against the unsharded bd_compress and the oracle; the
    stacked signs equal the unsharded ones bit for bit."""
    from bit_weight_delta_bd_gb300 import shard

    d_out, d_in = 1000, 1024
    wb, wf, _ = synth.single_problem(901, d_out, d_in, 1)
    wb_d, wf_d = to_dev(wb, dev), to_dev(wf, dev)
    s_all, a_all = gpu_compress(wb_d, wf_d, PM, dev)
    _, a_ref = oracle.compress(wb, wf, per_row=False)
    for bounds in ([0, 333, 334, 1000], [0, 500, 500, 1000], [0, 1, 999, 1000]):
        shares = torch.zeros(1, dtype=torch.float64, device=dev)
        parts = []
        for r0, r1 in zip(bounds[:-1], bounds[1:]):
            s = torch.empty((r1 - r0, d_in // 32), dtype=torch.int32, device=dev)
            a = torch.full((1,), float("nan"), dtype=torch.float32, device=dev)
            ws = bd.new_workspace(bd.bd_compress_workspace_size(r1 - r0, d_in, PM), dev)
            bd.bd_compress(wb_d[r0:r1], wf_d[r0:r1], PM, s, a, ws)
            assert bd.bd_check_async(ws) == bd.BD_OK
            shares += shard.alpha_share(a, r1 - r0)
            parts.append(s)
        alpha = shard.combine_alpha(shares, d_out)
        assert torch.equal(torch.cat(parts, dim=0), s_all)
        assert_alpha(alpha.cpu().numpy(), a_ref)
        assert_alpha(alpha.cpu().numpy(), a_all.cpu().numpy())


# ============================================================================ linear

def test_linear_tiny(dev):
    wb, wf, x = synth.single_problem(0, 256, 256, 4)
    s_ref, a_ref = oracle.compress(wb, wf, per_row=False)
    y_ref = oracle.linear(x, wb, s_ref, a_ref, per_row=False)
    wb_d = to_dev(wb, dev)
    s, a = gpu_compress(wb_d, to_dev(wf, dev), PM, dev)
    for f32 in (True, False):
        y = gpu_linear(to_dev(x, dev), wb_d, s, a, PM, dev, f32=f32)
        check_linear(y_host(y), y_ref, bf16_out=not f32,
                     bound=fp32_bound(x, wb, a.cpu().numpy(), False) if f32 else None, what=f"tiny f32={f32}")


@pytest.mark.parametrize("T", [1, 3, 8, 9, 17, 33, 64, 65, 130, 300])
@pytest.mark.parametrize("d_out,d_in", [(1, 128), (17, 384), (48, 1024), (200, 640)])
def test_linear_shapes(dev, T, d_out, d_in):
    wb, wf, x = synth.single_problem(T * 131 + d_out, d_out, d_in, T)
    s_ref, a_ref = oracle.compress(wb, wf, per_row=True)
    y_ref = oracle.linear(x, wb, s_ref, a_ref, per_row=True)
    wb_d = to_dev(wb, dev)
    s, a = gpu_compress(wb_d, to_dev(wf, dev), PR, dev)
    y = gpu_linear(to_dev(x, dev), wb_d, s, a, PR, dev)
    check_linear(y_host(y), y_ref, bf16_out=False,
                 bound=fp32_bound(x, wb, a.cpu().numpy(), True, weff_bf16=T >= PREFILL_MIN_T),
                 what=f"T={T} {d_out}x{d_in}")


def _dyadic_problem(seed, d_out, d_in, T, per_row):
    """x in {-4..4}, W_base in {k/64}, Delta = +-2^-e: every partial sum is exact in fp32."""
    rng = np.random.default_rng(seed)
    wb = rng.integers(-8, 9, size=(d_out, d_in)).astype(np.float32) / 64.0
    e = rng.integers(5, 9, size=d_out if per_row else 1).astype(np.float32)
    s = np.where(rng.random((d_out, d_in)) < 0.5, -1.0, 1.0).astype(np.float32)
    step = 2.0 ** -e
    wf = wb + s * (step[:, None] if per_row else step[0])
    x = rng.integers(-4, 5, size=(T, d_in)).astype(np.float32)
    return synth.f32_to_bf16_bits(wb), synth.f32_to_bf16_bits(wf), synth.f32_to_bf16_bits(x)


@pytest.mark.parametrize("per_row", [True, False])
@pytest.mark.parametrize("T", [1, 5, 16, 64, 100])
def test_linear_exact_dyadic_bit_identical(dev, per_row, T):
    wb, wf, x = _dyadic_problem(T, 40, 1024, T, per_row)
    s_ref, a_ref = oracle.compress(wb, wf, per_row=per_row)
    y_ref = oracle.linear(x, wb, s_ref, a_ref, per_row=per_row)
    mode = PR if per_row else PM
    wb_d = to_dev(wb, dev)
    s, a = gpu_compress(wb_d, to_dev(wf, dev), mode, dev)
    assert np.array_equal(u32(s), s_ref)
    assert np.array_equal(a.cpu().numpy(), a_ref)
    y = gpu_linear(to_dev(x, dev), wb_d, s, a, mode, dev)
    assert np.array_equal(y.cpu().numpy().astype(np.float64), y_ref)


@pytest.mark.parametrize("T", [1, 4, 16])
def test_linear_ffn_decode_sampled_rows(dev, decode_problem, T):
    wb, wf = decode_problem
    x = synth.activations(np.random.default_rng(100 + T), T, 8192)
    rows = synth.sample_rows(T, 28672, 384)
    s_rows, a_rows = oracle.compress_rows(wb, wf, rows)
    # the oracle indexes signs/alpha by absolute row: place the sampled rows
    s_full = np.zeros((28672, 256), np.uint32)
    a_full = np.zeros(28672, np.float32)
    s_full[rows], a_full[rows] = s_rows, a_rows
    y_ref = oracle.linear(x, wb, s_full, a_full, per_row=True, rows=rows)
    wb_d = to_dev(wb, dev)
    s, a = gpu_compress(wb_d, to_dev(wf, dev), PR, dev)
    assert np.array_equal(u32(s)[rows], s_rows)
    x_d = to_dev(x, dev)
    for f32 in (True, False):
        y = gpu_linear(x_d, wb_d, s, a, PR, dev, f32=f32)
        yg = y_host(y)[:, rows]
        check_linear(yg, y_ref, bf16_out=not f32,
                     bound=fp32_bound(x, wb, a.cpu().numpy(), True, rows=rows) if f32 else None,
                     what=f"ffn T={T} f32={f32}")


@pytest.mark.parametrize("T", [4, 64, 300])
def test_linear_row_sharding_is_bit_identical(dev, T):
    d_out, d_in = 300, 1024
    wb, wf, x = synth.single_problem(77, d_out, d_in, T)
    wb_d, x_d = to_dev(wb, dev), to_dev(x, dev)
    s, a = gpu_compress(wb_d, to_dev(wf, dev), PR, dev)
    y_full = gpu_linear(x_d, wb_d, s, a, PR, dev)
    parts = []
    for r0, r1 in [(0, 37), (37, 160), (160, 300)]:
        parts.append(gpu_linear(x_d, wb_d[r0:r1], s[r0:r1], a[r0:r1], PR, dev))
    assert torch.equal(torch.cat(parts, dim=1), y_full)


@pytest.mark.parametrize("d_out,d_in,per_row", [(256, 256, False), (100, 1024, True), (7, 128, True)])
def test_materialize_bit_exact(dev, d_out, d_in, per_row):
    """bd_materialize equals the oracle's one-rounding bf16 W_eff bit for bit."""
    wb, wf, _ = synth.single_problem(d_out + d_in, d_out, d_in, 1)
    mode = PR if per_row else PM
    s, a = oracle.compress(wb, wf, per_row=per_row)
    w_eff = torch.empty((d_out, d_in), dtype=torch.int16, device=dev)
    bd.bd_materialize(to_dev(wb, dev), to_dev(s, dev).view(torch.int32), to_dev(a, dev), mode, w_eff)
    assert np.array_equal(w_eff.cpu().numpy().view(np.uint16), oracle.materialize(wb, s, a, per_row))


def test_materialize_midpoint_sums(dev):
    """alpha = 2^-8 + 2^-30 on W_base = 1 + k 2^-7: every fp32 sum is a bf16
    midpoint and its lost 2^-30 decides the rounding (up for +alpha, toward
    zero for -alpha); random signs."""
    rng = np.random.default_rng(5)
    d_out, d_in = 64, 256
    k = rng.integers(0, 100, size=(d_out, d_in))
    wb = synth.f32_to_bf16_bits((1.0 + k * 2.0**-7).astype(np.float32))
    s = rng.integers(0, 2**32, size=(d_out, d_in // 32), dtype=np.uint64).astype(np.uint32)
    a = np.array([2.0**-8 + 2.0**-30], np.float32)
    w_eff = torch.empty((d_out, d_in), dtype=torch.int16, device=dev)
    bd.bd_materialize(to_dev(wb, dev), to_dev(s, dev).view(torch.int32), to_dev(a, dev), PM, w_eff)
    ref = oracle.materialize(wb, s, a, False)
    assert np.array_equal(w_eff.cpu().numpy().view(np.uint16), ref)
    # the plain fp32-then-bf16 double rounding would differ on about half of them
    dbl = synth.f32_to_bf16_bits(oracle.reconstruct(wb, s, a, False).astype(np.float32))
    assert np.mean(dbl != ref) > 0.25


def test_materialize_ffn_sampled_rows(dev, decode_problem):
    """The 28672 x 8192 decode matrix: every row written, sampled rows exact."""
    wb, wf = decode_problem
    wb_d = to_dev(wb, dev)
    s, a = gpu_compress(wb_d, to_dev(wf, dev), PR, dev)
    w_eff = torch.empty((28672, 8192), dtype=torch.int16, device=dev)
    bd.bd_materialize(wb_d, s, a, PR, w_eff)
    rows = synth.sample_rows(17, 28672, 64)
    s_h, a_h = s.cpu().numpy().view(np.uint32), a.cpu().numpy()
    ref = oracle.materialize(wb[rows], s_h[rows], a_h[rows], True)
    assert np.array_equal(w_eff.cpu().numpy().view(np.uint16)[rows], ref)


@pytest.fixture(scope="module")
def prefill_problem():
    """Prefill workload: 4096 tokens x W_base [8192 x 8192], one variant, per-row alpha."""
    return synth.single_problem(3, 8192, 8192, 4096)


def test_prefill_4096_tokens_sampled_rows(dev, prefill_problem):
    wb, wf, x = prefill_problem
    rows = synth.sample_rows(11, 8192, 48)
    s_rows, a_rows = oracle.compress_rows(wb, wf, rows)
    s_full = np.zeros((8192, 256), np.uint32)
    a_full = np.zeros(8192, np.float32)
    s_full[rows], a_full[rows] = s_rows, a_rows
    toks = np.unique(np.concatenate([np.arange(0, 4096, 37), [4095]]))
    y_ref = oracle.linear(x[toks], wb, s_full, a_full, per_row=True, rows=rows)
    wb_d = to_dev(wb, dev)
    s, a = gpu_compress(wb_d, to_dev(wf, dev), PR, dev)
    assert np.array_equal(u32(s)[rows], s_rows)
    x_d = to_dev(x, dev)
    for f32 in (True, False):
        y = gpu_linear(x_d, wb_d, s, a, PR, dev, f32=f32)
        yg = y_host(y)[np.ix_(toks, rows)]
        check_linear(yg, y_ref, bf16_out=not f32,
                     bound=fp32_bound(x[toks], wb, a.cpu().numpy(), True, rows=rows, weff_bf16=True) if f32 else None,
                     what=f"prefill f32={f32}")


def test_linear_zero_sizes_are_noops(dev):
    wb = torch.zeros((4, 128), dtype=torch.int16, device=dev)
    s = torch.zeros((4, 4), dtype=torch.int32, device=dev)
    a = torch.zeros(4, dtype=torch.float32, device=dev)
    ws = bd.new_workspace(256, dev)
    x0 = torch.zeros((0, 128), dtype=torch.int16, device=dev)
    y0 = torch.zeros((0, 4), dtype=torch.float32, device=dev)
    lib = bd.load()
    st = torch.cuda.current_stream().cuda_stream
    assert lib.bd_linear(x0.data_ptr(), 0, wb.data_ptr(), s.data_ptr(), a.data_ptr(), PR, 4, 128, y0.data_ptr(),
                         1, ws.data_ptr(), ws.numel(), st) == bd.BD_OK
    assert lib.bd_compress(wb.data_ptr(), wb.data_ptr(), 0, 128, PR, s.data_ptr(), a.data_ptr(), ws.data_ptr(),
                           ws.numel(), st) == bd.BD_OK


# ============================================================================ multi-variant

@pytest.fixture(scope="module")
def multi_problem():
    """8192 x 8192 shared W_base, 14 variants (b ~ U[5e-4, 2e-3]), 64 Zipf tokens."""
    return synth.multi_problem(0, 8192, 8192, 64, 14)


def test_multi_tenant_sampled_rows(dev, multi_problem):
    wb, wfs, x, vid, _ = multi_problem
    rows = synth.sample_rows(5, 8192, 256)
    refs = [oracle.compress_rows(wb, wf, rows) for wf in wfs]
    wb_d = to_dev(wb, dev)
    s_l, a_l = [], []
    for v, wf in enumerate(wfs):
        s, a = gpu_compress(wb_d, to_dev(wf, dev), PR, dev)
        assert np.array_equal(u32(s)[rows], refs[v][0]), f"variant {v} bits"
        assert_alpha(a.cpu().numpy()[rows], refs[v][1])
        s_l.append(s)
        a_l.append(a)
    s_full, a_full = [], []
    for s_rows, a_rows in refs:
        sf = np.zeros((8192, 256), np.uint32)
        af = np.zeros(8192, np.float32)
        sf[rows], af[rows] = s_rows, a_rows
        s_full.append(sf)
        a_full.append(af)
    y_ref = oracle.linear_multi(x, vid, s_full, a_full, True, wb, rows=rows)
    x_d, vid_d = to_dev(x, dev), to_dev(vid, dev)
    for f32 in (True, False):
        y = torch.empty((64, 8192), dtype=torch.float32 if f32 else torch.bfloat16, device=dev)
        ws = bd.new_workspace(bd.bd_linear_multi_workspace_size(64, 14, 8192, 8192), dev)
        bd.bd_linear_multi(x_d, vid_d, s_l, a_l, PR, wb_d, y, ws)
        assert bd.bd_check_async(ws) == bd.BD_OK
        bound = fp32_bound_multi(x, wb, [r[1] for r in refs], vid, rows) if f32 else None
        check_linear(y_host(y)[:, rows], y_ref, bf16_out=not f32, bound=bound, what=f"multi f32={f32}")


def _dyadic_multi(seed, V, d_out, d_in, T):
    rng = np.random.default_rng(seed)
    wb = rng.integers(-8, 9, size=(d_out, d_in)).astype(np.float32) / 64.0
    wfs = []
    for v in range(V):
        s = np.where(rng.random((d_out, d_in)) < 0.5, -1.0, 1.0).astype(np.float32)
        wfs.append(synth.f32_to_bf16_bits(wb + s * 2.0 ** -(3 + v % 6)))
    x = rng.integers(-4, 5, size=(T, d_in)).astype(np.float32)
    return synth.f32_to_bf16_bits(wb), wfs, synth.f32_to_bf16_bits(x)


@pytest.mark.parametrize("V,T", [(1, 1), (3, 10), (14, 64), (64, 64), (5, 150)])
def test_multi_exact_routing_signature(dev, V, T):
    """Distinct variant scales and sign patterns: a token routed to the wrong
    variant changes its output by an exact, visible amount."""
    d_out, d_in = 33, 512
    wb, wfs, x = _dyadic_multi(V * 1000 + T, V, d_out, d_in, T)
    rng = np.random.default_rng(T)
    vid = rng.integers(-1, V, size=T).astype(np.int32)
    refs = [oracle.compress(wb, wf, per_row=True) for wf in wfs]
    y_ref = oracle.linear_multi(x, vid, [r[0] for r in refs], [r[1] for r in refs], True, wb)
    wb_d = to_dev(wb, dev)
    s_l, a_l = zip(*[gpu_compress(wb_d, to_dev(wf, dev), PR, dev) for wf in wfs])
    y = torch.empty((T, d_out), dtype=torch.float32, device=dev)
    ws = bd.new_workspace(bd.bd_linear_multi_workspace_size(T, V, d_out, d_in), dev)
    bd.bd_linear_multi(to_dev(x, dev), to_dev(vid, dev), list(s_l), list(a_l), PR, wb_d, y, ws)
    assert bd.bd_check_async(ws) == bd.BD_OK
    assert np.array_equal(y.cpu().numpy().astype(np.float64), y_ref)


def _multi_case(dev, seed, V, d_out, d_in, vid, per_row=True, f32=True):
    """Runs bd_linear_multi on dyadic inputs (every partial sum exact in fp32,
    so the result must equal the fp64 oracle bit for bit) and compares."""
    T = len(vid)
    wb, wfs, x = _dyadic_multi(seed, V, d_out, d_in, T)
    refs = [oracle.compress(wb, wf, per_row=per_row) for wf in wfs]
    y_ref = oracle.linear_multi(x, np.asarray(vid, np.int32), [r[0] for r in refs], [r[1] for r in refs],
                                per_row, wb)
    wb_d = to_dev(wb, dev)
    mode = PR if per_row else PM
    s_l, a_l = zip(*[gpu_compress(wb_d, to_dev(wf, dev), mode, dev) for wf in wfs])
    y = torch.empty((T, d_out), dtype=torch.float32 if f32 else torch.bfloat16, device=dev)
    ws = bd.new_workspace(bd.bd_linear_multi_workspace_size(T, V, d_out, d_in), dev)
    bd.bd_linear_multi(to_dev(x, dev), to_dev(np.asarray(vid, np.int32), dev), list(s_l), list(a_l), mode, wb_d, y, ws)
    assert bd.bd_check_async(ws) == bd.BD_OK
    if f32:
        assert np.array_equal(y.cpu().numpy().astype(np.float64), y_ref)
    else:
        check_linear(y_host(y), y_ref, bf16_out=True, what="multi bf16")


@pytest.mark.parametrize("d_in", [128, 384, 640, 2176, 4096, 6144, 8320])
def test_multi_partial_stages(dev, d_in):
    """d_in slices whose chunk count is not a multiple of the stage size (the
    stages' chunk loop takes its runtime path), a single-chunk d_in, and
    chunk counts between the cluster-size steps (17, 48 and 65 chunks of 128
    columns: one, two and four K slices of unequal length)."""
    vid = [0, 1, 2, -1, 1, 0, 3, 3, 2, 1, 0, 0, 4, -1, 2, 1]
    _multi_case(dev, 11 + d_in, 5, 70, d_in, vid)


def test_multi_prefill_4096_tokens_sampled_rows(dev, multi_problem):
    """Multi-tenant prefill: 4096 Zipf-routed tokens (40 of them base-model
    tokens) over the 14 variants of the multi-tenant workload take the grouped
    tensor-core path; sampled rows against the oracle, bf16 and fp32 output."""
    wb, wfs, _, _, _ = multi_problem
    rng = np.random.default_rng(21)
    T, V = 4096, len(wfs)
    vid = synth.zipf_variant_ids(rng, T, V)
    vid[rng.choice(T, 40, replace=False)] = -1
    x = synth.activations(rng, T, 8192)
    rows = synth.sample_rows(23, 8192, 32)
    refs = [oracle.compress_rows(wb, wf, rows) for wf in wfs]
    s_full, a_full = [], []
    for s_rows, a_rows in refs:
        sf = np.zeros((8192, 256), np.uint32)
        af = np.zeros(8192, np.float32)
        sf[rows], af[rows] = s_rows, a_rows
        s_full.append(sf)
        a_full.append(af)
    y_ref = oracle.linear_multi(x, vid, s_full, a_full, True, wb, rows=rows)
    wb_d = to_dev(wb, dev)
    s_l, a_l = zip(*[gpu_compress(wb_d, to_dev(wf, dev), PR, dev) for wf in wfs])
    x_d, vid_d = to_dev(x, dev), to_dev(vid, dev)
    ws = bd.new_workspace(bd.bd_linear_multi_workspace_size(T, V, 8192, 8192), dev)
    for f32 in (False, True):
        y = torch.empty((T, 8192), dtype=torch.float32 if f32 else torch.bfloat16, device=dev)
        bd.bd_linear_multi(x_d, vid_d, list(s_l), list(a_l), PR, wb_d, y, ws)
        assert bd.bd_check_async(ws) == bd.BD_OK
        check_linear(y_host(y)[:, rows], y_ref, bf16_out=not f32, what=f"multi prefill f32={f32}")


def _sized_vid(rng, sizes):
    """Token ids with exactly sizes[k] tokens of key k (key 0 = base model, id -1), shuffled."""
    vid = np.concatenate([np.full(n, k - 1, np.int32) for k, n in enumerate(sizes)])
    return vid[rng.permutation(len(vid))]


@pytest.mark.parametrize("case", ["random", "block_edges", "many_tails", "mixed_sizes", "one_variant", "all_base"])
def test_multi_prefill_exact(dev, case):
    """Grouped tensor-core prefill on dyadic inputs: exact against the oracle.
    Segments of 1, 255, 256 and 257 tokens (blocks ending at, before and after
    a 256-token boundary); 15 keys of 1 to 300 tokens (tails of every
    16-column MMA width, bf16 output too); segments of 250, 10, 300 and 129
    tokens after an empty base segment; a single variant, and a batch of
    base-model tokens only; ragged d_out."""
    rng = np.random.default_rng(len(case))
    if case == "random":
        V, vid = 5, rng.integers(-1, 5, size=700).astype(np.int32)
    elif case == "block_edges":
        V, vid = 4, _sized_vid(rng, [331, 256, 257, 1, 255])
    elif case == "many_tails":
        V, vid = 14, _sized_vid(rng, [5, 1, 2, 3, 15, 16, 17, 31, 33, 63, 64, 65, 100, 7, 300])
    elif case == "mixed_sizes":
        V, vid = 4, _sized_vid(rng, [0, 250, 10, 300, 129])
    elif case == "one_variant":
        V, vid = 1, np.zeros(512, np.int32)
    else:
        V, vid = 14, np.full(600, -1, np.int32)
    _multi_case(dev, 400 + len(vid), V, 200, 512, vid.tolist())
    if case == "many_tails":  # bf16 output as well
        _multi_case(dev, 400 + len(vid), V, 200, 512, vid.tolist(), f32=False)


def test_multi_wide_range_activations(dev):
    """Activations spanning 30 binades inside one token, an all-zero token, a
    token with one huge element and a token of subnormal-range values (the
    pre-scaled x operand of the recoded sign MMA stays exact for all of them):
    every output stays within the fp32 bound."""
    T, V, d_out, d_in = 12, 3, 96, 1024
    rng = np.random.default_rng(77)
    wb, wfs, _, _, _ = synth.multi_problem(77, d_out, d_in, T, V)
    xf = rng.standard_normal((T, d_in)) * 2.0 ** rng.uniform(-20, 10, size=(T, d_in))
    xf[1] = 0.0
    xf[2] = rng.standard_normal(d_in) * 1e-3
    xf[2, 17] = 3.0e4
    xf[3] = rng.standard_normal(d_in) * 1e-38
    x = synth.f32_to_bf16_bits(xf.astype(np.float32))
    vid = np.array([0, 1, 2, 0, 1, 2, 0, 1, 2, -1, 0, 1], np.int32)
    refs = [oracle.compress(wb, wf, per_row=True) for wf in wfs]
    y_ref = oracle.linear_multi(x, vid, [r[0] for r in refs], [r[1] for r in refs], True, wb)
    wb_d = to_dev(wb, dev)
    s_l, a_l = zip(*[gpu_compress(wb_d, to_dev(wf, dev), PR, dev) for wf in wfs])
    y = torch.empty((T, d_out), dtype=torch.float32, device=dev)
    ws = bd.new_workspace(bd.bd_linear_multi_workspace_size(T, V, d_out, d_in), dev)
    bd.bd_linear_multi(to_dev(x, dev), to_dev(vid, dev), list(s_l), list(a_l), PR, wb_d, y, ws)
    assert bd.bd_check_async(ws) == bd.BD_OK
    bound = fp32_bound_multi(x, wb, [r[1] for r in refs], vid, np.arange(d_out))
    got = y.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - y_ref) <= bound), float(np.max(np.abs(got - y_ref) / bound))
    assert np.array_equal(got[1], y_ref[1])  # an all-zero token gives exact zeros


@pytest.mark.parametrize("n_heavy", [33, 40, 64])
def test_multi_variant_with_many_tokens(dev, n_heavy):
    """One variant with more than 32 tokens: its 5..8 padded tiles run as two
    phases (at most 4 tiles each)."""
    rng = np.random.default_rng(n_heavy)
    vid = np.full(64, 2, np.int32)
    others = rng.choice(64, 64 - n_heavy, replace=False)
    vid[others] = rng.integers(-1, 4, size=len(others))
    vid[others[vid[others] == 2]] = 1
    _multi_case(dev, 100 + n_heavy, 4, 160, 512, vid.tolist())


@pytest.mark.parametrize("V", [24, 30, 64])
def test_multi_many_variants_small_groups(dev, V):
    """Many variants: token groups shrink so that no group needs more padded
    tiles than tensor memory holds; 64 tokens over V variants."""
    rng = np.random.default_rng(V)
    vid = rng.integers(-1, V, size=64).astype(np.int32)
    _multi_case(dev, 200 + V, V, 129, 256, vid.tolist())


@pytest.mark.parametrize("T", [1, 7, 8, 9, 17, 33, 63])
def test_multi_token_counts(dev, T):
    """Token counts at and around the 8/16/32/64 tile boundaries, per-matrix
    alpha, bf16 output, ragged d_out."""
    rng = np.random.default_rng(T)
    vid = rng.integers(-1, 6, size=T).astype(np.int32)
    _multi_case(dev, 300 + T, 6, 200, 1024, vid.tolist(), per_row=False, f32=False)


def test_multi_bad_variant_flagged_and_computed_as_base(dev):
    V, d_out, d_in, T = 3, 20, 256, 12
    wb, wfs, x = _dyadic_multi(9, V, d_out, d_in, T)
    vid = np.array([0, 1, 2, -1, 7, -3, 2, 1, 0, 3, -1, 1], np.int32)
    refs = [oracle.compress(wb, wf, per_row=True) for wf in wfs]
    y_ref = oracle.linear_multi(x, vid, [r[0] for r in refs], [r[1] for r in refs], True, wb)
    wb_d = to_dev(wb, dev)
    s_l, a_l = zip(*[gpu_compress(wb_d, to_dev(wf, dev), PR, dev) for wf in wfs])
    y = torch.empty((T, d_out), dtype=torch.float32, device=dev)
    ws = bd.new_workspace(bd.bd_linear_multi_workspace_size(T, V, d_out, d_in), dev)
    bd.bd_linear_multi(to_dev(x, dev), to_dev(vid, dev), list(s_l), list(a_l), PR, wb_d, y, ws)
    assert bd.bd_check_async(ws) == bd.BD_ERR_BAD_VARIANT
    assert np.array_equal(y.cpu().numpy().astype(np.float64), y_ref)


# ============================================================================ router

@pytest.mark.parametrize("T,V", [(0, 3), (1, 0), (1, 1), (64, 14), (1000, 64), (5000, 7)])
def test_route_bit_exact(dev, T, V):
    rng = np.random.default_rng(T * 3 + V)
    vid = rng.integers(-1, max(V, 1), size=T).astype(np.int32) if V > 0 else -np.ones(T, np.int32)
    perm_ref, seg_ref, n_bad = oracle.route(vid, V)
    vid_d = to_dev(vid, dev) if T else torch.zeros(1, dtype=torch.int32, device=dev)
    perm = torch.full((max(T, 1),), -7, dtype=torch.int32, device=dev)
    seg = torch.full((V + 2,), -7, dtype=torch.int32, device=dev)
    ws = bd.new_workspace(bd.bd_route_workspace_size(T, V), dev)
    lib = bd.load()
    st = torch.cuda.current_stream().cuda_stream
    assert lib.bd_route(vid_d.data_ptr(), T, V, perm.data_ptr(), seg.data_ptr(), ws.data_ptr(), ws.numel(),
                        st) == bd.BD_OK
    assert bd.bd_check_async(ws) == (bd.BD_OK if n_bad == 0 else bd.BD_ERR_BAD_VARIANT)
    assert np.array_equal(perm.cpu().numpy()[:T], perm_ref)
    assert np.array_equal(seg.cpu().numpy(), seg_ref)


def test_route_flags_out_of_range(dev):
    vid = np.array([2, -1, 9, 0, -4, 1], np.int32)
    perm_ref, seg_ref, n_bad = oracle.route(vid, 3)
    assert n_bad == 2
    perm = torch.empty(6, dtype=torch.int32, device=dev)
    seg = torch.empty(5, dtype=torch.int32, device=dev)
    ws = bd.new_workspace(256, dev)
    bd.bd_route(to_dev(vid, dev), 3, perm, seg, ws)
    assert bd.bd_check_async(ws) == bd.BD_ERR_BAD_VARIANT
    assert np.array_equal(perm.cpu().numpy(), perm_ref)
    assert np.array_equal(seg.cpu().numpy(), seg_ref)


# ============================================================================ invariants / hygiene

@pytest.mark.parametrize("mode", [PR, PM])
def test_reconstruction_invariants_on_device(dev, mode):
    wb, wf, _ = synth.single_problem(31, 64, 512, 1)
    wb_d = to_dev(wb, dev)
    s, a = gpu_compress(wb_d, to_dev(wf, dev), mode, dev)
    weff = torch.empty((64, 512), dtype=torch.float32, device=dev)
    bd.bd_debug_reconstruct(wb_d, s, a, mode, weff)
    torch.cuda.synchronize()
    w = synth.bf16_bits_to_f32(wb).astype(np.float64)
    al = a.cpu().numpy().astype(np.float64)
    al = al[:, None] if mode == PR else al[0]
    diff = weff.cpu().numpy().astype(np.float64) - w
    delta = synth.bf16_bits_to_f32(wf).astype(np.float64) - w
    code = np.where(delta < 0, -1.0, 1.0)
    assert np.array_equal(np.sign(diff), code)  # sign(W_eff - W_base) = sign(Delta), sign(0) = +1
    np.testing.assert_allclose(np.abs(diff), np.broadcast_to(al, diff.shape), rtol=2 ** -16)  # |.| = alpha


def test_canary_guards_untouched(dev):
    """Outputs written inside larger buffers: the 64 KiB of 0xA5 after each must survive."""
    guard = 65536
    d_out, d_in, T = 37, 384, 19
    wb, wf, x = synth.single_problem(41, d_out, d_in, T)
    wb_d, wf_d, x_d = to_dev(wb, dev), to_dev(wf, dev), to_dev(x, dev)
    n_s = d_out * d_in // 32
    sbuf = torch.full((n_s + guard // 4,), -1515870811, dtype=torch.int32, device=dev)  # 0xA5A5A5A5
    abuf = torch.full((d_out + guard // 4,), 0.0, dtype=torch.float32, device=dev)
    abuf.view(torch.int32)[:] = -1515870811
    ybuf = torch.empty((T * d_out + guard // 4,), dtype=torch.float32, device=dev)
    ybuf.view(torch.int32)[:] = -1515870811
    ws = bd.new_workspace(bd.bd_linear_multi_workspace_size(T, 1, d_out, d_in), dev)
    s = sbuf[:n_s].view(d_out, d_in // 32)
    a = abuf[:d_out]
    bd.bd_compress(wb_d, wf_d, PR, s, a, ws)
    y = ybuf[:T * d_out].view(T, d_out)
    bd.bd_linear(x_d, wb_d, s, a, PR, y, ws)
    bd.bd_linear_multi(x_d, torch.zeros(T, dtype=torch.int32, device=dev), [s], [a], PR, wb_d, y, ws)
    assert bd.bd_check_async(ws) == bd.BD_OK
    for buf, n in ((sbuf, n_s), (abuf.view(torch.int32), d_out), (ybuf.view(torch.int32), T * d_out)):
        assert bool((buf[n:] == -1515870811).all())


def test_argument_errors(dev):
    lib = bd.load()
    st = torch.cuda.current_stream().cuda_stream
    wb = torch.zeros((16, 256), dtype=torch.int16, device=dev)
    s = torch.zeros((16, 8), dtype=torch.int32, device=dev)
    a = torch.zeros(16, dtype=torch.float32, device=dev)
    x = torch.zeros((4, 256), dtype=torch.int16, device=dev)
    y = torch.zeros((4, 16), dtype=torch.float32, device=dev)
    ws = bd.new_workspace(1024, dev)
    P = lambda t, off=0: t.data_ptr() + off  # noqa: E731
    assert lib.bd_linear(P(x, 2), 4, P(wb), P(s), P(a), PR, 16, 256, P(y), 1, P(ws), 1024, st) == bd.BD_ERR_MISALIGNED
    assert lib.bd_linear(P(x), 4, P(wb), P(s), P(a), PR, 16, 96, P(y), 1, P(ws), 1024, st) == \
        bd.BD_ERR_UNSUPPORTED_SHAPE
    assert lib.bd_linear(P(x), 4, P(wb), P(s), P(a), PR, 16, 256, P(y), 1, P(ws), 16, st) == bd.BD_ERR_WORKSPACE
    assert lib.bd_linear(P(x), 4, P(wb), P(s), P(a), PR, 16, 256, P(x), 1, P(ws), 1024, st) == \
        bd.BD_ERR_INVALID_ARG  # y aliases x
    assert lib.bd_linear(P(x), 4, P(wb), P(s), P(a), 7, 16, 256, P(y), 1, P(ws), 1024, st) == bd.BD_ERR_INVALID_ARG
    tab = (ctypes.c_void_p * 1)(P(s))
    atab = (ctypes.c_void_p * 1)(P(a))
    vid = torch.zeros(4, dtype=torch.int32, device=dev)
    assert lib.bd_linear_multi(P(x), 4, P(vid), 0, ctypes.addressof(tab), ctypes.addressof(atab), PR, P(wb), 16, 256,
                               P(y), 1, P(ws), 1024, st) == bd.BD_ERR_INVALID_ARG  # V = 0
    assert lib.bd_compress(P(wb), P(wb), 16, 256, PR, P(s), P(a), P(ws, 16), 1000, st) == bd.BD_ERR_MISALIGNED
