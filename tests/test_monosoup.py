"""MonoSoup merge on the GPU (bd_monosoup_merge) against the fp64 oracle:
section "MonoSoup" of the BitDelta post, tau_i = the rank-r truncated SVD of
Delta_i = W_i - W_base and W_merged = W_base + (1/k) sum_i tau_i.

The GPU computes the truncated SVD by randomized subspace iteration, the
oracle by a full SVD.  Two kinds of inputs:
  - rank-r task vectors (log-spaced singular values 4..1) plus only the bf16
    rounding of the checkpoints: the spectral gap at r is about 1e-3 and
    after one power iteration the two agree to fp32 accuracy;
  - the same plus Laplace(0, 1e-3) noise in every element (a noise floor of
    real size, which the truncation is meant to remove): there the
    randomized result meets an elementwise bound derived from the singular
    values of each task vector (``subspace_bound``)."""
import numpy as np
import pytest
import torch

import oracle
from bit_weight_delta_bd_gb300 import bitdelta as bd
from bit_weight_delta_bd_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available()
    import __graft_entry__

    __graft_entry__.build()
    return torch.device("cuda:0")


def to_dev(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)


def run_gpu(dev, wb, ws, om, rank, l, q, out_dtype):
    d_out, d_in = wb.shape
    wb_d = to_dev(wb, dev)
    ws_d = [to_dev(w, dev) for w in ws]
    om_d = torch.from_numpy(om).to(dev) if om is not None else None
    out = torch.empty((d_out, d_in), dtype=out_dtype, device=dev)
    wsp = bd.new_workspace(bd.bd_monosoup_workspace_size(d_out, d_in, len(ws), rank, l), dev)
    bd.bd_monosoup_merge(wb_d, ws_d, rank, l, q, om_d, out, wsp)
    assert bd.bd_check_async(wsp) == bd.BD_OK  # no bounded wait gave up
    return out.cpu()


def bf16_ulp(v):
    """Spacing of bf16 numbers at |v| (8 significant bits)."""
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -126)))
    return 2.0 ** (e - 7)


@pytest.mark.parametrize("d_out,d_in,k,r,l,q", [
    (256, 384, 3, 8, 16, 1),     # several tiles of every pass
    (300, 256, 2, 16, 24, 1),    # ragged rows
    (1000, 512, 4, 12, 32, 2),   # two power iterations, k = 4
    (8, 128, 2, 4, 16, 1),       # fewer rows than sketch columns (rank-deficient sketch)
    (512, 640, 1, 32, 64, 1),    # the widest sketch
])
def test_monosoup_matches_exact_truncated_svd(dev, d_out, d_in, k, r, l, q):
    wb, ws = synth.monosoup_checkpoints(7 + d_out, d_out, d_in, k, min(r, d_out))
    om = synth.gaussian_test_matrix(11 + d_in, d_in, l)
    ref = oracle.monosoup_merge(wb, ws, r)
    base = oracle.bf16_to_f64(wb)
    upd_ref = ref - base
    got = run_gpu(dev, wb, ws, om, r, l, q, torch.float32).double().numpy()
    rel = np.linalg.norm((got - base) - upd_ref) / np.linalg.norm(upd_ref)
    assert rel <= 1e-4, f"relative error of the merged update {rel:.3e}"
    # bf16 output: one rounding of a value this close to the oracle's lands
    # on one of the two bf16 neighbours of the exact result; near zero the
    # fp32 error of the update (about 1e-7 of its largest entry) dominates
    gb = run_gpu(dev, wb, ws, om, r, l, q, torch.bfloat16).float().double().numpy()
    assert np.all(np.abs(gb - ref) <= bf16_ulp(ref) + 1e-6 * np.abs(upd_ref).max())


@pytest.mark.parametrize("d_out,d_in,k,r,l,q", [
    (256, 384, 10, 4, 16, 1),    # two batches of checkpoints (8 + 2)
    (200, 256, 17, 4, 8, 1),     # three batches (8 + 8 + 1), ragged rows
    (512, 640, 3, 24, 64, 1),    # l = 64: CUDA-core products, three checkpoints in one batch
    (256, 384, 10, 24, 64, 1),   # k l r = 15360: the merge factors read U from device memory, two batches
])
def test_monosoup_batches_and_wide_sketches(dev, d_out, d_in, k, r, l, q):
    wb, ws = synth.monosoup_checkpoints(23 + k, d_out, d_in, k, min(r, d_out))
    om = synth.gaussian_test_matrix(29 + l, d_in, l)
    ref = oracle.monosoup_merge(wb, ws, r)
    base = oracle.bf16_to_f64(wb)
    upd_ref = ref - base
    got = run_gpu(dev, wb, ws, om, r, l, q, torch.float32).double().numpy()
    rel = np.linalg.norm((got - base) - upd_ref) / np.linalg.norm(upd_ref)
    assert rel <= 1e-4, f"relative error of the merged update {rel:.3e}"


def subspace_bound(delta: np.ndarray, omega: np.ndarray, r: int, q: int) -> float:
    """Elementwise bound on |tau_randomized - tau_exact| for one task vector,
    in exact arithmetic.  With sigma_j the singular values of Delta, V its
    right singular vectors, gamma = sigma_(r+1) / sigma_r, Omega_1 = V_r^T
    Omega and Omega_2 = V_perp^T Omega, randomized subspace iteration with q
    power iterations gives a basis Q whose angle to the top-r left singular
    subspace U_r satisfies sin(theta) <= s = gamma^(2q+1) ||Omega_2
    Omega_1^+||_2 (Saibaba 2019, "Randomized subspace iteration: analysis of
    canonical angles and unitarily invariant norms", Thm. 1).  The rank-r
    truncation of Q^T Delta then spans U_hat with sin(U_hat, U_r) <= s +
    gamma s / (sqrt(1 - s^2) - gamma) (Wedin's theorem applied inside
    range(Q): the part of Delta outside U_r moves the subspace by at most
    sigma_(r+1) s over the gap).  Both truncations are projections of Delta
    (tau = U_r U_r^T Delta, tau_hat = U_hat U_hat^T Delta), so every entry of
    their difference is at most sin(U_hat, U_r) sigma_1."""
    u, sv, vh = np.linalg.svd(delta, full_matrices=False)
    g = sv[r] / sv[r - 1] if r < len(sv) else 0.0
    v = vh.T
    o1, o2 = v[:, :r].T @ omega, v[:, r:].T @ omega
    s = min(1.0, g ** (2 * q + 1) * np.linalg.norm(o2 @ np.linalg.pinv(o1), 2))
    if s >= 1.0 or np.sqrt(1 - s * s) <= g:
        return float(sv[0])
    return float(sv[0] * (s + g * s / (np.sqrt(1 - s * s) - g)))


@pytest.mark.parametrize("d_out,d_in,k,r,l,q", [
    (512, 768, 3, 8, 16, 1),
    (512, 768, 3, 8, 16, 2),
    (1024, 1024, 3, 16, 32, 2),
    (300, 512, 2, 8, 24, 3),
])
def test_monosoup_noisy_task_vectors_elementwise(dev, d_out, d_in, k, r, l, q):
    """Task vectors = rank-r signal + Laplace(0, 1e-3) noise.  Elementwise:
    |W_gpu - W_oracle| <= (1/k) sum_i subspace_bound_i + an fp32 term of
    2^-16 sigma_1 (the sketches and projections are fp32 sums of at most
    d_in or d_out exact products, the bases are orthonormalised through
    float-float Gram matrices and Cholesky factors; 256 fp32 roundings of the
    largest singular value cover them with room to spare).  bf16 output: the
    same plus half a bf16 ulp."""
    wb, ws = synth.monosoup_noisy_checkpoints(17 + d_out, d_out, d_in, k, r)
    om = synth.gaussian_test_matrix(19 + d_in, d_in, l)
    ref = oracle.monosoup_merge(wb, ws, r)
    base = oracle.bf16_to_f64(wb)
    deltas = [oracle.bf16_to_f64(w) - base for w in ws]
    alg = sum(subspace_bound(dl, om.astype(np.float64), r, q) for dl in deltas) / k
    sig1 = max(np.linalg.norm(dl, 2) for dl in deltas)
    bound = alg + 2.0 ** -16 * sig1
    upd = ref - base
    assert bound < 0.05 * np.abs(upd).max() or q == 1, "the bound must say something at q >= 2"
    got = run_gpu(dev, wb, ws, om, r, l, q, torch.float32).double().numpy()
    err = np.abs(got - ref)
    assert err.max() <= bound, f"max |err| {err.max():.3e} > bound {bound:.3e}"
    rel = np.linalg.norm((got - base) - upd) / np.linalg.norm(upd)
    assert rel <= 1e-3, rel
    gb = run_gpu(dev, wb, ws, om, r, l, q, torch.bfloat16).float().double().numpy()
    assert np.all(np.abs(gb - ref) <= bound + bf16_ulp(ref) / 2)


def test_monosoup_without_power_iteration(dev):
    """q = 0: the range finder alone; the error is set by the spectral gap
    (about 1e-3 here), not by the arithmetic."""
    wb, ws = synth.monosoup_checkpoints(3, 256, 256, 2, 8)
    om = synth.gaussian_test_matrix(4, 256, 24)
    ref = oracle.monosoup_merge(wb, ws, 8)
    base = oracle.bf16_to_f64(wb)
    got = run_gpu(dev, wb, ws, om, 8, 24, 0, torch.float32).double().numpy()
    rel = np.linalg.norm((got - base) - (ref - base)) / np.linalg.norm(ref - base)
    assert rel <= 1e-2


def test_monosoup_rank_zero_is_the_base(dev):
    wb, ws = synth.monosoup_checkpoints(5, 64, 256, 3, 4)
    got = run_gpu(dev, wb, ws, None, 0, 8, 1, torch.bfloat16)
    assert np.array_equal(got.view(torch.int16).numpy().view(np.uint16), wb)


def test_monosoup_full_rank_one_checkpoint(dev):
    """k = 1 and rank = d_out <= l: the sketch spans every row direction, so
    the merge returns the checkpoint itself (to fp32 accuracy)."""
    wb, ws = synth.monosoup_checkpoints(6, 16, 256, 1, 16)
    om = synth.gaussian_test_matrix(8, 256, 32)
    got = run_gpu(dev, wb, ws, om, 16, 32, 1, torch.float32).double().numpy()
    np.testing.assert_allclose(got, oracle.bf16_to_f64(ws[0]), rtol=0, atol=2e-6)


@pytest.mark.parametrize("name,d_out,d_in,k,spectrum,l,q", [
    # two clusters of four equal singular values
    ("clusters", 512, 384, 2, [2.0] * 4 + [1.0] * 4, 16, 1),
    # one cluster of sixteen: every leading eigenvalue of the projected problem the same
    ("one_cluster", 640, 512, 3, [1.5] * 16, 32, 1),
    # a slow decay: neighbouring eigenvalues about 0.3 % of the largest apart, just
    # outside any cluster, where inverse iteration alone leaves the vectors
    # about 1e-4 from orthogonal
    ("slow_decay", 640, 512, 3, [2.0 * (1.0 - 0.0015 * j) for j in range(16)], 32, 1),
])
def test_monosoup_repeated_and_close_singular_values(dev, name, d_out, d_in, k, spectrum, l, q):
    """Task vectors whose leading singular values repeat or nearly repeat
    (beyond them only the bf16 rounding of the checkpoints): the truncation
    at r = len(spectrum) is still unique, and the randomized result must
    match it to fp32 accuracy whatever basis of a repeated singular subspace
    the eigensolver picks."""
    r = len(spectrum)
    wb, ws = synth.monosoup_spectrum_checkpoints(31 + d_out + r, d_out, d_in, k, spectrum)
    om = synth.gaussian_test_matrix(37 + d_in, d_in, l)
    ref = oracle.monosoup_merge(wb, ws, r)
    base = oracle.bf16_to_f64(wb)
    upd_ref = ref - base
    got = run_gpu(dev, wb, ws, om, r, l, q, torch.float32).double().numpy()
    rel = np.linalg.norm((got - base) - upd_ref) / np.linalg.norm(upd_ref)
    assert rel <= 1e-4, f"{name}: relative error of the merged update {rel:.3e}"


def test_monosoup_zero_task_vector(dev):
    """One checkpoint equal to the base (Delta = 0: every pivot of its
    CholeskyQR is dropped and its eigenproblem is the zero matrix): its term
    is zero and the merge is W_base + (1/3)(tau_1 + tau_2)."""
    wb, ws = synth.monosoup_checkpoints(41, 384, 256, 2, 8)
    ws = [ws[0], wb.copy(), ws[1]]
    om = synth.gaussian_test_matrix(43, 256, 16)
    ref = oracle.monosoup_merge(wb, ws, 8)
    base = oracle.bf16_to_f64(wb)
    got = run_gpu(dev, wb, ws, om, 8, 16, 1, torch.float32).double().numpy()
    rel = np.linalg.norm((got - base) - (ref - base)) / np.linalg.norm(ref - base)
    assert rel <= 1e-4, rel


@pytest.mark.parametrize("d_out,d_in,k,l", [
    (4, 128, 2, 4),     # the narrowest sketch, rank = l = d_out
    (64, 256, 1, 64),   # the widest sketch, rank = l = d_out (CUDA-core products)
])
def test_monosoup_rank_equals_sketch_width(dev, d_out, d_in, k, l):
    """rank = l = d_out: every eigenvector of the projected problem is kept
    and the sketch spans every row direction, so each tau_i is Delta_i and
    the merge is the mean of the checkpoints (to fp32 accuracy)."""
    wb, ws = synth.monosoup_checkpoints(47 + l, d_out, d_in, k, d_out)
    om = synth.gaussian_test_matrix(53 + l, d_in, l)
    got = run_gpu(dev, wb, ws, om, l, l, 1, torch.float32).double().numpy()
    ref = oracle.monosoup_merge(wb, ws, l)
    np.testing.assert_allclose(ref, sum(oracle.bf16_to_f64(w) for w in ws) / k, rtol=0, atol=1e-12)
    np.testing.assert_allclose(got, ref, rtol=0, atol=4e-6)


def test_monosoup_ffn_sized(dev):
    """2048 x 2048, 3 checkpoints, rank 16: the oracle's full SVD still runs
    in seconds; the same bound as the small cases."""
    wb, ws = synth.monosoup_checkpoints(9, 2048, 2048, 3, 16)
    om = synth.gaussian_test_matrix(10, 2048, 32)
    ref = oracle.monosoup_merge(wb, ws, 16)
    base = oracle.bf16_to_f64(wb)
    got = run_gpu(dev, wb, ws, om, 16, 32, 1, torch.float32).double().numpy()
    rel = np.linalg.norm((got - base) - (ref - base)) / np.linalg.norm(ref - base)
    assert rel <= 1e-4, rel
