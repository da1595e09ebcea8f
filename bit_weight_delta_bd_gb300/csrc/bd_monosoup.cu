// MonoSoup merge of k fine-tuned checkpoints of one base matrix (section
// "MonoSoup" of the BitDelta post):
//
//   Delta_i = W_i - W_base,  tau_i = rank-r truncated SVD of Delta_i,
//   W_merged = W_base + (1/k) * sum_i tau_i.
//
// The truncated SVD is computed by randomized subspace iteration (Halko,
// Martinsson and Tropp, "Finding structure with randomness", 2011: the range
// finder with power iterations, then the SVD of the small projected matrix):
//   Y = Delta * Omega          (Omega [d_in][l], Gaussian, given by the caller)
//   Q = orth(Y); q times: Z = orth(Delta^T Q), Q = orth(Delta Z)
//   B^T = Delta^T Q            ([d_in][l])
//   B B^T = U_B Lambda U_B^T   (l x l symmetric eigenproblem, Jacobi)
//   tau = (Q U_r) (U_r^T B)    (U_r: the r leading eigenvectors)
// which is U_r S_r V_r^T of the rank-l approximation Q Q^T Delta.  Every pass
// over Delta reads W_i and W_base (bf16) and forms Delta in fp32 on the fly.
// Orthonormalisation is CholeskyQR: the Gram matrix is accumulated in fp64,
// factored in one CTA, and Y <- Y R^-1 applied (twice, CholeskyQR2, for the
// final basis); directions whose pivot falls below 1e-12 of the largest are
// dropped (rank-deficient sketches).
// The merge is one pass: W_base + (1/k) [L_1 .. L_k][R_1 .. R_k]^T with
// L_i = Q_i U_r, R_i = B_i^T U_r, rounded once to the output type.
//
// All arithmetic is fp32 on the CUDA cores except the Gram matrices and the
// Cholesky factor (fp64).  No kernel waits on another CTA; the passes are
// plain stream-ordered launches.
#include <cuda_bf16.h>

#include <cmath>

#include <atomic>

#include "bd_device.cuh"
#include "bd_tma.h"

namespace bd {
namespace {

constexpr int kMaxL = 64;        // sketch width l (columns of Y, Q, B^T)
constexpr int kGramBlocks = 152;  // CTAs of one Gram pass (fixed-order fp64 partials)
constexpr int kSlices = 16;       // split of the long dimension in the two products with Delta
// dynamic shared memory of the Cholesky kernel: two fp64 [64][65] matrices
constexpr size_t kSmallSmem = 2 * sizeof(double) * kMaxL * (kMaxL + 1);

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// Delta for 8 consecutive columns from two 16-byte loads of bf16 bits.
__device__ __forceinline__ void delta8(const uint16_t* w, const uint16_t* wb, float* out)
{
    const uint4 a = *reinterpret_cast<const uint4*>(w);
    const uint4 b = *reinterpret_cast<const uint4*>(wb);
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        out[2 * q] = bf16_bits_to_float(av[q] & 0xFFFFu) - bf16_bits_to_float(bv[q] & 0xFFFFu);
        out[2 * q + 1] = bf16_bits_to_float(av[q] >> 16) - bf16_bits_to_float(bv[q] >> 16);
    }
}

// ypart[s][row][c] = sum over slice s of the columns j of Delta[row][j] *
// Om[j][c]  (c < l).  32 rows per CTA, blockIdx.y = slice (cols_per columns,
// a multiple of 64), 64-column chunks; each thread holds 2 rows x NC columns.
// NC = output columns per thread (kW = 16 NC columns per CTA, kW >= l).
template <int NC>
__global__ void __launch_bounds__(256) sketch_kernel(const uint16_t* __restrict__ w, const uint16_t* __restrict__ wb,
                                                     int64_t d_out, int64_t d_in, const float* __restrict__ om, int l,
                                                     int64_t cols_per, float* __restrict__ ypart)
{
    constexpr int kW = 16 * NC;
    const int64_t jbeg = static_cast<int64_t>(blockIdx.y) * cols_per;
    const int64_t jend = jbeg + cols_per < d_in ? jbeg + cols_per : d_in;
    float* y = ypart + static_cast<int64_t>(blockIdx.y) * d_out * l;
    __shared__ float sd[32][65];
    __shared__ __align__(16) float so[64][kW];
    const int tid = threadIdx.x;
    const int64_t r0 = static_cast<int64_t>(blockIdx.x) * 32;
    const int tr = (tid >> 4) * 2, tc = (tid & 15) * NC;
    float acc[2][NC] = {};
    for (int64_t j0 = jbeg; j0 < jend; j0 += 64) {
        {
            const int rr = tid >> 3, cc = (tid & 7) * 8;
            const int64_t row = r0 + rr;
            float d[8] = {};
            if (row < d_out) delta8(w + row * d_in + j0 + cc, wb + row * d_in + j0 + cc, d);
#pragma unroll
            for (int q = 0; q < 8; ++q) sd[rr][cc + q] = d[q];
        }
        for (int e = tid; e < 64 * kW; e += 256) {
            const int jj = e / kW, c = e % kW;
            so[jj][c] = c < l ? om[(j0 + jj) * l + c] : 0.0f;
        }
        __syncthreads();
#pragma unroll 8
        for (int jj = 0; jj < 64; ++jj) {
            const float a0 = sd[tr][jj], a1 = sd[tr + 1][jj];
            float o[NC];
#pragma unroll
            for (int q = 0; q < NC; ++q) o[q] = so[jj][tc + q];
#pragma unroll
            for (int q = 0; q < NC; ++q) {
                acc[0][q] = fmaf(a0, o[q], acc[0][q]);
                acc[1][q] = fmaf(a1, o[q], acc[1][q]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int x = 0; x < 2; ++x) {
        const int64_t row = r0 + tr + x;
        if (row >= d_out) continue;
#pragma unroll
        for (int q = 0; q < NC; ++q)
            if (tc + q < l) y[row * l + tc + q] = acc[x][q];
    }
}

// btpart[s][j][c] = sum over slice s of the rows of Delta[row][j] *
// Q[row][c]  (c < l).  32 columns of Delta per CTA, blockIdx.y = slice
// (rows_per rows, a multiple of 64), 64-row chunks; each thread holds 2
// columns x NC.
template <int NC>
__global__ void __launch_bounds__(256) left_kernel(const uint16_t* __restrict__ w, const uint16_t* __restrict__ wb,
                                                   int64_t d_out, int64_t d_in, const float* __restrict__ q, int l,
                                                   int64_t rows_per, float* __restrict__ btpart)
{
    constexpr int kW = 16 * NC;
    const int64_t rbeg = static_cast<int64_t>(blockIdx.y) * rows_per;
    const int64_t rend = rbeg + rows_per < d_out ? rbeg + rows_per : d_out;
    float* bt = btpart + static_cast<int64_t>(blockIdx.y) * d_in * l;
    __shared__ float sd[64][33];
    __shared__ __align__(16) float sq[64][kW];
    const int tid = threadIdx.x;
    const int64_t j0 = static_cast<int64_t>(blockIdx.x) * 32;
    const int tj = (tid >> 4) * 2, tc = (tid & 15) * NC;
    float acc[2][NC] = {};
    for (int64_t r0 = rbeg; r0 < rend; r0 += 64) {
        {
            const int rr = tid >> 2, cc = (tid & 3) * 8;
            const int64_t row = r0 + rr;
            float d[8] = {};
            if (row < rend) delta8(w + row * d_in + j0 + cc, wb + row * d_in + j0 + cc, d);
#pragma unroll
            for (int e = 0; e < 8; ++e) sd[rr][cc + e] = d[e];
        }
        for (int e = tid; e < 64 * kW; e += 256) {
            const int rr = e / kW, c = e % kW;
            const int64_t row = r0 + rr;
            sq[rr][c] = (c < l && row < rend) ? q[row * l + c] : 0.0f;
        }
        __syncthreads();
#pragma unroll 8
        for (int rr = 0; rr < 64; ++rr) {
            const float a0 = sd[rr][tj], a1 = sd[rr][tj + 1];
            float o[NC];
#pragma unroll
            for (int qq = 0; qq < NC; ++qq) o[qq] = sq[rr][tc + qq];
#pragma unroll
            for (int qq = 0; qq < NC; ++qq) {
                acc[0][qq] = fmaf(a0, o[qq], acc[0][qq]);
                acc[1][qq] = fmaf(a1, o[qq], acc[1][qq]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int qq = 0; qq < NC; ++qq)
            if (tc + qq < l) bt[(j0 + tj + x) * l + tc + qq] = acc[x][qq];
}

// out[e] = sum_s part[s][e], e < n (fixed order).
__global__ void __launch_bounds__(256) sum_slices_kernel(const float* __restrict__ part, int nslice, int64_t n,
                                                         float* __restrict__ out)
{
    const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (e >= n) return;
    float s = part[e];
    for (int k = 1; k < nslice; ++k) s += part[k * n + e];
    out[e] = s;
}

// Partial Gram matrices of A [n][l]: CTA b sums A^T A over its contiguous row
// range in fp64 into part[b][l * l] (entry i * l + j).
__global__ void __launch_bounds__(256) gram_kernel(const float* __restrict__ a, int64_t n, int l,
                                                   double* __restrict__ part)
{
    __shared__ double sa[32][kMaxL + 1];  // converted once per element, not once per product
    const int tid = threadIdx.x;
    const int64_t per = (n + kGramBlocks - 1) / kGramBlocks;
    const int64_t b0 = static_cast<int64_t>(blockIdx.x) * per;
    const int64_t b1 = b0 + per < n ? b0 + per : n;
    const int ll = l * l;
    double acc[16];
#pragma unroll
    for (int m = 0; m < 16; ++m) acc[m] = 0.0;
    for (int64_t r0 = b0; r0 < b1; r0 += 32) {
        for (int e = tid; e < 32 * kMaxL; e += 256) {
            const int rr = e / kMaxL, c = e % kMaxL;
            const int64_t row = r0 + rr;
            sa[rr][c] = (row < b1 && c < l) ? static_cast<double>(a[row * l + c]) : 0.0;
        }
        __syncthreads();
        for (int rr = 0; rr < 32; ++rr) {
#pragma unroll
            for (int m = 0; m < 16; ++m) {
                const int p = tid + 256 * m;
                if (p < ll) acc[m] = fma(sa[rr][p / l], sa[rr][p % l], acc[m]);
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int m = 0; m < 16; ++m) {
        const int p = tid + 256 * m;
        if (p < ll) part[static_cast<int64_t>(blockIdx.x) * ll + p] = acc[m];
    }
}

// g[e] = sum_b part[b][e], e < l * l (fixed order, one thread per entry).
__global__ void __launch_bounds__(256) gram_sum_kernel(const double* __restrict__ part, int l, double* __restrict__ g)
{
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    const int ll = l * l;
    if (e >= ll) return;
    double s = 0.0;
    for (int b = 0; b < kGramBlocks; ++b) s += part[static_cast<int64_t>(b) * ll + e];
    g[e] = s;
}

// Loads the summed Gram matrix G [l][l] into g[64][65], zero past l.
__device__ __forceinline__ void load_gram(const double* __restrict__ G, int l, double (*g)[kMaxL + 1])
{
    for (int e = threadIdx.x; e < kMaxL * kMaxL; e += blockDim.x) {
        const int i = e >> 6, j = e & 63;
        g[i][j] = (i < l && j < l) ? G[i * l + j] : 0.0;
    }
}

// One CTA: G = R^T R (Cholesky, R upper); minv = R^-1
// as fp32 [l][l].  A pivot below 1e-12 of the largest diagonal entry drops
// its direction (its row and column of R^-1 are zero).
__global__ void __launch_bounds__(256) chol_inv_kernel(const double* __restrict__ G, int l,
                                                       float* __restrict__ minv)
{
    extern __shared__ double dsm[];  // kSmallSmem bytes: g, then ri
    double (*g)[kMaxL + 1] = reinterpret_cast<double (*)[kMaxL + 1]>(dsm);
    double (*ri)[kMaxL + 1] = reinterpret_cast<double (*)[kMaxL + 1]>(dsm + kMaxL * (kMaxL + 1));
    __shared__ double dmax;
    __shared__ int dead[kMaxL];
    const int tid = threadIdx.x;
    load_gram(G, l, g);
    __syncthreads();
    if (tid == 0) {
        double m = 0.0;
        for (int i = 0; i < l; ++i) m = fmax(m, g[i][i]);
        dmax = m;
    }
    __syncthreads();
    const double tol = 1e-12 * dmax;
    for (int k = 0; k < l; ++k) {
        // g holds the trailing Schur complement; row k of R replaces row k of g
        const double d = g[k][k];
        const bool live = d > tol && d > 0.0;
        __syncthreads();
        if (tid == 0) dead[k] = live ? 0 : 1;
        const double rkk = live ? sqrt(d) : 0.0;
        const double inv = live ? 1.0 / rkk : 0.0;
        for (int j = k + tid; j < l; j += blockDim.x) g[k][j] = live ? (j == k ? rkk : g[k][j] * inv) : 0.0;
        __syncthreads();
        for (int e = tid; e < l * l; e += blockDim.x) {
            const int i = e / l, j = e % l;
            if (i > k && j >= i) g[i][j] -= g[k][i] * g[k][j];
        }
        __syncthreads();
    }
    // R^-1 (upper triangular) by back substitution, one column per thread,
    // with the diagonal's reciprocals taken once
    __shared__ double dinv[kMaxL];
    for (int i = tid; i < l; i += blockDim.x) dinv[i] = dead[i] ? 0.0 : 1.0 / g[i][i];
    __syncthreads();
    for (int j = tid; j < l; j += blockDim.x) {
        for (int i = 0; i < l; ++i) ri[i][j] = 0.0;
        if (!dead[j]) {
            ri[j][j] = dinv[j];
            for (int i = j - 1; i >= 0; --i) {
                if (dead[i]) continue;
                double s = 0.0;
                for (int m = i + 1; m <= j; ++m) s += g[i][m] * ri[m][j];
                ri[i][j] = -s * dinv[i];
            }
        }
    }
    __syncthreads();
    for (int e = tid; e < l * l; e += blockDim.x) minv[e] = static_cast<float>(ri[e / l][e % l]);
}

// One CTA: the symmetric eigenproblem of G by cyclic Jacobi in fp32 with the
// round-robin pair order (l/2 disjoint rotations per round) until the
// off-diagonal mass is below 1e-12 of the diagonal's (at most 40 sweeps);
// ur[i][m] = the eigenvector of the m-th largest eigenvalue, m < r.  Only
// the r leading eigenvectors are used, and they are set apart by the
// spectral gap, so fp32 (fp64 rotations are slow on GB300's few fp64 units)
// costs about 1e-6 of them.
__global__ void __launch_bounds__(256) jacobi_kernel(const double* __restrict__ G, int l, int r,
                                                     float* __restrict__ ur)
{
    __shared__ float A[kMaxL][kMaxL + 1];
    __shared__ float V[kMaxL][kMaxL + 1];
    __shared__ float cs[kMaxL / 2], sn[kMaxL / 2];
    __shared__ int pp[kMaxL / 2], qq[kMaxL / 2];
    __shared__ float red[2][256];
    __shared__ int idx[kMaxL];
    const int tid = threadIdx.x;
    for (int e = tid; e < kMaxL * kMaxL; e += blockDim.x) {
        const int i = e >> 6, j = e & 63;
        A[i][j] = (i < l && j < l) ? static_cast<float>(G[i * l + j]) : 0.0f;
        V[i][j] = i == j ? 1.0f : 0.0f;
    }
    __syncthreads();
    const int n = l + (l & 1);  // even number of players; index l is a dummy when l is odd
    for (int sweep = 0; sweep < 40; ++sweep) {
        float off = 0.0f, dia = 0.0f;
        for (int e = tid; e < l * l; e += blockDim.x) {
            const float v = A[e / l][e % l];
            if (e / l == e % l)
                dia += v * v;
            else
                off += v * v;
        }
        red[0][tid] = off;
        red[1][tid] = dia;
        __syncthreads();
        for (int s = 128; s > 0; s >>= 1) {
            if (tid < s) {
                red[0][tid] += red[0][tid + s];
                red[1][tid] += red[1][tid + s];
            }
            __syncthreads();
        }
        const bool done = !(red[0][0] > 1e-12f * red[1][0]);
        __syncthreads();
        if (done) break;
        for (int t = 0; t + 1 < n; ++t) {
            if (tid < n / 2) {
                const int a = tid == 0 ? 0 : 1 + (tid - 1 + t) % (n - 1);
                const int b = 1 + (n - 2 - tid + t) % (n - 1);
                const int p = a < b ? a : b, q = a < b ? b : a;
                float c = 1.0f, s = 0.0f;
                if (q < l) {
                    const float apq = A[p][q];
                    if (fabsf(apq) > 1e-30f) {
                        const float th = (A[q][q] - A[p][p]) / (2.0f * apq);
                        const float tt = (th >= 0.0f ? 1.0f : -1.0f) / (fabsf(th) + sqrtf(th * th + 1.0f));
                        c = 1.0f / sqrtf(tt * tt + 1.0f);
                        s = tt * c;
                    }
                }
                cs[tid] = c;
                sn[tid] = s;
                pp[tid] = p;
                qq[tid] = q;
            }
            __syncthreads();
            // A <- A P and V <- V P (columns p, q of every disjoint pair)
            for (int e = tid; e < (n / 2) * l; e += blockDim.x) {
                const int i = e / l, row = e % l;
                const int p = pp[i], q = qq[i];
                if (q >= l) continue;
                const float c = cs[i], s = sn[i];
                const float ap = A[row][p], aq = A[row][q];
                A[row][p] = c * ap - s * aq;
                A[row][q] = s * ap + c * aq;
                const float vp = V[row][p], vq = V[row][q];
                V[row][p] = c * vp - s * vq;
                V[row][q] = s * vp + c * vq;
            }
            __syncthreads();
            // A <- P^T A (rows p, q)
            for (int e = tid; e < (n / 2) * l; e += blockDim.x) {
                const int i = e / l, col = e % l;
                const int p = pp[i], q = qq[i];
                if (q >= l) continue;
                const float c = cs[i], s = sn[i];
                const float ap = A[p][col], aq = A[q][col];
                A[p][col] = c * ap - s * aq;
                A[q][col] = s * ap + c * aq;
            }
            __syncthreads();
        }
    }
    if (tid == 0) {
        for (int i = 0; i < l; ++i) idx[i] = i;
        for (int i = 0; i < l; ++i) {  // selection sort, largest eigenvalue first (ties: lower index)
            int best = i;
            for (int j = i + 1; j < l; ++j)
                if (A[idx[j]][idx[j]] > A[idx[best]][idx[best]]) best = j;
            const int tmp = idx[i];
            idx[i] = idx[best];
            idx[best] = tmp;
        }
    }
    __syncthreads();
    for (int e = tid; e < l * r; e += blockDim.x) ur[e] = V[e / r][idx[e % r]];
}

// dst[row][j] = sum_c src[row][c] * M[c][j]  (c < l, j < m); one row per
// thread, read whole before any write, so dst may be src when m == l.
__global__ void __launch_bounds__(256) apply_kernel(const float* src, int64_t n, int l, const float* __restrict__ M,
                                                    int m, float* dst)
{
    __shared__ float sm[kMaxL][kMaxL];
    for (int e = threadIdx.x; e < kMaxL * kMaxL; e += blockDim.x) {
        const int c = e >> 6, j = e & 63;
        sm[c][j] = (c < l && j < m) ? M[c * m + j] : 0.0f;
    }
    __syncthreads();
    const int64_t row = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (row >= n) return;
    float v[kMaxL];
#pragma unroll
    for (int c = 0; c < kMaxL; ++c) v[c] = c < l ? src[row * l + c] : 0.0f;
    for (int j = 0; j < m; ++j) {
        float s = 0.0f;
#pragma unroll
        for (int c = 0; c < kMaxL; ++c) s = fmaf(v[c], sm[c][j], s);
        dst[row * m + j] = s;
    }
}

// out[row][j] = W_base[row][j] + inv_k * sum_e L[e][row] Rt[e][j], e over the
// k * r factor columns (L [k][d_out][r], Rt [k][d_in][r]); 64 x 64 outputs per
// CTA, 4 x 4 per thread, factor columns in chunks of 32.
__global__ void __launch_bounds__(256) merge_kernel(const uint16_t* __restrict__ wb, int64_t d_out, int64_t d_in,
                                                    const float* __restrict__ L, const float* __restrict__ Rt, int k,
                                                    int r, float inv_k, void* __restrict__ out, int out_f32)
{
    __shared__ float sl[64][33];
    __shared__ float sr[64][33];
    const int tid = threadIdx.x;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 64, j0 = static_cast<int64_t>(blockIdx.x) * 64;
    const int tr = (tid >> 4) * 4, tc = (tid & 15) * 4;
    float acc[4][4] = {};
    const int K = k * r;
    for (int e0 = 0; e0 < K; e0 += 32) {
        for (int e = tid; e < 64 * 32; e += 256) {
            const int rr = e >> 5, ee = e & 31, f = e0 + ee;
            const int fi = f / (r > 0 ? r : 1), fc = f - fi * r;
            const int64_t row = r0 + rr, col = j0 + rr;
            sl[rr][ee] = (f < K && row < d_out) ? L[(static_cast<int64_t>(fi) * d_out + row) * r + fc] : 0.0f;
            sr[rr][ee] = (f < K && col < d_in) ? Rt[(static_cast<int64_t>(fi) * d_in + col) * r + fc] : 0.0f;
        }
        __syncthreads();
#pragma unroll 4
        for (int ee = 0; ee < 32; ++ee) {
            float a[4], b[4];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                a[x] = sl[tr + x][ee];
                b[x] = sr[tc + x][ee];
            }
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(a[x], b[y], acc[x][y]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        const int64_t row = r0 + tr + x;
        if (row >= d_out) continue;
#pragma unroll
        for (int y = 0; y < 4; ++y) {
            const int64_t col = j0 + tc + y;
            const float v = bf16_bits_to_float(wb[row * d_in + col]) + inv_k * acc[x][y];
            if (out_f32)
                static_cast<float*>(out)[row * d_in + col] = v;
            else
                static_cast<__nv_bfloat16*>(out)[row * d_in + col] = __float2bfloat16_rn(v);
        }
    }
}

size_t up256(size_t b) { return (b + 255) / 256 * 256; }

struct MonoSoupWs {
    size_t y, z, ypart, zpart, part, g, m, L, Rt, total;
};

MonoSoupWs ws_layout(int64_t d_out, int64_t d_in, int k, int r, int l)
{
    MonoSoupWs w{};
    size_t off = 256;  // error word area (unused by these kernels, kept for the common layout)
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += up256(bytes);
        return at;
    };
    w.y = take(static_cast<size_t>(d_out) * l * 4);
    w.z = take(static_cast<size_t>(d_in) * l * 4);
    w.ypart = take(static_cast<size_t>(kSlices) * d_out * l * 4);
    w.zpart = take(static_cast<size_t>(kSlices) * d_in * l * 4);
    w.part = take(static_cast<size_t>(kGramBlocks) * l * l * 8);
    w.g = take(static_cast<size_t>(l) * l * 8);
    w.m = take(static_cast<size_t>(kMaxL) * kMaxL * 4);
    w.L = take(static_cast<size_t>(k) * d_out * (r > 0 ? r : 1) * 4);
    w.Rt = take(static_cast<size_t>(k) * d_in * (r > 0 ? r : 1) * 4);
    w.total = off;
    return w;
}

unsigned blocks_for(int64_t n) { return static_cast<unsigned>((n + 255) / 256); }

}  // namespace

int monosoup_max_l() { return kMaxL; }

size_t monosoup_workspace_size(int64_t d_out, int64_t d_in, int k, int r, int l)
{
    return ws_layout(d_out, d_in, k, r, l).total;
}

cudaError_t launch_monosoup(const MonoSoupArgs& a, cudaStream_t st)
{
    static std::atomic<size_t> chol_set[kHostMaxDevices];
    const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(chol_inv_kernel), kSmallSmem, chol_set);
    if (e != cudaSuccess) return e;
    const MonoSoupWs lay = ws_layout(a.d_out, a.d_in, a.k, a.rank, a.l);
    char* w = static_cast<char*>(a.ws);
    float* Y = reinterpret_cast<float*>(w + lay.y);
    float* Z = reinterpret_cast<float*>(w + lay.z);
    float* Yp = reinterpret_cast<float*>(w + lay.ypart);
    float* Zp = reinterpret_cast<float*>(w + lay.zpart);
    double* part = reinterpret_cast<double*>(w + lay.part);
    double* G = reinterpret_cast<double*>(w + lay.g);
    float* M = reinterpret_cast<float*>(w + lay.m);
    float* L = reinterpret_cast<float*>(w + lay.L);
    float* Rt = reinterpret_cast<float*>(w + lay.Rt);
    const int l = a.l, r = a.rank;
    // the two products with Delta, each split in kSlices along its long
    // dimension and summed in slice order
    const int64_t ncol = a.d_in / 64, nrow = (a.d_out + 63) / 64;
    const int64_t cs = (ncol + kSlices - 1) / kSlices, rs = (nrow + kSlices - 1) / kSlices;
    const dim3 gsk(static_cast<unsigned>((a.d_out + 31) / 32), static_cast<unsigned>((ncol + cs - 1) / cs));
    const dim3 glf(static_cast<unsigned>(a.d_in / 32), static_cast<unsigned>((nrow + rs - 1) / rs));
    // tiles as wide as l needs: 32 columns (2 per thread) up to l = 32, else 64
    auto sketch = [&](const uint16_t* wi, const float* om) {  // Y = Delta om
        if (l <= 32)
            sketch_kernel<2><<<gsk, 256, 0, st>>>(wi, a.w_base, a.d_out, a.d_in, om, l, 64 * cs, Yp);
        else
            sketch_kernel<4><<<gsk, 256, 0, st>>>(wi, a.w_base, a.d_out, a.d_in, om, l, 64 * cs, Yp);
        sum_slices_kernel<<<blocks_for(a.d_out * l), 256, 0, st>>>(Yp, static_cast<int>(gsk.y), a.d_out * l, Y);
    };
    auto left = [&](const uint16_t* wi) {  // Z = Delta^T Y
        if (l <= 32)
            left_kernel<2><<<glf, 256, 0, st>>>(wi, a.w_base, a.d_out, a.d_in, Y, l, 64 * rs, Zp);
        else
            left_kernel<4><<<glf, 256, 0, st>>>(wi, a.w_base, a.d_out, a.d_in, Y, l, 64 * rs, Zp);
        sum_slices_kernel<<<blocks_for(a.d_in * l), 256, 0, st>>>(Zp, static_cast<int>(glf.y), a.d_in * l, Z);
    };
    auto gram = [&](const float* A, int64_t n) {  // G = A^T A
        gram_kernel<<<kGramBlocks, 256, 0, st>>>(A, n, l, part);
        gram_sum_kernel<<<blocks_for(static_cast<int64_t>(l) * l), 256, 0, st>>>(part, l, G);
    };
    // A <- A R^-1 (CholeskyQR), `passes` times: two (CholeskyQR2) for the Q
    // that B is projected on, one for the intermediate bases of the power
    // iterations, where only the spanned subspace matters
    auto orth = [&](float* A, int64_t n, int passes) {
        for (int pass = 0; pass < passes; ++pass) {
            gram(A, n);
            chol_inv_kernel<<<1, 256, kSmallSmem, st>>>(G, l, M);
            apply_kernel<<<blocks_for(n), 256, 0, st>>>(A, n, l, M, l, A);
        }
    };
    if (r > 0) {
        for (int i = 0; i < a.k; ++i) {
            const uint16_t* wi = a.w_ft[i];
            sketch(wi, a.omega);
            orth(Y, a.d_out, a.power_iters > 0 ? 1 : 2);
            for (int it = 0; it < a.power_iters; ++it) {
                left(wi);
                orth(Z, a.d_in, 1);
                sketch(wi, Z);
                orth(Y, a.d_out, it + 1 == a.power_iters ? 2 : 1);
            }
            left(wi);  // Z = B^T
            gram(Z, a.d_in);                                        // B B^T
            jacobi_kernel<<<1, 256, 0, st>>>(G, l, r, M);  // U_r [l][r]
            apply_kernel<<<blocks_for(a.d_out), 256, 0, st>>>(Y, a.d_out, l, M, r,
                                                              L + static_cast<size_t>(i) * a.d_out * r);
            apply_kernel<<<blocks_for(a.d_in), 256, 0, st>>>(Z, a.d_in, l, M, r,
                                                             Rt + static_cast<size_t>(i) * a.d_in * r);
        }
    }
    const dim3 grid(static_cast<unsigned>(a.d_in / 64), static_cast<unsigned>((a.d_out + 63) / 64));
    merge_kernel<<<grid, 256, 0, st>>>(a.w_base, a.d_out, a.d_in, L, Rt, r > 0 ? a.k : 0, r,
                                       1.0f / static_cast<float>(a.k), a.out, a.out_f32);
    return cudaGetLastError();
}

}  // namespace bd
