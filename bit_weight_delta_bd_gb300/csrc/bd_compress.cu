// BitDelta compression on sm_103a: Delta = W_ft - W_base, packed sign bits
// and alpha = mean|Delta| (section "Matematiksel temel", eqs. (1)-(3) of the
// BitDelta post; storage format of section "Altyapi ayrintilari").
//
// One warp owns one row and walks it in 256-column stripes: every lane loads
// 16 bytes (8 bf16) of W_base and of W_ft with streaming 128-bit loads, forms
// the 8 deltas in fp32 (the sign of a difference of two bf16 values is always
// exact), builds one byte of sign bits, and four neighbouring lanes OR their
// bytes into one 32-bit word with two shuffles.  |Delta| is summed in fp32
// over each lane's 8 values and then in fp64, so alpha (rounded to float32
// once) is accurate to ~1e-7 relative and independent of launch timing.
// The kernel is bound by HBM bandwidth: per element it reads 4 bytes and
// writes 1/8 byte.
#include "bd_device.cuh"
#include "bd_internal.h"

namespace bd {
namespace {

constexpr int kStripe = 256;  // columns per warp step (32 lanes x 8 bf16)
constexpr int kUnroll = 4;    // stripes in flight per lane (8 x 16-byte loads)

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Eight consecutive columns: returns their sign bits (bit k = column k,
// 1 <=> Delta >= 0, so sign(0) = +1) and adds sum |Delta| to `sum`.
__device__ __forceinline__ uint32_t delta8(const uint4 b, const uint4 f, float& sum)
{
    const uint32_t bw[4] = {b.x, b.y, b.z, b.w};
    const uint32_t fw[4] = {f.x, f.y, f.z, f.w};
    uint32_t byte = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float d0 = __fsub_rn(bf16_lo(fw[i]), bf16_lo(bw[i]));
        const float d1 = __fsub_rn(bf16_hi(fw[i]), bf16_hi(bw[i]));
        byte |= (d0 < 0.0f ? 0u : 1u) << (2 * i);
        byte |= (d1 < 0.0f ? 0u : 1u) << (2 * i + 1);
        sum = __fadd_rn(sum, fabsf(d0));
        sum = __fadd_rn(sum, fabsf(d1));
    }
    return byte;
}

__global__ void __launch_bounds__(32 * kCompressRowsPerCta)
    compress_kernel(const uint16_t* __restrict__ w_base, const uint16_t* __restrict__ w_ft, int64_t d_out,
                    int64_t d_in, int per_row, uint32_t* __restrict__ signs, float* __restrict__ alpha,
                    double* __restrict__ partials, uint32_t* err)
{
    __shared__ double warp_sum[kCompressRowsPerCta];
    grid_launch_dependents();  // a kernel launched after this one with programmatic dependent launch may start
    grid_dependency_wait();    // the previous kernel's results are visible
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kCompressRowsPerCta + warp;

    double acc = 0.0;
    if (row < d_out) {
        const uint16_t* pb = w_base + row * d_in;
        const uint16_t* pf = w_ft + row * d_in;
        uint32_t* ps = signs + row * (d_in / 32);
        const int64_t n_stripes = (d_in + kStripe - 1) / kStripe;
        for (int64_t s0 = 0; s0 < n_stripes; s0 += kUnroll) {
            uint4 vb[kUnroll], vf[kUnroll];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t col = (s0 + u) * kStripe + lane * 8;
                if (s0 + u < n_stripes && col < d_in && bd_in_range(kBkCompress, row * d_in + col, 8, d_out * d_in)) {
                    vb[u] = ld_stream_v4(pb + col);
                    vf[u] = ld_stream_v4(pf + col);
                } else {
                    vb[u] = make_uint4(0u, 0u, 0u, 0u);
                    vf[u] = vb[u];
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                const int64_t s = s0 + u;
                if (s >= n_stripes) break;  // warp-uniform
                const bool valid = (s * kStripe + lane * 8) < d_in;
                float part = 0.0f;
                const uint32_t byte = delta8(vb[u], vf[u], part);
                acc += static_cast<double>(part);  // zero for lanes past d_in
                // lanes 4w..4w+3 hold columns 32w..32w+31 of this stripe
                uint32_t word = byte << (8 * (lane & 3));
                word |= __shfl_xor_sync(0xffffffffu, word, 1);
                word |= __shfl_xor_sync(0xffffffffu, word, 2);
                const int64_t wi = s * (kStripe / 32) + (lane >> 2);
                if ((lane & 3) == 0 && valid && bd_in(kBkCompress, row * (d_in / 32) + wi, d_out * (d_in / 32)))
                    ps[wi] = word;
            }
        }
    }
    // Fixed butterfly: every lane ends with the same fp64 sum.
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);

    if (per_row) {
        if (lane == 0 && row < d_out) {
            if (!isfinite(acc)) raise_error(err, kErrNonFinite);
            if (bd_in(kBkCompress, row, d_out)) alpha[row] = static_cast<float>(acc / static_cast<double>(d_in));
        }
        return;
    }
    if (lane == 0) warp_sum[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        double total = 0.0;
        for (int w = 0; w < kCompressRowsPerCta; ++w) total += warp_sum[w];
        if (!isfinite(total)) raise_error(err, kErrNonFinite);
        if (bd_in(kBkCompress, blockIdx.x, (d_out + kCompressRowsPerCta - 1) / kCompressRowsPerCta))
            partials[blockIdx.x] = total;
    }
}

// Per-matrix alpha: one CTA sums the per-CTA partials in a fixed order.
__global__ void __launch_bounds__(1024)
    alpha_finalize_kernel(const double* __restrict__ partials, int64_t n_parts, double n_elems, float* alpha)
{
    __shared__ double sm[1024];
    grid_launch_dependents();
    grid_dependency_wait();
    double s = 0.0;
    for (int64_t i = threadIdx.x; i < n_parts; i += 1024)
        if (bd_in(kBkAlphaFinalize, i, n_parts)) s += partials[i];
    sm[threadIdx.x] = s;
    __syncthreads();
    for (int o = 512; o > 0; o >>= 1) {
        if (threadIdx.x < o) sm[threadIdx.x] += sm[threadIdx.x + o];
        __syncthreads();
    }
    if (threadIdx.x == 0) alpha[0] = static_cast<float>(sm[0] / n_elems);
}

__global__ void debug_reconstruct_kernel(const uint16_t* __restrict__ w_base, const uint32_t* __restrict__ signs,
                                         const float* __restrict__ alpha, int per_row, int64_t d_out, int64_t d_in,
                                         float* __restrict__ w_eff)
{
    const int64_t n = d_out * d_in;
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < n;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = e / d_in, c = e % d_in;
        if (!bd_in(kBkReconstruct, e, n) || !bd_in(kBkReconstruct, r * (d_in / 32) + c / 32, d_out * (d_in / 32)) ||
            !bd_in(kBkReconstruct, per_row ? r : 0, per_row ? d_out : 1))
            continue;
        const float w = __uint_as_float(static_cast<uint32_t>(w_base[e]) << 16);
        const uint32_t bit = (signs[r * (d_in / 32) + c / 32] >> (c % 32)) & 1u;
        const float a = per_row ? alpha[r] : alpha[0];
        w_eff[e] = __fadd_rn(w, bit ? a : -a);
    }
}

}  // namespace

cudaError_t launch_compress(const uint16_t* w_base, const uint16_t* w_ft, int64_t d_out, int64_t d_in, bool per_row,
                            uint32_t* signs, float* alpha, double* partials, uint32_t* err, cudaStream_t stream)
{
    const int64_t grid = (d_out + kCompressRowsPerCta - 1) / kCompressRowsPerCta;
    // programmatic dependent launches: each kernel's launch overlaps the end of the one before it
    cudaError_t e = cudaSuccess;
    launch_dep(e, compress_kernel, dim3(static_cast<unsigned>(grid)), dim3(32 * kCompressRowsPerCta), 0, stream, w_base,
               w_ft, d_out, d_in, per_row ? 1 : 0, signs, alpha, partials, err);
    if (e != cudaSuccess || per_row) return e;
    launch_dep(e, alpha_finalize_kernel, dim3(1), dim3(1024), 0, stream, static_cast<const double*>(partials), grid,
               static_cast<double>(d_out) * static_cast<double>(d_in), alpha);
    return e;
}

cudaError_t launch_debug_reconstruct(const uint16_t* w_base, const uint32_t* signs, const float* alpha, bool per_row,
                                     int64_t d_out, int64_t d_in, float* w_eff, cudaStream_t stream)
{
    const int64_t n = d_out * d_in;
    const int64_t blocks = (n + 255) / 256 < 65535 ? (n + 255) / 256 : 65535;
    debug_reconstruct_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(w_base, signs, alpha,
                                                                                 per_row ? 1 : 0, d_out, d_in, w_eff);
    return cudaGetLastError();
}

BD_BOUNDS_TAKE(bounds_take_compress)

}  // namespace bd
