// Materialised variant weights (the reading of the BitDelta post's "Sunum
// mimarisi" section in which the effective weights are built once and a
// standard matmul follows; the fused path never does this):
//   W_eff[r][j] = RN_bf16(W_base[r][j] + alpha_r * s_rj)
// rounded once from the exact sum.  Rounding the fp32 sum to bf16 (nearest,
// ties to even) is already the correct rounding of the exact sum except when
// the fp32 sum is itself a bf16 midpoint; only then is the addition's exact
// rounding error formed (Knuth's TwoSum) and its sign decides.  Group g of
// 8 weights in a row takes its 8 sign bits from byte g of the row's words
// (bit b of word w is column 32w + b, little-endian bytes).
#include "bd_device.cuh"

namespace bd {
namespace {

__device__ __forceinline__ uint32_t add_round_bf16(float w, float d)
{
    const float s = w + d;
    const uint32_t b = __float_as_uint(s);
    if ((b & 0xFFFFu) == 0x8000u) {
        // s is a bf16 midpoint (rare): the exact sum lies beyond it on the
        // side of the addition's rounding error, if there is one
        const float bb = s - w;
        const float e = (w - (s - bb)) + (d - bb);  // s + e == w + d exactly
        if (e != 0.0f) return (b >> 16) + ((e > 0.0f) == (s > 0.0f) ? 1u : 0u);
    }
    return (b + 0x7FFFu + ((b >> 16) & 1u)) >> 16;  // nearest, ties to even
}

// 8 weights of one row: W_base bits in u, sign bits in the low byte of bits.
// The fp32 sums are rounded to bf16 pairs by the conversion unless one of
// them, in any lane of the warp, is a bf16 midpoint; then every lane takes
// the exact path.
__device__ __forceinline__ uint4 materialize8(uint4 u, uint32_t bits, uint32_t ab)
{
    const uint32_t in[4] = {u.x, u.y, u.z, u.w};
    const uint32_t nb = ~bits;
    float w[8], d[8], s[8];
    uint32_t mid = 0;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        w[2 * h] = __uint_as_float(in[h] << 16);
        w[2 * h + 1] = __uint_as_float(in[h] & 0xFFFF0000u);
        d[2 * h] = __uint_as_float(ab ^ ((nb << (31 - 2 * h)) & 0x80000000u));
        d[2 * h + 1] = __uint_as_float(ab ^ ((nb << (30 - 2 * h)) & 0x80000000u));
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        s[k] = __fadd_rn(w[k], d[k]);
        mid |= (__float_as_uint(s[k]) & 0xFFFFu) == 0x8000u ? 1u : 0u;
    }
    uint32_t o[4];
    if (__any_sync(0xffffffffu, mid)) {
#pragma unroll
        for (int h = 0; h < 4; ++h)
            o[h] = (add_round_bf16(w[2 * h], d[2 * h]) & 0xFFFFu) | (add_round_bf16(w[2 * h + 1], d[2 * h + 1]) << 16);
    } else {
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const __nv_bfloat162 r = __floats2bfloat162_rn(s[2 * h], s[2 * h + 1]);
            o[h] = *reinterpret_cast<const uint32_t*>(&r);
        }
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Blocks stride over rows; in a row, thread t handles groups of 8 weights
// t, t + 256, ... so that every warp-wide 16-byte load and store covers 512
// contiguous bytes; four groups are loaded before any is written.
__global__ void __launch_bounds__(256) materialize_kernel(const uint16_t* __restrict__ w,
                                                          const uint32_t* __restrict__ signs,
                                                          const float* __restrict__ alpha, int per_row,
                                                          int64_t d_out, int64_t d_in, uint16_t* __restrict__ out)
{
    const int64_t gpr = d_in / 8;  // groups of 8 weights per row (a multiple of 16)
    for (int64_t r = blockIdx.x; r < d_out; r += gridDim.x) {
        if (!bd_in(kBkMaterialize, per_row ? r : 0, per_row ? d_out : 1)) continue;
        const uint32_t ab = __float_as_uint(alpha[per_row ? r : 0]);
        const uint16_t* wr = w + r * d_in;
        const uint8_t* sr = reinterpret_cast<const uint8_t*>(signs + r * (d_in / 32));  // byte g: bits of group g
        uint16_t* orow = out + r * d_in;
        int64_t g = threadIdx.x;
        const int64_t nw = d_out * d_in, nb = d_out * (d_in / 8);  // weights, sign bytes
        for (; g + 3 * 256 < gpr; g += 4 * 256) {
            if (!bd_in_range(kBkMaterialize, r * d_in + 8 * g, 8 * (3 * 256 + 1), nw) ||
                !bd_in_range(kBkMaterialize, r * (d_in / 8) + g, 3 * 256 + 1, nb))
                continue;
            uint4 u[4];
            uint32_t bits[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                u[k] = ld_nc_v4(wr + 8 * (g + 256 * k));
                bits[k] = __ldg(sr + g + 256 * k);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k)
                *reinterpret_cast<uint4*>(orow + 8 * (g + 256 * k)) = materialize8(u[k], bits[k], ab);
        }
        for (; g < gpr; g += 256)
            if (bd_in_range(kBkMaterialize, r * d_in + 8 * g, 8, nw) && bd_in(kBkMaterialize, r * (d_in / 8) + g, nb))
                *reinterpret_cast<uint4*>(orow + 8 * g) = materialize8(ld_nc_v4(wr + 8 * g), __ldg(sr + g), ab);
    }
}

}  // namespace

cudaError_t launch_materialize(const uint16_t* w_base, const uint32_t* signs, const float* alpha, int per_row,
                               int64_t d_out, int64_t d_in, uint16_t* w_eff, int sm_count, cudaStream_t stream)
{
    if (d_out == 0 || d_in == 0) return cudaSuccess;
    const int64_t cap = static_cast<int64_t>(sm_count > 0 ? sm_count : 1) * 8;  // 8 blocks of 256 per SM
    const unsigned grid = static_cast<unsigned>(d_out < cap ? d_out : cap);
    materialize_kernel<<<grid, 256, 0, stream>>>(w_base, signs, alpha, per_row, d_out, d_in, w_eff);
    return cudaGetLastError();
}

BD_BOUNDS_TAKE(bounds_take_materialize)

}  // namespace bd
