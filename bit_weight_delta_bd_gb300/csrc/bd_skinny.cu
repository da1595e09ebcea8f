// Fused BitDelta linear for decode-sized token counts (T <= 64), one or many
// variants sharing one W_base (section "Sunum mimarisi" of the BitDelta post:
// the fused reconstruct+matmul kernel and the shared-read base weights under
// a per-request delta cache).
//
//   y[t][r] = sum_j x[t][j] * W_base[r][j]  +  alpha_v(t)[r] * sum_j x[t][j] * s_v(t)[r][j]
//
// which is exactly x . (W_base + alpha*s)^T with no rounding of W_eff: the
// base and the sign contraction are separate bf16 MMAs (s in {-1,+1} is exact
// in bf16) that share the x operand, accumulated in fp32.
//
// Work split.  A CTA owns 16 output rows (one m16 MMA tile) and KS warps;
// warp k reduces the k-th of KS equal slices of d_in (KS depends only on
// d_in, so a row's arithmetic never depends on d_out).  Each warp runs its
// own pipeline of `stages` shared-memory stages filled by bulk async copies
// (cp.async.bulk + mbarrier): a stage holds 16 rows x 128 columns of W_base
// (row pitch 272 B, so the fragment loads below are bank-conflict free) and,
// per active variant, 16 rows x 4 sign words.  x is read straight from L2.
//
// Fragments.  mma.m16n8k16 wants, per thread (g = lane/4, q = lane%4), A
// elements (row g / g+8, k = 2q,2q+1,2q+8,2q+9) and B elements (token g,
// same k).  Any permutation of k applied to both operands leaves the sum
// unchanged, so logical k {2q,2q+1,2q+8,2q+9} of MMA step m is mapped to
// physical columns 16q+4m+{0,1,2,3} of the 64-column half-chunk: every
// thread then reads 16 consecutive columns (two 16-byte loads) of its rows
// and of its token, and the 16 sign bits of those columns are one half-word.
// Bits become bf16 +-1 pairs with 2 integer ops per register.
//
// Multi-variant.  The CTA groups its tokens by variant (stable counting
// sort, key = vid+1, so base tokens come first) and walks 8-token tiles of
// that order.  The base MMA runs once per tile; for every variant present in
// the tile it expands that variant's bits once and runs the sign MMA with x
// masked to the tile's tokens of that variant.  W_base is read once per CTA
// whatever the number of variants; the sign bits of every active variant are
// read once.
#include "bd_device.cuh"

namespace bd {
namespace {

constexpr int kChunk = 128;                 // columns per pipeline stage
constexpr int kWPitch = 272;                // staged W row pitch (256 data + 16 pad)
constexpr int kWStageBytes = 16 * kWPitch;  // 4352
constexpr int kSignTileBytes = 16 * 16;     // 16 rows x 4 words
constexpr int kMaxStages = 4;
constexpr int kMaxWarps = 8;
constexpr int kMaxKeys = kMaxVariants + 1;

struct alignas(16) SkinnyShared {
    uint64_t mbar[kMaxWarps][kMaxStages];
    const uint32_t* sign_ptr[kSkinnyMaxTokens];  // per active slot
    const float* alpha_ptr[kSkinnyMaxTokens];
    int key[kSkinnyMaxTokens];       // key of token t (caller order)
    int perm[kSkinnyMaxTokens];      // sorted position -> token
    int keyp[kSkinnyMaxTokens];      // sorted position -> key
    int seg[kMaxKeys + 1];
    int slot_of_key[kMaxKeys];
    int tile_first[kSkinnyMaxTokens / 8];
    int tile_last[kSkinnyMaxTokens / 8];
    int n_act;
};

// 16 sign bits (bit b = column b) -> 8 registers of bf16 pairs (+1 / -1);
// register p holds columns 2p (low half) and 2p+1 (high half).
__device__ __forceinline__ void expand_signs(uint32_t h, uint32_t (&s)[8])
{
    const uint32_t z = (h | (h << 15)) & 0x55555555u;  // bit 2p -> 2p, bit 2p+1 -> 2p+16
#pragma unroll
    for (int p = 0; p < 8; ++p) s[p] = 0xBF80BF80u ^ ((z << (15 - 2 * p)) & 0x80008000u);
}

__device__ __forceinline__ void mma4(float (&acc)[4], const uint32_t (&r0)[8], const uint32_t (&r1)[8],
                                     const uint4 xa, const uint4 xb)
{
    mma_bf16_16816(acc, r0[0], r1[0], r0[1], r1[1], xa.x, xa.y);
    mma_bf16_16816(acc, r0[2], r1[2], r0[3], r1[3], xa.z, xa.w);
    mma_bf16_16816(acc, r0[4], r1[4], r0[5], r1[5], xb.x, xb.y);
    mma_bf16_16816(acc, r0[6], r1[6], r0[7], r1[7], xb.z, xb.w);
}

// Two CTAs per SM fit the register file only for the smaller token tiles.
template <int NT, bool MULTI>
constexpr int ctas_per_sm() { return (MULTI || NT >= 4) ? 1 : 2; }

template <int NT, bool MULTI>
__global__ void __launch_bounds__(32 * kMaxWarps, ctas_per_sm<NT, MULTI>())
    skinny_kernel(const __grid_constant__ SkinnyArgs a, int KS, int stages, int sign_slots)
{
    extern __shared__ __align__(128) uint8_t dyn_smem[];
    __shared__ SkinnyShared sh;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, q = lane & 3;
    const int T = static_cast<int>(a.T);
    const int64_t d_in = a.d_in;
    const int64_t row0 = static_cast<int64_t>(blockIdx.x) * 16;
    const int valid_rows = static_cast<int>(a.d_out - row0 < 16 ? a.d_out - row0 : 16);

    // ---------------------------------------------------------------- routing (per CTA)
    if (MULTI) {
        if (tid < kSkinnyMaxTokens) {
            int k = kMaxKeys;  // past T: never counted
            if (tid < T) {
                const int v = a.vid[tid];
                const bool ok = (v >= -1 && v < a.V);
                if (!ok && blockIdx.x == 0) raise_error(a.err, kErrBadVariant);
                k = ok ? v + 1 : 0;
            }
            sh.key[tid] = k;
        }
        __syncthreads();
        if (tid == 0) {
            int cnt[kMaxKeys];
            for (int k = 0; k <= a.V; ++k) cnt[k] = 0;
            for (int t = 0; t < T; ++t) ++cnt[sh.key[t]];
            sh.seg[0] = 0;
            int n_act = 0;
            for (int k = 0; k <= a.V; ++k) {
                sh.seg[k + 1] = sh.seg[k] + cnt[k];
                sh.slot_of_key[k] = -1;
                if (k >= 1 && cnt[k] > 0) {
                    sh.slot_of_key[k] = n_act;
                    sh.sign_ptr[n_act] = a.signs[k - 1];
                    sh.alpha_ptr[n_act] = a.alpha[k - 1];
                    ++n_act;
                }
            }
            sh.n_act = n_act;
        }
        __syncthreads();
        if (tid < T) {
            const int k = sh.key[tid];
            int rank = 0;
            for (int t = 0; t < tid; ++t) rank += (sh.key[t] == k);
            sh.perm[sh.seg[k] + rank] = tid;
            sh.keyp[sh.seg[k] + rank] = k;
        }
    } else {
        if (tid < T) {
            sh.perm[tid] = tid;
            sh.keyp[tid] = 1;
        }
        if (tid == 0) {
            sh.n_act = 1;
            sh.slot_of_key[0] = -1;
            sh.slot_of_key[1] = 0;
            sh.sign_ptr[0] = a.signs[0];
            sh.alpha_ptr[0] = a.alpha[0];
        }
    }
    if (lane == 0 && warp < KS)
        for (int s = 0; s < stages; ++s) mbar_init(&sh.mbar[warp][s], 1);
    __syncthreads();
    if (tid < NT) {
        const int p0 = 8 * tid;
        const int p1 = (8 * tid + 7 < T - 1) ? 8 * tid + 7 : T - 1;
        sh.tile_first[tid] = p0 < T ? sh.keyp[p0] : 1;
        sh.tile_last[tid] = p0 < T ? sh.keyp[p1] : 0;  // empty range past T
    }
    __syncthreads();

    // ---------------------------------------------------------------- per-warp K slice
    const int n_act = sh.n_act;
    const int stage_bytes = kWStageBytes + sign_slots * kSignTileBytes;
    const int nc = static_cast<int>(d_in / kChunk);
    const int c_begin = static_cast<int>(static_cast<int64_t>(warp) * nc / KS);
    const int c_end = static_cast<int>(static_cast<int64_t>(warp + 1) * nc / KS);
    const int n_chunks = c_end - c_begin;
    uint8_t* wsm = dyn_smem + static_cast<size_t>(warp) * stages * stage_bytes;
    const uint32_t tx_bytes = static_cast<uint32_t>(valid_rows) * (256u + 16u * n_act);
    const int64_t sign_row_words = d_in / 32;

    auto issue = [&](int c, int s) {
        uint8_t* st = wsm + s * stage_bytes;
        uint64_t* bar = &sh.mbar[warp][s];
        if (lane == 0) mbar_arrive_expect_tx(bar, tx_bytes);
        __syncwarp();
        if (lane < valid_rows)
            bulk_g2s(st + lane * kWPitch, a.w_base + (row0 + lane) * d_in + static_cast<int64_t>(c) * kChunk, 256,
                     bar);
        for (int idx = lane; idx < n_act * 16; idx += 32) {
            const int slot = idx >> 4, i = idx & 15;
            if (i < valid_rows)
                bulk_g2s(st + kWStageBytes + slot * kSignTileBytes + i * 16,
                         sh.sign_ptr[slot] + (row0 + i) * sign_row_words + c * 4, 16, bar);
        }
    };

    float accb[NT][4], accs[NT][4];
    int my_key[NT];
    const uint16_t* xrow[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
        for (int e = 0; e < 4; ++e) accb[j][e] = accs[j][e] = 0.0f;
        const int p = 8 * j + g;
        my_key[j] = p < T ? sh.keyp[p] : -1;
        xrow[j] = p < T ? a.x + static_cast<int64_t>(sh.perm[p]) * d_in : nullptr;
    }

    bool timed_out = false;
    int issued = 0;
    if (warp < KS) {
        const int pre = n_chunks < stages ? n_chunks : stages;
        for (int i = 0; i < pre; ++i) issue(c_begin + i, i);
        issued = pre;
        for (int i = 0; i < n_chunks; ++i) {
            const int s = i % stages;
            const uint32_t parity = static_cast<uint32_t>(i / stages) & 1u;
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&sh.mbar[warp][s], parity))) {
                timed_out = true;
                // drain what is still in flight before the smem is reused
                for (int k = i + 1; k < issued; ++k)
                    mbar_wait_bounded(&sh.mbar[warp][k % stages], static_cast<uint32_t>(k / stages) & 1u);
                break;
            }
            const uint8_t* st = wsm + s * stage_bytes;
            const int c = c_begin + i;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint4* w0 = reinterpret_cast<const uint4*>(st + g * kWPitch + h * 128 + q * 32);
                const uint4* w1 = reinterpret_cast<const uint4*>(st + (g + 8) * kWPitch + h * 128 + q * 32);
                uint32_t W0[8], W1[8];
                {
                    const uint4 u0 = w0[0], u1 = w0[1], v0 = w1[0], v1 = w1[1];
                    W0[0] = u0.x; W0[1] = u0.y; W0[2] = u0.z; W0[3] = u0.w;
                    W0[4] = u1.x; W0[5] = u1.y; W0[6] = u1.z; W0[7] = u1.w;
                    W1[0] = v0.x; W1[1] = v0.y; W1[2] = v0.z; W1[3] = v0.w;
                    W1[4] = v1.x; W1[5] = v1.y; W1[6] = v1.z; W1[7] = v1.w;
                }
                const int sign_word = 2 * h + (q >> 1);
                const uint32_t sign_shift = 16u * (q & 1);
                uint32_t S0[8], S1[8];
                int cur_slot = -1;
                if (!MULTI) {
                    const uint32_t* sb = reinterpret_cast<const uint32_t*>(st + kWStageBytes);
                    expand_signs((sb[g * 4 + sign_word] >> sign_shift) & 0xFFFFu, S0);
                    expand_signs((sb[(g + 8) * 4 + sign_word] >> sign_shift) & 0xFFFFu, S1);
                }
                const int64_t xcol = static_cast<int64_t>(c) * kChunk + h * 64 + q * 16;
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    uint4 xa = make_uint4(0u, 0u, 0u, 0u), xb = xa;
                    if (xrow[j] != nullptr) {
                        xa = ld_nc_v4(xrow[j] + xcol);
                        xb = ld_nc_v4(xrow[j] + xcol + 8);
                    }
                    mma4(accb[j], W0, W1, xa, xb);
                    if (!MULTI) {
                        mma4(accs[j], S0, S1, xa, xb);
                    } else {
                        const int kf = sh.tile_first[j] > 1 ? sh.tile_first[j] : 1;
                        const int kl = sh.tile_last[j];
                        for (int k = kf; k <= kl; ++k) {
                            const int slot = sh.slot_of_key[k];
                            if (slot < 0) continue;
                            if (slot != cur_slot) {
                                cur_slot = slot;
                                const uint32_t* sb =
                                    reinterpret_cast<const uint32_t*>(st + kWStageBytes + slot * kSignTileBytes);
                                expand_signs((sb[g * 4 + sign_word] >> sign_shift) & 0xFFFFu, S0);
                                expand_signs((sb[(g + 8) * 4 + sign_word] >> sign_shift) & 0xFFFFu, S1);
                            }
                            const bool mine = (my_key[j] == k);
                            const uint4 z = make_uint4(0u, 0u, 0u, 0u);
                            mma4(accs[j], S0, S1, mine ? xa : z, mine ? xb : z);
                        }
                    }
                }
            }
            __syncwarp();
            if (i + stages < n_chunks) {
                fence_proxy_async_smem();
                issue(c + stages, s);
                ++issued;
            }
        }
        if (timed_out && lane == 0) raise_error(a.err, kErrTimeout);
    }

    // ---------------------------------------------------------------- K-slice reduction
    constexpr int Tpad = NT * 8;
    __syncthreads();  // every warp has drained its pipeline: reuse the stage memory
    float* red_b = reinterpret_cast<float*>(dyn_smem);
    float* red_s = red_b + KS * 16 * Tpad;
    if (warp < KS) {
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const int p = 8 * j + 2 * q;
            float* rb0 = red_b + (warp * 16 + g) * Tpad + p;
            float* rb1 = red_b + (warp * 16 + g + 8) * Tpad + p;
            float* rs0 = red_s + (warp * 16 + g) * Tpad + p;
            float* rs1 = red_s + (warp * 16 + g + 8) * Tpad + p;
            rb0[0] = accb[j][0]; rb0[1] = accb[j][1]; rb1[0] = accb[j][2]; rb1[1] = accb[j][3];
            rs0[0] = accs[j][0]; rs0[1] = accs[j][1]; rs1[0] = accs[j][2]; rs1[1] = accs[j][3];
        }
    }
    __syncthreads();
    for (int o = tid; o < 16 * T; o += blockDim.x) {
        const int p = o >> 4, r = o & 15;
        if (r >= valid_rows) continue;
        float b = 0.0f, s = 0.0f;
        for (int k = 0; k < KS; ++k) {
            b += red_b[(k * 16 + r) * Tpad + p];
            s += red_s[(k * 16 + r) * Tpad + p];
        }
        const int key = sh.keyp[p];
        const int slot = key >= 1 ? sh.slot_of_key[key] : -1;
        const int64_t row = row0 + r;
        float y = b;
        if (slot >= 0) {
            const float al = sh.alpha_ptr[slot][a.per_row ? row : 0];
            y = fmaf(al, s, b);
        }
        const int64_t idx = static_cast<int64_t>(sh.perm[p]) * a.d_out + row;
        if (a.out_f32)
            static_cast<float*>(a.y)[idx] = y;
        else
            static_cast<__nv_bfloat16*>(a.y)[idx] = __float2bfloat16_rn(y);
    }
}

template <int NT, bool MULTI>
cudaError_t launch_nt(const SkinnyArgs& a, int KS, int stages, int sign_slots, size_t smem, cudaStream_t stream)
{
    auto kern = skinny_kernel<NT, MULTI>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>((a.d_out + 15) / 16);
    kern<<<grid, 32 * kMaxWarps, smem, stream>>>(a, KS, stages, sign_slots);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_skinny(const SkinnyArgs& a, int /*sm_count*/, cudaStream_t stream)
{
    const bool multi = a.vid != nullptr;
    const int nc = static_cast<int>(a.d_in / kChunk);
    const int T = static_cast<int>(a.T);
    const int nt = T <= 8 ? 1 : T <= 16 ? 2 : T <= 32 ? 4 : 8;
    int sign_slots = 1;
    if (multi) sign_slots = a.V < T ? a.V : T;
    const size_t stage_bytes = kWStageBytes + static_cast<size_t>(sign_slots) * kSignTileBytes;
    // Two CTAs per SM (<= ~110 KB each) where the registers allow it, else one
    // (<= ~200 KB).
    const size_t budget = (multi || nt >= 4) ? 200u * 1024u : 110u * 1024u;
    // K slices: up to 8, each warp needing at least two stages in the budget.
    // The count depends on d_in (and, for many variants, on the stage size),
    // never on d_out.
    int KS = nc < kMaxWarps ? nc : kMaxWarps;
    while (KS > 1 && static_cast<size_t>(KS) * 2 * stage_bytes > budget) --KS;
    int stages = kMaxStages;
    while (stages > 2 && static_cast<size_t>(KS) * stages * stage_bytes > budget) --stages;
    const size_t pipe = static_cast<size_t>(KS) * stages * stage_bytes;
    const size_t red = 2u * KS * 16u * (nt * 8u) * sizeof(float);
    const size_t smem = pipe > red ? pipe : red;
    if (smem > 227u * 1024u) return cudaErrorInvalidConfiguration;
    if (multi) {
        switch (nt) {
            case 1: return launch_nt<1, true>(a, KS, stages, sign_slots, smem, stream);
            case 2: return launch_nt<2, true>(a, KS, stages, sign_slots, smem, stream);
            case 4: return launch_nt<4, true>(a, KS, stages, sign_slots, smem, stream);
            default: return launch_nt<8, true>(a, KS, stages, sign_slots, smem, stream);
        }
    }
    switch (nt) {
        case 1: return launch_nt<1, false>(a, KS, stages, sign_slots, smem, stream);
        case 2: return launch_nt<2, false>(a, KS, stages, sign_slots, smem, stream);
        case 4: return launch_nt<4, false>(a, KS, stages, sign_slots, smem, stream);
        default: return launch_nt<8, false>(a, KS, stages, sign_slots, smem, stream);
    }
}

}  // namespace bd
