// Multi-variant fused BitDelta linear for decode-sized token groups (T <= 64)
// (section "Sunum mimarisi" of the BitDelta post: one W_base in device
// memory shared by every variant's 1-bit delta, a router that sends each
// request to its variant, and the fused reconstruct+matmul kernel).
//
//   y[t][r] = sum_j x[t][j] W_base[r][j]  +  alpha_v(t)[r] * sum_j x[t][j] s_v(t)[r][j]
//
// Work split.  A CTA owns 128 output rows (8 consumer warps of 16 rows) and
// one of CK equal slices of d_in; the CK CTAs of a thread-block cluster cover
// d_in and sum their partial results through distributed shared memory in
// rank order (CK depends on d_in only).  One producer thread streams stages
// through a two-slot shared-memory ring (TMA, full/empty mbarriers, all waits
// bounded).  The CTA runs its slice in phases:
//   base phase     x . W_base^T for every token of the group: W_base boxes
//                  [128 rows x 64 columns] and x boxes [8*NT tokens x 64],
//                  both with the 128-byte swizzle, mma.sync m16n8k16 bf16;
//   variant phases one per variant that has tokens: its sign words (boxes
//                  [128 rows x 4 words]) against its own tokens only, which
//                  the prepare pass has packed into zero-padded 8-token tiles
//                  (plain bulk copies).  No MMA carries another variant's
//                  token, so nothing is masked; each variant's bits are read
//                  and expanded once per CTA.
// W_base is read from device memory once per CTA for all variants.  At the end
// of a variant phase the warp adds alpha * (its sign sums) into the per-token
// accumulators of the base phase through a small per-warp shared buffer.
//
// Sign operand recoding (exact).  Expanding 16 sign bits into eight bf16 +-1
// pairs needs a shift and a mask per pair.  Here each operand element is
// v = a_c + b instead, with b the sign bit (1 for s = +1) and a_c a constant
// of the column residue c = j mod 4: the bit stays where it is and becomes
// mantissa bit 4, 5 or 6 of a bf16 whose exponent gives that bit the value
// exactly 1 (a = 8, 4, 2 for c = 0, 1, 2), or the sign bit of +-0.5
// (a = -0.5, c = 3).  A 32-bit sign word rotated by 0, 4, 8 and 12 bits puts
// every one of its bits on such a place, so each bf16 pair of the MMA operand
// is one (rotated word & mask) ^ constant.  With s = 2b - 1:
//   sum_j x_j s_j = 2 M - C,   M = sum_j x_j v_j,   C = sum_j x_j (2 a_j + 1),
// where C depends on the token only and is computed once by the prepare pass
// (fp64, rounded to fp32).  Every product x_j v_j is exact in fp32 (at most
// 12 significant bits); M is accumulated in fp32 like the plain form.  The
// x operand of the sign MMA is permuted inside every 32-column group to the
// order in which the rotated words deliver the bits; both operands use the
// same permutation of k, so the contraction is unchanged.
#include <cooperative_groups.h>

#include "bd_device.cuh"
#include "bd_tma.h"

namespace cg = cooperative_groups;

namespace bd {
namespace {

constexpr int kConsumers = 8;
constexpr int kRows = 16 * kConsumers;  // output rows per CTA
constexpr int kThreads = 32 * (kConsumers + 1);
constexpr int kStages = 2;
constexpr int kChunk = 128;           // d_in columns per chunk
constexpr int kHalfRowBytes = 128;    // 64 bf16 columns: one 128-byte swizzle atom
constexpr int kWHalf = kRows * kHalfRowBytes;  // 16 KB
constexpr int kSignChunk = kRows * 16;          // 4 sign words x 128 rows = 2 KB
constexpr int kPadTile = 8 * kChunk * 2;       // one 8-token tile of one chunk = 2 KB
constexpr int kMaxTok = kSkinnyMaxTokens;
constexpr int kMaxKeys = kMaxVariants + 1;
constexpr int kMaxGroup = 8;          // chunks per variant stage

// Recoding: kind k = column residue mod 4.  Bit positions lo (k) and hi (k+16)
// of the operand register, their mask, and the constant bf16 pair a_k (the
// sign-bit kind stores -0.5 and the XOR flips it to +0.5 when the bit is 1).
__host__ __device__ constexpr uint32_t recode_mask(int k)
{
    return k == 0 ? 0x00100010u : k == 1 ? 0x00200020u : k == 2 ? 0x00400040u : 0x80008000u;
}
__host__ __device__ constexpr uint32_t recode_const(int k)  // 8, 4, 2, -0.5 (bf16 pairs)
{
    return k == 0 ? 0x41004100u : k == 1 ? 0x40804080u : k == 2 ? 0x40004000u : 0xBF00BF00u;
}
__host__ __device__ constexpr int recode_lo_bit(int k) { return k == 0 ? 4 : k == 1 ? 5 : k == 2 ? 6 : 15; }
// 2 a_k + 1 for the per-token correction C.
__host__ __device__ constexpr double recode_corr(int k) { return k == 0 ? 17.0 : k == 1 ? 9.0 : k == 2 ? 5.0 : 0.0; }

struct MultiParams {
    CUtensorMap sign_map[kMaxVariants];  // [d_out][d_in/32] uint32, box 4 x 128 rows
    CUtensorMap w_map;                   // [d_out][d_in] bf16, box 64 x 128 rows, 128B swizzle
    CUtensorMap x_map;                   // sorted x [T][d_in] bf16, box 64 x 8*NT, 128B swizzle
    const uint8_t* xp;                   // padded, permuted tiles of the variant phases
    const float* corr;                   // C per sorted position
    const int32_t* vid;
    const float* alpha[kMaxVariants];
    void* y;
    uint32_t* err;
    int64_t T, d_out, d_in;
    int V, per_row, out_f32, CK;
};

// Result of the per-CTA router (identical in every CTA and in the prepare pass).
struct Routing {
    int key[kMaxTok];    // key of token t (caller order); key = vid + 1, 0 = base model
    int perm[kMaxTok];   // sorted position -> token
    int keyp[kMaxTok];   // sorted position -> key
    int seg[kMaxKeys + 1];
    int slot_of_key[kMaxKeys];
    int act[kMaxTok];    // slot -> variant id
    int len[kMaxTok];    // slot -> padded 8-token tiles of that variant
    int ptile[kMaxTok];  // slot -> first padded tile (over all slots)
    int n_act;
    int n_ptiles;
};

struct MultiShared {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    Routing rt;
    int grp[kMaxTok];    // slot -> chunks per variant stage
    volatile int abort;
    float flush[kConsumers][16 * 8];
};

// Stable counting sort of the T (<= 64) tokens by key = vid + 1 (ids outside
// [-1, V) become base tokens and are flagged by block 0 of a launch), then
// the active variants in key order and their padded tiles.  Uses threads
// 0..63 of the block and ends with __syncthreads.
__device__ void route_group(Routing& rt, const int32_t* vid, int T, int V, uint32_t* err, int tid)
{
    if (tid < kMaxTok) {
        int k = kMaxKeys;  // past T: never counted
        if (tid < T) {
            const int v = vid[tid];
            const bool ok = (v >= -1 && v < V);
            if (!ok && blockIdx.x == 0 && blockIdx.y == 0) raise_error(err, kErrBadVariant);
            k = ok ? v + 1 : 0;
        }
        rt.key[tid] = k;
    }
    __syncthreads();
    if (tid == 0) {
        int cnt[kMaxKeys];
        for (int k = 0; k <= V; ++k) cnt[k] = 0;
        for (int t = 0; t < T; ++t) ++cnt[rt.key[t]];
        rt.seg[0] = 0;
        int n_act = 0, pt = 0;
        for (int k = 0; k <= V; ++k) {
            rt.seg[k + 1] = rt.seg[k] + cnt[k];
            rt.slot_of_key[k] = -1;
            if (k >= 1 && cnt[k] > 0) {
                rt.slot_of_key[k] = n_act;
                rt.act[n_act] = k - 1;
                rt.len[n_act] = (cnt[k] + 7) / 8;
                rt.ptile[n_act] = pt;
                pt += rt.len[n_act];
                ++n_act;
            }
        }
        rt.n_act = n_act;
        rt.n_ptiles = pt;
    }
    __syncthreads();
    if (tid < T) {
        const int k = rt.key[tid];
        int r = 0;
        for (int t = 0; t < tid; ++t) r += (rt.key[t] == k);
        rt.perm[rt.seg[k] + r] = tid;
        rt.keyp[rt.seg[k] + r] = k;
    }
    __syncthreads();
}

// ---------------------------------------------------------------- prepare pass

// One block per sorted token position (blocks 0..T-1) and one per empty row
// of a padded tile (the rest).  Writes, for the CTA-level layout of the main
// kernel:
//   xs   [T][d_in]   x in sorted order (base phase);
//   xp   padded tiles: for slot a, chunk c, tile r (of len_a), a 2 KB block
//        at ((ptile_a * nc + c * len_a + r) * 2 KB) whose 16-byte piece
//        (i, g, q) at ((i * 8 + g) * 4 + q) * 16 holds token row g of the
//        tile, columns 32q + 8i .. 32q + 8i + 7 of the chunk in recoded order;
//   corr [T]         C = sum_j x_j (2 a_(j mod 4) + 1) per sorted position.
__global__ void __launch_bounds__(256) multi_prepare_kernel(const uint16_t* __restrict__ x,
                                                            const int32_t* __restrict__ vid, int T, int V,
                                                            int64_t d_in, uint16_t* __restrict__ xs,
                                                            uint8_t* __restrict__ xp, float* __restrict__ corr)
{
    __shared__ Routing rt;
    __shared__ double part[8];
    const int tid = threadIdx.x;
    route_group(rt, vid, T, V, nullptr, tid);
    const int nc = static_cast<int>(d_in / kChunk);
    int slot = -1, local = 0, pos = -1;
    if (static_cast<int>(blockIdx.x) < T) {
        pos = blockIdx.x;
        const int k = rt.keyp[pos];
        if (k >= 1) {
            slot = rt.slot_of_key[k];
            local = pos - rt.seg[k];
        }
    } else {
        int e = static_cast<int>(blockIdx.x) - T;
        for (int a = 0; a < rt.n_act && slot < 0; ++a) {
            const int n = rt.seg[rt.act[a] + 2] - rt.seg[rt.act[a] + 1];
            const int empties = 8 * rt.len[a] - n;
            if (e < empties) {
                slot = a;
                local = n + e;
            } else {
                e -= empties;
            }
        }
        if (slot < 0) return;  // more blocks than empty rows
    }
    const uint16_t* xrow = pos >= 0 ? x + static_cast<int64_t>(rt.perm[pos]) * d_in : nullptr;
    double c_sum = 0.0;
    for (int task = tid; task < nc * 4; task += blockDim.x) {
        const int c = task >> 2, q = task & 3;
        const int64_t col0 = static_cast<int64_t>(c) * kChunk + 32 * q;
        uint16_t v[32];
        if (xrow) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint4 w = ld_nc_v4(xrow + col0 + 8 * u);
                *reinterpret_cast<uint4*>(xs + static_cast<int64_t>(pos) * d_in + col0 + 8 * u) = w;
                v[8 * u + 0] = static_cast<uint16_t>(w.x); v[8 * u + 1] = static_cast<uint16_t>(w.x >> 16);
                v[8 * u + 2] = static_cast<uint16_t>(w.y); v[8 * u + 3] = static_cast<uint16_t>(w.y >> 16);
                v[8 * u + 4] = static_cast<uint16_t>(w.z); v[8 * u + 5] = static_cast<uint16_t>(w.z >> 16);
                v[8 * u + 6] = static_cast<uint16_t>(w.w); v[8 * u + 7] = static_cast<uint16_t>(w.w >> 16);
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                const __nv_bfloat16 b = __ushort_as_bfloat16(v[j]);
                c_sum += static_cast<double>(__bfloat162float(b)) * recode_corr(j & 3);
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0;  // padding row of a tile
        }
        if (slot >= 0) {
            const int r = local >> 3, g = local & 7;
            uint8_t* tile = xp + (static_cast<int64_t>(rt.ptile[slot]) * nc + static_cast<int64_t>(c) * rt.len[slot] + r) *
                                     kPadTile;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t o[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int lo = (recode_lo_bit(k) + 4 * i) & 31, hi = (recode_lo_bit(k) + 16 + 4 * i) & 31;
                    o[k] = static_cast<uint32_t>(v[lo]) | (static_cast<uint32_t>(v[hi]) << 16);
                }
                *reinterpret_cast<uint4*>(tile + ((i * 8 + g) * 4 + q) * 16) = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    }
    if (pos < 0) return;
    // fixed-order block reduction of C (deterministic)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c_sum += __shfl_xor_sync(0xffffffffu, c_sum, o);
    if ((tid & 31) == 0) part[tid >> 5] = c_sum;
    __syncthreads();
    if (tid == 0) {
        double s = 0.0;
        for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) s += part[w];
        corr[pos] = static_cast<float>(s);
    }
}

// ---------------------------------------------------------------- main kernel

__device__ __forceinline__ bool wait_or_abort(MultiShared& sh, uint64_t* bar, uint32_t parity, uint32_t* err)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (sh.abort) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            sh.abort = 1;
            raise_error(err, kErrTimeout);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void mma4(float (&acc)[4], const uint32_t (&r0)[8], const uint32_t (&r1)[8],
                                     const uint4 xa, const uint4 xb)
{
    mma_bf16_16816(acc, r0[0], r1[0], r0[1], r1[1], xa.x, xa.y);
    mma_bf16_16816(acc, r0[2], r1[2], r0[3], r1[3], xa.z, xa.w);
    mma_bf16_16816(acc, r0[4], r1[4], r0[5], r1[5], xb.x, xb.y);
    mma_bf16_16816(acc, r0[6], r1[6], r0[7], r1[7], xb.z, xb.w);
}

constexpr int base_stage_bytes(int nt) { return 2 * kWHalf + 2 * (8 * nt) * kHalfRowBytes; }

// Consumer side of one variant phase with L padded tiles: the sign MMAs over
// the CTA's d_in slice, then alpha * 2M added into the base accumulators.
// Returns false when the pipeline was aborted.  i_stage is the running stage
// counter shared with the producer's schedule.
template <int NT, int L>
__device__ __forceinline__ bool variant_phase(MultiShared& sh, const MultiParams& p, uint8_t* ring, int stage_bytes,
                                              int slot, int n_chunks, int& i_stage, float (&acc_b)[NT][4],
                                              int warp, int g, int q, int64_t row0)
{
    float acc[L][4];
#pragma unroll
    for (int r = 0; r < L; ++r)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[r][e] = 0.0f;
    const int rl0 = 16 * warp + g;
    const int grp = sh.grp[slot];
    bool ok = true;
    for (int c0 = 0; c0 < n_chunks; c0 += grp) {
        const int cnt = n_chunks - c0 < grp ? n_chunks - c0 : grp;
        const int s = i_stage % kStages;
        if (!__all_sync(0xffffffffu, wait_or_abort(sh, &sh.full[s], static_cast<uint32_t>(i_stage / kStages) & 1u,
                                                   p.err))) {
            ok = false;
            break;
        }
        const uint8_t* st = ring + static_cast<size_t>(s) * stage_bytes;
        const uint8_t* pads = st + cnt * kSignChunk;
        for (int cc = 0; cc < cnt; ++cc) {
            const uint32_t* sg = reinterpret_cast<const uint32_t*>(st + cc * kSignChunk);
            const uint32_t w0 = sg[rl0 * 4 + q], w1 = sg[(rl0 + 8) * 4 + q];
            const uint8_t* pc = pads + cc * L * kPadTile + ((g * 4 + q) << 4);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t u0 = __funnelshift_r(w0, w0, 4 * i), u1 = __funnelshift_r(w1, w1, 4 * i);
                uint32_t a0[4], a1[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    a0[k] = (u0 & recode_mask(k)) ^ recode_const(k);
                    a1[k] = (u1 & recode_mask(k)) ^ recode_const(k);
                }
#pragma unroll
                for (int r = 0; r < L; ++r) {
                    const uint4 xv = *reinterpret_cast<const uint4*>(pc + r * kPadTile + i * 512);
                    mma_bf16_16816(acc[r], a0[0], a1[0], a0[1], a1[1], xv.x, xv.y);
                    mma_bf16_16816(acc[r], a0[2], a1[2], a0[3], a1[3], xv.z, xv.w);
                }
            }
        }
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(&sh.empty[s]);
        ++i_stage;
    }
    if (!ok) return false;
    // alpha * 2M into the base accumulators of the variant's tokens
    const Routing& rt = sh.rt;
    const int v = rt.act[slot];
    const int seg0 = rt.seg[v + 1], n = rt.seg[v + 2] - seg0;
    const int64_t ra = row0 + rl0, rb = ra + 8;
    const float* al = p.alpha[v];
    const float a2a = ra < p.d_out ? 2.0f * al[p.per_row ? ra : 0] : 0.0f;
    const float a2b = rb < p.d_out ? 2.0f * al[p.per_row ? rb : 0] : 0.0f;
    float* fl = sh.flush[warp];
#pragma unroll
    for (int r = 0; r < L; ++r) {
        fl[g * 8 + 2 * q] = acc[r][0];
        fl[g * 8 + 2 * q + 1] = acc[r][1];
        fl[(g + 8) * 8 + 2 * q] = acc[r][2];
        fl[(g + 8) * 8 + 2 * q + 1] = acc[r][3];
        __syncwarp();
        const int lo = seg0 + 8 * r;
        const int hi = seg0 + (8 * r + 8 < n ? 8 * r + 8 : n);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            if (8 * j + 8 <= lo || 8 * j >= hi) continue;  // warp-uniform
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int d = 8 * j + 2 * q + e;
                if (d >= lo && d < hi) {
                    acc_b[j][e] = fmaf(a2a, fl[g * 8 + (d - lo)], acc_b[j][e]);
                    acc_b[j][2 + e] = fmaf(a2b, fl[(g + 8) * 8 + (d - lo)], acc_b[j][2 + e]);
                }
            }
        }
        __syncwarp();
    }
    return true;
}

template <int NT>
__device__ __forceinline__ bool run_variant(int len, MultiShared& sh, const MultiParams& p, uint8_t* ring,
                                            int stage_bytes, int slot, int n_chunks, int& i_stage,
                                            float (&acc_b)[NT][4], int warp, int g, int q, int64_t row0)
{
    switch (len) {
        case 1: return variant_phase<NT, 1>(sh, p, ring, stage_bytes, slot, n_chunks, i_stage, acc_b, warp, g, q, row0);
        case 2:
            if constexpr (NT >= 2)
                return variant_phase<NT, 2>(sh, p, ring, stage_bytes, slot, n_chunks, i_stage, acc_b, warp, g, q, row0);
            break;
        case 3:
            if constexpr (NT >= 4)
                return variant_phase<NT, 3>(sh, p, ring, stage_bytes, slot, n_chunks, i_stage, acc_b, warp, g, q, row0);
            break;
        case 4:
            if constexpr (NT >= 4)
                return variant_phase<NT, 4>(sh, p, ring, stage_bytes, slot, n_chunks, i_stage, acc_b, warp, g, q, row0);
            break;
        case 5:
            if constexpr (NT >= 8)
                return variant_phase<NT, 5>(sh, p, ring, stage_bytes, slot, n_chunks, i_stage, acc_b, warp, g, q, row0);
            break;
        case 6:
            if constexpr (NT >= 8)
                return variant_phase<NT, 6>(sh, p, ring, stage_bytes, slot, n_chunks, i_stage, acc_b, warp, g, q, row0);
            break;
        case 7:
            if constexpr (NT >= 8)
                return variant_phase<NT, 7>(sh, p, ring, stage_bytes, slot, n_chunks, i_stage, acc_b, warp, g, q, row0);
            break;
        case 8:
            if constexpr (NT >= 8)
                return variant_phase<NT, 8>(sh, p, ring, stage_bytes, slot, n_chunks, i_stage, acc_b, warp, g, q, row0);
            break;
        default: break;
    }
    // unreachable: a variant never holds more padded tiles than the group has token tiles
    sh.abort = 1;
    raise_error(p.err, kErrTimeout);
    return false;
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 2) multi_kernel(const __grid_constant__ MultiParams p)
{
    constexpr int Tpad = 8 * NT;
    constexpr int kXHalf = Tpad * kHalfRowBytes;
    constexpr int kStageBytes = (base_stage_bytes(NT) + 1023) & ~1023;

    extern __shared__ uint8_t dyn_raw[];
    __shared__ MultiShared sh;
    uint8_t* ring = dyn_raw + ((1024u - (smem_u32(dyn_raw) & 1023u)) & 1023u);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, q = lane & 3;
    const int T = static_cast<int>(p.T);
    const int CK = p.CK;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int64_t row0 = static_cast<int64_t>(blockIdx.x / CK) * kRows;
    const int valid_rows = static_cast<int>(p.d_out - row0 < kRows ? p.d_out - row0 : kRows);

    route_group(sh.rt, p.vid, T, p.V, p.err, tid);
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], kConsumers);
        }
        sh.abort = 0;
        fence_mbarrier_init();
    }
    if (tid < sh.rt.n_act) {
        // chunks per variant stage: as many as fit one ring slot (at most 8)
        const int per_chunk = kSignChunk + sh.rt.len[tid] * kPadTile;
        int grp = kMaxGroup;
        while (grp > 1 && grp * per_chunk > kStageBytes) grp >>= 1;
        sh.grp[tid] = grp;
    }
    __syncthreads();

    const int n_act = sh.rt.n_act;
    const int nc = static_cast<int>(p.d_in / kChunk);
    const int c_begin = static_cast<int>(static_cast<int64_t>(rank) * nc / CK);
    const int c_end = static_cast<int>(static_cast<int64_t>(rank + 1) * nc / CK);
    const int n_chunks = c_end - c_begin;

    float acc_b[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc_b[j][e] = 0.0f;

    if (warp == kConsumers) {
        // ------------------------------------------------------------ producer warp
        int i = 0;
        bool ok = true;
        auto acquire = [&](int& s) -> bool {
            s = i % kStages;
            if (i >= kStages &&
                !__all_sync(0xffffffffu, wait_or_abort(sh, &sh.empty[s], static_cast<uint32_t>(i / kStages - 1) & 1u,
                                                       p.err)))
                return false;
            return true;
        };
        for (int c = 0; c < n_chunks && ok; ++c) {
            int s;
            if (!(ok = acquire(s))) break;
            uint8_t* st = ring + static_cast<size_t>(s) * kStageBytes;
            const int col = (c_begin + c) * kChunk;
            if (lane == 0) {
                mbar_arrive_expect_tx(&sh.full[s], static_cast<uint32_t>(2 * kWHalf + 2 * kXHalf));
                tma_load_2d(st, &p.w_map, col, static_cast<int>(row0), &sh.full[s]);
                tma_load_2d(st + kWHalf, &p.w_map, col + 64, static_cast<int>(row0), &sh.full[s]);
                tma_load_2d(st + 2 * kWHalf, &p.x_map, col, 0, &sh.full[s]);
                tma_load_2d(st + 2 * kWHalf + kXHalf, &p.x_map, col + 64, 0, &sh.full[s]);
            }
            __syncwarp();
            ++i;
        }
        for (int a = 0; a < n_act && ok; ++a) {
            const int v = sh.rt.act[a], len = sh.rt.len[a], grp = sh.grp[a];
            const uint8_t* src = p.xp + static_cast<int64_t>(sh.rt.ptile[a]) * nc * kPadTile;
            for (int c0 = 0; c0 < n_chunks; c0 += grp) {
                const int cnt = n_chunks - c0 < grp ? n_chunks - c0 : grp;
                int s;
                if (!(ok = acquire(s))) break;
                uint8_t* st = ring + static_cast<size_t>(s) * kStageBytes;
                if (lane == 0) {
                    const uint32_t pad_bytes = static_cast<uint32_t>(cnt * len * kPadTile);
                    mbar_arrive_expect_tx(&sh.full[s], static_cast<uint32_t>(cnt * kSignChunk) + pad_bytes);
                    for (int cc = 0; cc < cnt; ++cc)
                        tma_load_2d(st + cc * kSignChunk, &p.sign_map[v], (c_begin + c0 + cc) * 4,
                                    static_cast<int>(row0), &sh.full[s]);
                    bulk_g2s(st + cnt * kSignChunk, src + static_cast<int64_t>(c_begin + c0) * len * kPadTile,
                             pad_bytes, &sh.full[s]);
                }
                __syncwarp();
                ++i;
            }
        }
        // every issued stage must have landed before the CTA reuses the memory
        for (int k = (i > kStages ? i - kStages : 0); k < i; ++k) {
            const int s = k % kStages;
            const uint32_t par = static_cast<uint32_t>(k / kStages) & 1u;
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(&sh.full[s], par) && global_timer_ns() - t0 < kWaitLimitNs) {
            }
        }
    } else {
        // ------------------------------------------------------------ consumer warps
        const int rl0 = 16 * warp + g;  // local rows rl0 and rl0 + 8 (both = g mod 8)
        const int c0 = ((2 * q) ^ g) << 4, c1 = ((2 * q + 1) ^ g) << 4;  // swizzled chunk offsets
        int i = 0;
        bool ok = true;
        for (int c = 0; c < n_chunks; ++c) {
            const int s = i % kStages;
            if (!__all_sync(0xffffffffu,
                            wait_or_abort(sh, &sh.full[s], static_cast<uint32_t>(i / kStages) & 1u, p.err))) {
                ok = false;
                break;
            }
            const uint8_t* st = ring + static_cast<size_t>(s) * kStageBytes;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint8_t* wst = st + h * kWHalf;
                const uint8_t* xst = st + 2 * kWHalf + h * kXHalf;
                uint32_t W0[8], W1[8];
                {
                    const uint8_t* r0p = wst + rl0 * kHalfRowBytes;
                    const uint8_t* r1p = wst + (rl0 + 8) * kHalfRowBytes;
                    const uint4 u0 = *reinterpret_cast<const uint4*>(r0p + c0);
                    const uint4 u1 = *reinterpret_cast<const uint4*>(r0p + c1);
                    const uint4 v0 = *reinterpret_cast<const uint4*>(r1p + c0);
                    const uint4 v1 = *reinterpret_cast<const uint4*>(r1p + c1);
                    W0[0] = u0.x; W0[1] = u0.y; W0[2] = u0.z; W0[3] = u0.w;
                    W0[4] = u1.x; W0[5] = u1.y; W0[6] = u1.z; W0[7] = u1.w;
                    W1[0] = v0.x; W1[1] = v0.y; W1[2] = v0.z; W1[3] = v0.w;
                    W1[4] = v1.x; W1[5] = v1.y; W1[6] = v1.z; W1[7] = v1.w;
                }
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const uint8_t* xr = xst + (8 * j + g) * kHalfRowBytes;
                    mma4(acc_b[j], W0, W1, *reinterpret_cast<const uint4*>(xr + c0),
                         *reinterpret_cast<const uint4*>(xr + c1));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.empty[s]);
            ++i;
        }
        for (int a = 0; a < n_act && ok; ++a)
            ok = run_variant<NT>(sh.rt.len[a], sh, p, ring, kStageBytes, a, n_chunks, i, acc_b, warp, g, q, row0);
    }

    // ---------------------------------------------------------------- cluster K reduction
    __syncthreads();  // pipeline drained: the ring becomes the reduction buffer
    float* red = reinterpret_cast<float*>(ring);
    if (warp < kConsumers) {
        const int r0 = 16 * warp + g;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const int pos = 8 * j + 2 * q;
            red[r0 * Tpad + pos] = acc_b[j][0];
            red[r0 * Tpad + pos + 1] = acc_b[j][1];
            red[(r0 + 8) * Tpad + pos] = acc_b[j][2];
            red[(r0 + 8) * Tpad + pos + 1] = acc_b[j][3];
        }
    }
    cluster.sync();
    const Routing& rt = sh.rt;
    const int r_lo = rank * kRows / CK, r_hi = (rank + 1) * kRows / CK;
    const int nr = r_hi - r_lo;
    for (int o = tid; o < nr * T; o += kThreads) {
        const int pos = o / nr, r = r_lo + o % nr;
        if (r >= valid_rows) continue;
        float y = 0.0f;
        for (int k = 0; k < CK; ++k) y += cluster.map_shared_rank(red, k)[r * Tpad + pos];
        const int key = rt.keyp[pos];
        const int64_t row = row0 + r;
        if (key >= 1) y = fmaf(-p.alpha[key - 1][p.per_row ? row : 0], p.corr[pos], y);
        const int64_t idx = static_cast<int64_t>(rt.perm[pos]) * p.d_out + row;
        if (p.out_f32)
            static_cast<float*>(p.y)[idx] = y;
        else
            static_cast<__nv_bfloat16*>(p.y)[idx] = __float2bfloat16_rn(y);
    }
    cluster.sync();  // peers may still read this CTA's partials until here
}

template <int NT>
cudaError_t launch_nt(const MultiParams& prm, size_t smem, unsigned grid, cudaStream_t stream)
{
    auto kern = multi_kernel<NT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(prm.CK);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, prm);
}

int tiles_for(int T) { return T <= 8 ? 1 : T <= 16 ? 2 : T <= 32 ? 4 : 8; }

}  // namespace

int multi_max_ptiles(int T, int V)
{
    const int t = T < kMaxTok ? T : kMaxTok;
    const int a = t < V ? t : V;
    return (t + 7 * a) / 8;
}

cudaError_t launch_multi(const MultiArgs& a, cudaStream_t stream)
{
    const int T = static_cast<int>(a.T);
    if (T < 1 || T > kMaxTok || a.V < 1 || a.V > kMaxVariants) return cudaErrorInvalidValue;
    if (!a.x_sorted || !a.xp || !a.corr) return cudaErrorInvalidValue;
    const int nt = tiles_for(T);
    static thread_local MultiParams prm;  // ~9 KB: kept off the stack
    prm.xp = a.xp;
    prm.corr = a.corr;
    prm.vid = a.vid;
    prm.y = a.y;
    prm.err = a.err;
    prm.T = a.T;
    prm.d_out = a.d_out;
    prm.d_in = a.d_in;
    prm.V = a.V;
    prm.per_row = a.per_row;
    prm.out_f32 = a.out_f32;
    for (int v = 0; v < a.V; ++v) {
        prm.alpha[v] = a.alpha[v];
        if (!encode_tma_2d(&prm.sign_map[v], CU_TENSOR_MAP_DATA_TYPE_UINT32, a.signs[v],
                           static_cast<uint64_t>(a.d_in / 32), static_cast<uint64_t>(a.d_out),
                           static_cast<uint64_t>(a.d_in / 8), 4, static_cast<uint32_t>(kRows),
                           CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    if (!encode_tma_2d(&prm.w_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.w_base, static_cast<uint64_t>(a.d_in),
                       static_cast<uint64_t>(a.d_out), static_cast<uint64_t>(a.d_in) * 2, 64,
                       static_cast<uint32_t>(kRows), CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tma_2d(&prm.x_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x_sorted, static_cast<uint64_t>(a.d_in),
                       static_cast<uint64_t>(a.T), static_cast<uint64_t>(a.d_in) * 2, 64,
                       static_cast<uint32_t>(8 * nt), CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    // K slices per cluster: a function of d_in only (one per 2048 columns, at most 4)
    const int nc = static_cast<int>(a.d_in / kChunk);
    int ck = nc / 16;
    ck = ck < 1 ? 1 : ck > 4 ? 4 : ck;
    prm.CK = ck;
    const size_t stage = static_cast<size_t>((base_stage_bytes(nt) + 1023) & ~1023);
    const size_t red = static_cast<size_t>(kRows) * (8 * nt) * sizeof(float);
    size_t smem = kStages * stage;
    smem = (smem > red ? smem : red) + 1024;

    const int prep_blocks = T + 7 * (T < a.V ? T : a.V);
    multi_prepare_kernel<<<prep_blocks, 256, 0, stream>>>(a.x, a.vid, T, a.V, a.d_in, a.x_sorted, a.xp, a.corr);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>((a.d_out + kRows - 1) / kRows * ck);
    switch (nt) {
        case 1: return launch_nt<1>(prm, smem, grid, stream);
        case 2: return launch_nt<2>(prm, smem, grid, stream);
        case 4: return launch_nt<4>(prm, smem, grid, stream);
        default: return launch_nt<8>(prm, smem, grid, stream);
    }
}

}  // namespace bd
