// Multi-variant fused BitDelta linear for decode-sized token groups (T <= 64)
// (section "Sunum mimarisi" of the BitDelta post: one W_base in device
// memory shared by every variant's 1-bit delta, a router that sends each
// request to its variant, and the fused reconstruct+matmul kernel).
//
//   y[t][r] = sum_j x[t][j] W_base[r][j]  +  alpha_v(t)[r] * sum_j x[t][j] s_v(t)[r][j]
//
// Two launches per group of tokens:
//   multi_prepare_kernel  routes the tokens (stable counting sort by vid + 1)
//                         and writes each variant's tokens into zero-padded
//                         8-token tiles in the order and scaling of the
//                         recoded sign operand (below), plus per-token
//                         partial corrections C;
//   multi_kernel          one CTA per 128 output rows and one of CK slices of
//                         d_in (a thread-block cluster of CK CTAs covers d_in;
//                         CK depends on d_in only), three roles running
//                         concurrently:
//     warp 9   base phase: x . W_base^T for every token on the tensor cores
//              (W_base [128 x 64] and x [Npad x 64] TMA boxes, tcgen05.mma
//              M = 128, N = Npad, K = 16, fp32 accumulator in tensor memory);
//     warp 8   streams the variant phases: for each active variant, its sign
//              words (TMA boxes [128 rows x 4 words]) and its padded x tiles;
//     warps 0-7 run the variant phases: mma.sync m16n8k16 of each variant's
//              recoded sign operand against its own tokens only (no masking),
//              and store alpha * 2M per token into a shared per-token buffer.
//   The epilogue adds the tensor-memory base sums, sums the cluster's slices
//   (every CTA stores its partial sums into the owning peer's receive slots,
//   then each owner adds its slots in rank order) and writes y = base +
//   alpha * (2M - C) in the caller's token order.
// W_base is read from device memory once per CTA for all variants; each
// active variant's bits once.
//
// Sign operand recoding (exact).  Expanding 16 sign bits into eight bf16 +-1
// pairs needs a shift and a mask per pair.  Here the sign contraction runs on
// operand elements v = a_c + b instead, with b the sign bit (1 for s = +1) and
// a_c a constant of the column residue c = j mod 4 (a = 8, 4, 2, -0.5).  The
// bit is never moved: each bf16 pair of the operand is
// (rotated sign word & mask_c) ^ const, a -0.5 whose mantissa bit 4, 5 or 6
// (c = 0, 1, 2) or sign bit (c = 3) is the sign bit, and the x operand is
// pre-scaled by -16, -8, -4 or 1 so that each product equals x_j (a_c + b_j)
// exactly.  A 32-bit sign word rotated by 0, 4, 8 and 12 bits puts every one
// of its bits on such a place.  With s = 2b - 1:
//   sum_j x_j s_j = 2 M - C,   M = sum_j x_j v_j,   C = sum_j x_j (2 a_j + 1),
// where C depends on the token only (computed once by the prepare pass, fp32
// partial sums in a fixed order).  Every product is exact in fp32 (at most 12
// significant bits); M is accumulated in fp32 like the plain form.  The x
// operand of the sign MMA is also permuted inside every 32-column group to
// the order in which the rotated words deliver the bits; both operands use
// the same permutation of k, so the contraction is unchanged.
#include <cooperative_groups.h>

#include "bd_device.cuh"
#include "bd_tcgen05.cuh"
#include "bd_tma.h"

namespace cg = cooperative_groups;

namespace bd {
namespace {

constexpr int kConsumers = 8;                 // warps 0..7: variant phases, then the epilogue
constexpr int kProducerWarp = kConsumers;     // warp 8: TMA of the variant phases
constexpr int kBaseWarp = kConsumers + 1;     // warp 9: tensor memory, base-phase TMA and tcgen05 MMAs
constexpr int kRows = 16 * kConsumers;        // 128 output rows per CTA = tensor-memory lanes
constexpr int kThreads = 32 * (kConsumers + 2);
constexpr int kChunk = 128;                   // d_in columns per chunk
constexpr int kHalfRowBytes = 128;            // 64 bf16 columns: one 128-byte swizzle atom
constexpr int kWTile = kRows * kHalfRowBytes; // W_base box [128 rows x 64 columns] = 16 KB
constexpr int kBaseStages = 2;
constexpr int kVarStages = 3;
constexpr int kVarSlot = 20 * 1024;
constexpr int kSignChunk = kRows * 16;        // 4 sign words x 128 rows = 2 KB
constexpr int kPadTile = 8 * kChunk * 2;      // one 8-token tile of one chunk = 2 KB
constexpr int kMaxTok = kSkinnyMaxTokens;
constexpr int kMaxKeys = kMaxVariants + 1;
constexpr int kPhaseTiles = 4;                // padded tiles per variant phase (more: several phases)
constexpr int kTmemCols = 256;               // base sums: columns 0..63; variant sums: 8 per padded tile
constexpr int kVarCol = 64;
constexpr int kMaxVarTiles = (kTmemCols - kVarCol) / 8;  // padded tiles one group may hold

// ---- multi_prepare_kernel
constexpr int kPrepThreads = 128;             // one task (chunk, 32-column group) per thread
constexpr int kPrepChunks = kPrepThreads / 4; // chunks per prepare block (column split)

// Chunks per variant stage for a phase of L padded tiles: the largest power
// of two (at most 8) whose stage fits one ring slot, so that it divides the
// chunk count of a slice in the common case and the chunk loop unrolls.
__host__ __device__ constexpr int phase_group(int L)
{
    return kVarSlot >= 8 * (kSignChunk + L * kPadTile)   ? 8
           : kVarSlot >= 4 * (kSignChunk + L * kPadTile) ? 4
           : kVarSlot >= 2 * (kSignChunk + L * kPadTile) ? 2
                                                           : 1;
}

// Recoding: kind k = column residue mod 4.  The operand pair of kind k is
// (rotated word & recode_mask(k)) ^ kRecodeConst: one bf16 -0.5 per half with
// the kind's bit placed into mantissa bit 4, 5 or 6 (value -0.5 - b/16,
// -0.5 - b/8, -0.5 - b/4) or XORed into the sign bit (-0.5 + b).  The x
// operand of kind k is pre-scaled by recode_sigma(k) = -16, -8, -4, 1 (exact
// power-of-two scalings), which makes every product x * (a_k + b) with
// a_k = 8, 4, 2, -0.5.
constexpr uint32_t kRecodeConst = 0xBF00BF00u;
__host__ __device__ constexpr uint32_t recode_mask(int k)
{
    return k == 0 ? 0x00100010u : k == 1 ? 0x00200020u : k == 2 ? 0x00400040u : 0x80008000u;
}
__host__ __device__ constexpr int recode_lo_bit(int k) { return k == 0 ? 4 : k == 1 ? 5 : k == 2 ? 6 : 15; }
__host__ __device__ constexpr float recode_sigma(int k) { return k == 0 ? -16.0f : k == 1 ? -8.0f : k == 2 ? -4.0f : 1.0f; }
// 2 a_k + 1 for the per-token correction C.
__host__ __device__ constexpr float recode_corr(int k) { return k == 0 ? 17.0f : k == 1 ? 9.0f : k == 2 ? 5.0f : 0.0f; }

struct MultiParams {
    CUtensorMap sign_map[kMaxVariants];  // [d_out][d_in/32] uint32, box 4 x 128 rows
    CUtensorMap w_map;                   // [d_out][d_in] bf16, box 64 x 128 rows, 128B swizzle
    CUtensorMap x_map;                   // x [T][d_in] bf16 (caller order), box 64 x max(16, 8*NT), 128B swizzle
    const uint8_t* xp;                   // padded, permuted, scaled tiles of the variant phases
    int64_t xp_bytes;                    // their extent (bounds-checked builds)
    const float* corr;                   // [T][nsplit] partial corrections C per sorted position
    const int32_t* vid;
    const float* alpha[kMaxVariants];
    void* y;
    uint32_t* err;
    int64_t T, d_out, d_in;
    int V, per_row, out_f32, CK, nsplit;
    // kRecodeConst, passed at run time so that it sits in a register and each
    // operand pair is a single three-input logic op (mask immediate, constant
    // register) instead of two ops with two immediates
    uint32_t recode_const;
};

// Result of the per-block router (identical in every block of a group).
struct Routing {
    int key[kMaxTok];    // key of token t (caller order); key = vid + 1, 0 = base model
    int perm[kMaxTok];   // sorted position -> token
    int keyp[kMaxTok];   // sorted position -> key
    int rank[kMaxTok];   // token t -> rank among the earlier tokens with its key
    int cnt[kMaxKeys];   // tokens per key
    int cnt0[kMaxKeys];  // tokens per key among tokens 0..31
    int seg[kMaxKeys + 1];
    int slot_of_key[kMaxKeys];
    int act[kMaxTok];    // slot -> variant id
    int len[kMaxTok];    // slot -> padded 8-token tiles of that variant
    int ptile[kMaxTok];  // slot -> first padded tile (over all slots)
    int invp[kMaxTok];   // token -> sorted position
    int n_act;
    int n_ptiles;
};

// Stable counting sort of the T (<= 64) tokens by key = vid + 1 (ids outside
// [-1, V) become base tokens and are flagged by block 0 of a launch when err
// is set), then the active variants in key order and their padded tiles.
// Needs at least 96 threads; ends with __syncthreads.  Ranks come from
// __match_any_sync inside each 32-token warp plus warp 0's per-key counts; the
// per-key offsets, slots and padded-tile offsets from one warp's prefix scans.
__device__ void route_group(Routing& rt, const int32_t* vid, int T, int V, uint32_t* err, int tid)
{
    const int lane = tid & 31, warp = tid >> 5;
    if (tid < kMaxKeys) {
        rt.cnt[tid] = 0;
        rt.cnt0[tid] = 0;
    }
    __syncthreads();
    if (tid < kMaxTok) {
        int k = -1;
        if (tid < T) {
            const int v = bd_in(kBkMulti, tid, T) ? vid[tid] : -1;
            const bool ok = (v >= -1 && v < V);
            if (!ok && blockIdx.x == 0 && blockIdx.y == 0) raise_error(err, kErrBadVariant);
            k = ok ? v + 1 : 0;
            rt.key[tid] = k;
        }
        // lanes past T get distinct negative labels and never match a real key
        const unsigned peers = __match_any_sync(0xffffffffu, tid < T ? k : -1 - lane);
        if (tid < T) {
            rt.rank[tid] = __popc(peers & ((1u << lane) - 1u));
            if (lane == __ffs(peers) - 1) {
                atomicAdd(&rt.cnt[k], __popc(peers));
                if (warp == 0) rt.cnt0[k] = __popc(peers);
            }
        }
    }
    __syncthreads();
    if (warp == 0) {
        int carry_seg = 0, carry_slot = 0, carry_pt = 0;
        for (int base = 0; base <= V; base += 32) {
            const int k = base + lane;
            const int c = k <= V ? rt.cnt[k] : 0;
            const int a = (k >= 1 && c > 0) ? 1 : 0;
            const int ln = a ? (c + 7) / 8 : 0;
            int sc = c, sa = a, sl = ln;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int tc = __shfl_up_sync(0xffffffffu, sc, o);
                const int ta = __shfl_up_sync(0xffffffffu, sa, o);
                const int tl = __shfl_up_sync(0xffffffffu, sl, o);
                if (lane >= o) {
                    sc += tc;
                    sa += ta;
                    sl += tl;
                }
            }
            if (k <= V) {
                rt.seg[k] = carry_seg + sc - c;
                rt.slot_of_key[k] = a ? carry_slot + sa - 1 : -1;
                if (a) {
                    rt.act[carry_slot + sa - 1] = k - 1;
                    rt.len[carry_slot + sa - 1] = ln;
                    rt.ptile[carry_slot + sa - 1] = carry_pt + sl - ln;
                }
            }
            carry_seg += __shfl_sync(0xffffffffu, sc, 31);
            carry_slot += __shfl_sync(0xffffffffu, sa, 31);
            carry_pt += __shfl_sync(0xffffffffu, sl, 31);
        }
        if (lane == 0) {
            rt.seg[V + 1] = carry_seg;
            rt.n_act = carry_slot;
            rt.n_ptiles = carry_pt;
        }
    }
    __syncthreads();
    if (tid < T) {
        const int k = rt.key[tid];
        const int pos = rt.seg[k] + rt.rank[tid] + (warp == 1 ? rt.cnt0[k] : 0);
        rt.perm[pos] = tid;
        rt.keyp[pos] = k;
        rt.invp[tid] = pos;
    }
    __syncthreads();
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p)
{
    return p + ((1024u - (smem_u32(p) & 1023u)) & 1023u);
}

// Bounded wait that also gives up as soon as another warp of the CTA has
// timed out (sets the CTA-wide abort flag and the error word on timeout).
__device__ __forceinline__ bool wait_or_abort(volatile int& abort, uint64_t* bar, uint32_t parity, uint32_t* err)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (abort) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            abort = 1;
            raise_error(err, kErrTimeout);
            return false;
        }
    }
    return true;
}

// ---------------------------------------------------------------- prepare pass

// bf16 bits of sigma * x for a power-of-two sigma (exact up to overflow).
__device__ __forceinline__ uint16_t scaled_bits(uint16_t xb, float sigma)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(sigma * __bfloat162float(__ushort_as_bfloat16(xb))));
}

// Block (b, s): b < T handles sorted token position b, b >= T one empty row
// of a padded tile; s is a split of kPrepChunks chunks of d_in.  Writes:
//   xp    padded tiles: for slot a, chunk c, tile r (of len_a), a 2 KB block
//         at ((ptile_a * nc + c * len_a + r) * 2 KB) whose 16-byte piece
//         (i, g, q) at ((i * 8 + g) * 4 + q) * 16 holds token row g of the
//         tile, columns 32q + 8i .. 32q + 8i + 7 of the chunk in recoded order
//         and scaling;
//   corr  [T][nsplit] partial C = sum_j x_j (2 a_(j mod 4) + 1) of split s
//         (fp32, fixed summation order).
__global__ void __launch_bounds__(kPrepThreads) multi_prepare_kernel(const uint16_t* __restrict__ x,
                                                                     const int32_t* __restrict__ vid, int T, int V,
                                                                     int64_t d_in, uint8_t* __restrict__ xp,
                                                                     float* __restrict__ corr, int nsplit,
                                                                     int64_t xp_bytes)
{
    __shared__ Routing rt;
    __shared__ float part[kPrepThreads / 32];
    const int tid = threadIdx.x;
    // the fused kernel that follows may start now: its routing and base phase
    // read only the caller's inputs; it waits for this grid before it reads
    // the padded tiles or the corrections
    grid_launch_dependents();
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
    const int c = static_cast<int>(blockIdx.y) * kPrepChunks + (tid >> 2), q = tid & 3;
    float c_sum = 0.0f;
    if (c < nc) {
        const int64_t col0 = static_cast<int64_t>(c) * kChunk + 32 * q;
        uint16_t v[32];
        if (xrow && bd_in_range(kBkMultiPrepare, static_cast<int64_t>(rt.perm[pos]) * d_in + col0, 32,
                                static_cast<int64_t>(T) * d_in)) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint4 w = ld_nc_v4(xrow + col0 + 8 * u);
                v[8 * u + 0] = static_cast<uint16_t>(w.x); v[8 * u + 1] = static_cast<uint16_t>(w.x >> 16);
                v[8 * u + 2] = static_cast<uint16_t>(w.y); v[8 * u + 3] = static_cast<uint16_t>(w.y >> 16);
                v[8 * u + 4] = static_cast<uint16_t>(w.z); v[8 * u + 5] = static_cast<uint16_t>(w.z >> 16);
                v[8 * u + 6] = static_cast<uint16_t>(w.w); v[8 * u + 7] = static_cast<uint16_t>(w.w >> 16);
            }
#pragma unroll
            for (int j = 0; j < 32; ++j)
                c_sum = fmaf(__bfloat162float(__ushort_as_bfloat16(v[j])), recode_corr(j & 3), c_sum);
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
                    o[k] = static_cast<uint32_t>(scaled_bits(v[lo], recode_sigma(k))) |
                           (static_cast<uint32_t>(scaled_bits(v[hi], recode_sigma(k))) << 16);
                }
                if (bd_in_range(kBkMultiPrepare, (tile - xp) + ((i * 8 + g) * 4 + q) * 16, 16, xp_bytes))
                    *reinterpret_cast<uint4*>(tile + ((i * 8 + g) * 4 + q) * 16) = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
    }
    if (pos < 0) return;
    // fixed-order block reduction of this split's share of C (deterministic)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c_sum += __shfl_xor_sync(0xffffffffu, c_sum, o);
    if ((tid & 31) == 0) part[tid >> 5] = c_sum;
    __syncthreads();
    if (tid == 0) {
        float s = 0.0f;
        for (int w = 0; w < kPrepThreads / 32; ++w) s += part[w];
        if (bd_in(kBkMultiPrepare, static_cast<int64_t>(pos) * nsplit + blockIdx.y, static_cast<int64_t>(T) * nsplit))
            corr[static_cast<int64_t>(pos) * nsplit + blockIdx.y] = s;
    }
}

// ---------------------------------------------------------------- variant phases and the fused kernel

struct MultiShared {
    uint64_t full[kVarStages];      // variant stage landed (TMA)
    uint64_t empty[kVarStages];     // variant stage consumed (8 consumer warps)
    uint64_t full_b[kBaseStages];   // base stage landed (TMA)
    uint64_t empty_b[kBaseStages];  // base stage read by the tensor core (tcgen05.commit)
    uint64_t accum;                 // every base MMA complete
    uint32_t tmem_base;
    volatile int abort;
    Routing rt;
    int col2pos[kMaxVarTiles * 8];  // variant tensor-memory column -> sorted position (-1: padding)
};

// Consumer side of one variant phase over L padded tiles (tiles t0 ..
// t0 + L - 1 of the variant in slot `slot`): the sign MMAs over the CTA's
// d_in slice, then alpha * 2M of each padded tile stored into the tile's 8
// tensor-memory columns (one 16-lane x 8-column store per tile, whose thread
// layout is that of the MMA accumulator).  Returns false when the pipeline was
// aborted.  i_stage is the running variant-stage counter shared with the
// producer's schedule; rl0 is the warp's first row (its 16 rows lie in the
// warp's tensor-memory lane quarter).
template <int L>
__device__ __forceinline__ bool variant_phase(MultiShared& sh, const MultiParams& p, const uint8_t* vring, int slot,
                                              int t0, int n_chunks, int& i_stage, uint32_t tmem_rows, int rl0, int g,
                                              int q, int64_t row0)
{
    constexpr int grp = phase_group(L);
    // Variants with one or two tiles keep two accumulator sets (even and odd
    // MMA steps) so that consecutive MMAs do not wait on each other.
    constexpr int NS = L <= 2 ? 2 : 1;
    float acc[L][NS][4];
#pragma unroll
    for (int r = 0; r < L; ++r)
#pragma unroll
        for (int h = 0; h < NS; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[r][h][e] = 0.0f;
    rl0 += g;
    const uint32_t rc = p.recode_const;
    bool ok = true;
    for (int c0 = 0; c0 < n_chunks; c0 += grp) {
        const int cnt = n_chunks - c0 < grp ? n_chunks - c0 : grp;
        const int s = i_stage % kVarStages;
        if (!__all_sync(0xffffffffu, wait_or_abort(sh.abort, &sh.full[s],
                                                   static_cast<uint32_t>(i_stage / kVarStages) & 1u, p.err))) {
            ok = false;
            break;
        }
        const uint8_t* st = vring + static_cast<size_t>(s) * kVarSlot;
        const uint8_t* pads = st + cnt * kSignChunk;
        auto chunk = [&](int cc) {
            const uint32_t* sg = reinterpret_cast<const uint32_t*>(st + cc * kSignChunk);
            const uint32_t w0 = sg[rl0 * 4 + q], w1 = sg[(rl0 + 8) * 4 + q];
            const uint8_t* pc = pads + cc * L * kPadTile + ((g * 4 + q) << 4);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t u0 = __funnelshift_r(w0, w0, 4 * i), u1 = __funnelshift_r(w1, w1, 4 * i);
                uint32_t a0[4], a1[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    a0[k] = (u0 & recode_mask(k)) ^ rc;
                    a1[k] = (u1 & recode_mask(k)) ^ rc;
                }
#pragma unroll
                for (int r = 0; r < L; ++r) {
                    const uint4 xv = *reinterpret_cast<const uint4*>(pc + r * kPadTile + i * 512);
                    mma_bf16_16816(acc[r][0], a0[0], a1[0], a0[1], a1[1], xv.x, xv.y);
                    mma_bf16_16816(acc[r][NS - 1], a0[2], a1[2], a0[3], a1[3], xv.z, xv.w);
                }
            }
        };
        if (cnt == grp) {
#pragma unroll
            for (int cc = 0; cc < grp; ++cc) chunk(cc);  // full stage: addresses are immediates
        } else {
            for (int cc = 0; cc < cnt; ++cc) chunk(cc);
        }
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(&sh.empty[s]);
        ++i_stage;
    }
    if (!ok) return false;
    // alpha * 2M of the phase's tiles into tensor memory
    const Routing& rt = sh.rt;
    const int v = rt.act[slot];
    const int64_t ra = row0 + rl0, rb = ra + 8;
    const float* al = p.alpha[v];
    const int64_t na = p.per_row ? p.d_out : 1;
    const float a2a = ra < p.d_out && bd_in(kBkMulti, p.per_row ? ra : 0, na) ? 2.0f * al[p.per_row ? ra : 0] : 0.0f;
    const float a2b = rb < p.d_out && bd_in(kBkMulti, p.per_row ? rb : 0, na) ? 2.0f * al[p.per_row ? rb : 0] : 0.0f;
#pragma unroll
    for (int r = 0; r < L; ++r) {
        float m[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) m[e] = NS == 2 ? acc[r][0][e] + acc[r][NS - 1][e] : acc[r][0][e];
        const uint32_t col = static_cast<uint32_t>(kVarCol + 8 * (rt.ptile[slot] + t0 + r));
        tmem_st_16x256b(tmem_rows + col, __float_as_uint(a2a * m[0]), __float_as_uint(a2a * m[1]),
                        __float_as_uint(a2b * m[2]), __float_as_uint(a2b * m[3]));
    }
    tmem_wait_st();
    return true;
}

template <int NT>
__device__ __forceinline__ bool run_phase(int L, MultiShared& sh, const MultiParams& p, const uint8_t* vring, int slot,
                                          int t0, int n_chunks, int& i_stage, uint32_t tmem_rows, int rl0, int g,
                                          int q, int64_t row0)
{
    switch (L) {
        case 1: return variant_phase<1>(sh, p, vring, slot, t0, n_chunks, i_stage, tmem_rows, rl0, g, q, row0);
        case 2:
            if constexpr (NT >= 2)
                return variant_phase<2>(sh, p, vring, slot, t0, n_chunks, i_stage, tmem_rows, rl0, g, q, row0);
            break;
        case 3:
            if constexpr (NT >= 4)
                return variant_phase<3>(sh, p, vring, slot, t0, n_chunks, i_stage, tmem_rows, rl0, g, q, row0);
            break;
        case 4:
            if constexpr (NT >= 4)
                return variant_phase<4>(sh, p, vring, slot, t0, n_chunks, i_stage, tmem_rows, rl0, g, q, row0);
            break;
        default: break;
    }
    // unreachable: a phase never holds more tiles than the group has token tiles
    sh.abort = 1;
    raise_error(p.err, kErrTimeout);
    return false;
}

// The fused multi-variant linear over one CTA's 128 rows and d_in slice (see
// the file comment for the three roles), then the epilogue.
template <int NT>
__global__ void __launch_bounds__(kThreads, 2) multi_kernel(const __grid_constant__ MultiParams p)
{
    constexpr int Tpad = 8 * NT;                    // per-token sum columns (sorted positions)
    constexpr int Npad = Tpad < 16 ? 16 : Tpad;     // tcgen05 N (M = 128 needs N % 16 == 0)
    constexpr int kXTile = Npad * kHalfRowBytes;    // x box [Npad tokens x 64 columns]
    constexpr int kBaseStage = kWTile + kXTile;
    constexpr int kRedStride = Tpad + 1;            // odd: conflict-free column walks
    constexpr uint32_t kIdesc = idesc_bf16_f32(kRows, Npad);

    extern __shared__ uint8_t dyn_raw[];
    __shared__ MultiShared sh;
    uint8_t* bring = align1024(dyn_raw);            // base ring (1024-byte aligned stages)
    uint8_t* vring = bring + kBaseStages * kBaseStage;

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, q = lane & 3;
    const int T = static_cast<int>(p.T);
    const int CK = p.CK;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int64_t row0 = static_cast<int64_t>(blockIdx.x / CK) * kRows;

    route_group(sh.rt, p.vid, T, p.V, p.err, tid);
    if (tid == 0) {
        for (int s = 0; s < kVarStages; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], kConsumers);
        }
        for (int s = 0; s < kBaseStages; ++s) {
            mbar_init(&sh.full_b[s], 1);
            mbar_init(&sh.empty_b[s], 1);
        }
        mbar_init(&sh.accum, 1);
        sh.abort = 0;
        fence_mbarrier_init();
    }
    for (int c = tid; c < kMaxVarTiles * 8; c += kThreads) sh.col2pos[c] = -1;
    if (warp == kBaseWarp) tmem_alloc(&sh.tmem_base, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    // variant tensor-memory column of every routed token (padding columns stay -1)
    if (tid < T && sh.rt.keyp[tid] >= 1) {
        const int k = sh.rt.keyp[tid];
        const int a = sh.rt.slot_of_key[k];
        const int col = 8 * sh.rt.ptile[a] + (tid - sh.rt.seg[k]);
        if (col < kMaxVarTiles * 8) sh.col2pos[col] = tid;
    }

    const int n_act = sh.rt.n_act;
    const int nc = static_cast<int>(p.d_in / kChunk);
    const int c_begin = static_cast<int>(static_cast<int64_t>(rank) * nc / CK);
    const int c_end = static_cast<int>(static_cast<int64_t>(rank + 1) * nc / CK);
    const int n_chunks = c_end - c_begin;

    if (warp == kBaseWarp) {
        // ------------------------------------------------------------ base phase (one thread)
        // x . W_base^T on the tensor cores, concurrently with the variant
        // phases: 64-column stages of W_base [128 x 64] and x [Npad x 64]
        // (caller token order), tcgen05.mma M = 128, N = Npad, K = 16, fp32
        // accumulator in tensor memory.  A slot is refilled as soon as the MMAs
        // reading it complete (a few hundred cycles after they are issued), so
        // that kBaseStages - 1 stages stay in flight while the next one lands.
        if (lane == 0) {
            const int nk = 2 * n_chunks;
            int issued = 0, done = 0;
            auto issue = [&](int k) {
                const int s = k % kBaseStages;
                uint8_t* st = bring + static_cast<size_t>(s) * kBaseStage;
                const int col = c_begin * kChunk + 64 * k;
                mbar_arrive_expect_tx(&sh.full_b[s], static_cast<uint32_t>(kBaseStage));
                tma_load_2d(st, &p.w_map, col, static_cast<int>(row0), &sh.full_b[s]);
                tma_load_2d(st + kWTile, &p.x_map, col, 0, &sh.full_b[s]);
            };
            for (; issued < (nk < kBaseStages ? nk : kBaseStages); ++issued) issue(issued);
            for (int k = 0; k < nk; ++k) {
                const int s = k % kBaseStages;
                if (!wait_or_abort(sh.abort, &sh.full_b[s], static_cast<uint32_t>(k / kBaseStages) & 1u, p.err))
                    break;
                tc_fence_after();
                const uint8_t* st = bring + static_cast<size_t>(s) * kBaseStage;
                const uint64_t adesc = smem_desc_sw128(smem_u32(st));
                const uint64_t bdesc = smem_desc_sw128(smem_u32(st + kWTile));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_ss(tmem, adesc + static_cast<uint64_t>(2 * kk), bdesc + static_cast<uint64_t>(2 * kk), kIdesc,
                           (k | kk) != 0 ? 1u : 0u);
                mma_commit(&sh.empty_b[s]);
                ++done;
                // stage k + kBaseStages into this slot once its MMAs are done
                if (issued < nk) {
                    if (!wait_or_abort(sh.abort, &sh.empty_b[s], static_cast<uint32_t>(k / kBaseStages) & 1u, p.err))
                        break;
                    issue(issued++);
                }
            }
            mma_commit(&sh.accum);  // fires once every MMA issued above has completed
            // copies still in flight must land before the CTA reuses the memory
            for (int k = done; k < issued; ++k) {
                const int s = k % kBaseStages;
                const uint32_t par = static_cast<uint32_t>(k / kBaseStages) & 1u;
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(&sh.full_b[s], par) && global_timer_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
        __syncwarp();
    } else if (warp == kProducerWarp) {
        // ------------------------------------------------------------ variant-phase producer
        grid_dependency_wait();  // the padded tiles come from the prepare pass
        int i = 0;
        bool ok = true;
        for (int a = 0; a < n_act && ok; ++a) {
            const int v = sh.rt.act[a], len = sh.rt.len[a];
            const uint8_t* src = p.xp + static_cast<int64_t>(sh.rt.ptile[a]) * nc * kPadTile;
            for (int t0 = 0; t0 < len && ok; t0 += kPhaseTiles) {
                const int L = len - t0 < kPhaseTiles ? len - t0 : kPhaseTiles;
                const int grp = phase_group(L);
                for (int c0 = 0; c0 < n_chunks; c0 += grp) {
                    const int cnt = n_chunks - c0 < grp ? n_chunks - c0 : grp;
                    const int s = i % kVarStages;
                    if (i >= kVarStages &&
                        !__all_sync(0xffffffffu, wait_or_abort(sh.abort, &sh.empty[s],
                                                               static_cast<uint32_t>(i / kVarStages - 1) & 1u, p.err))) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = vring + static_cast<size_t>(s) * kVarSlot;
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&sh.full[s], static_cast<uint32_t>(cnt * (kSignChunk + L * kPadTile)));
                        for (int cc = 0; cc < cnt; ++cc) {
                            const int c = c_begin + c0 + cc;
                            tma_load_2d(st + cc * kSignChunk, &p.sign_map[v], 4 * c, static_cast<int>(row0),
                                        &sh.full[s]);
                            const uint8_t* from = src + (static_cast<int64_t>(c) * len + t0) * kPadTile;
                            if (bd_in_range(kBkMulti, from - p.xp, static_cast<int64_t>(L) * kPadTile, p.xp_bytes))
                                bulk_g2s(st + cnt * kSignChunk + cc * L * kPadTile, from,
                                         static_cast<uint32_t>(L * kPadTile), &sh.full[s]);
                        }
                    }
                    __syncwarp();
                    ++i;
                }
            }
        }
        // every issued stage must have landed before the CTA reuses the memory
        for (int k = (i > kVarStages ? i - kVarStages : 0); k < i; ++k) {
            const int s = k % kVarStages;
            const uint32_t par = static_cast<uint32_t>(k / kVarStages) & 1u;
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(&sh.full[s], par) && global_timer_ns() - t0 < kWaitLimitNs) {
            }
        }
    } else {
        // ------------------------------------------------------------ consumer warps: variant phases
        // warp w owns rows 32 (w % 4) + 16 (w / 4) .. + 15: inside its tensor-memory lane quarter
        const int rl0 = 32 * (warp & 3) + 16 * (warp >> 2);
        const uint32_t tmem_rows = tmem + (static_cast<uint32_t>(rl0) << 16);
        int i = 0;
        bool ok = true;
        for (int a = 0; a < n_act && ok; ++a) {
            const int len = sh.rt.len[a];
            for (int t0 = 0; t0 < len && ok; t0 += kPhaseTiles) {
                const int L = len - t0 < kPhaseTiles ? len - t0 : kPhaseTiles;
                ok = run_phase<NT>(L, sh, p, vring, a, t0, n_chunks, i, tmem_rows, rl0, g, q, row0);
            }
        }
    }

    // ---------------------------------------------------------------- epilogue
    // 1. per-token sums of this CTA's slice, gathered from tensor memory into
    //    shared memory (the variant ring is free): base columns (caller token
    //    order) plus variant tile columns (alpha * 2M), by sorted position.
    //    The indices (and, for the variant columns, the current sums) of a
    //    block of columns are all loaded before its first store, so that the
    //    loads overlap instead of each waiting for the store before it.
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const Routing& rt = sh.rt;
    float* red = reinterpret_cast<float*>(vring);  // [128][Tpad + 1]
    if (warp < 4) {
        const bool base_ok = __all_sync(0xffffffffu, wait_or_abort(sh.abort, &sh.accum, 0u, p.err));
        tc_fence_after();
        const int row = 32 * warp + lane;  // tensor-memory lane = local row
        float* rr = red + row * kRedStride;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * warp) << 16);
        if (base_ok) {
            // every sorted position below T is written: invp is a bijection
#pragma unroll
            for (int cb = 0; cb < (Tpad + 31) / 32; ++cb) {
                uint32_t d[32];
                tmem_ld32(lane_addr + 32 * cb, d);
                int ip[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) ip[j] = 32 * cb + j < T ? rt.invp[32 * cb + j] : -1;
#pragma unroll
                for (int j = 0; j < 32; ++j)
                    if (ip[j] >= 0) rr[ip[j]] = __uint_as_float(d[j]);
            }
        } else {
            for (int pos = 0; pos < Tpad; ++pos) rr[pos] = 0.0f;
        }
        const int vcols = 8 * (rt.n_ptiles < kMaxVarTiles ? rt.n_ptiles : kMaxVarTiles);
        for (int cb = 0; cb < vcols; cb += 32) {
            uint32_t d[32];
            tmem_ld32(lane_addr + kVarCol + cb, d);
#pragma unroll
            for (int h = 0; h < 32; h += 16) {
                int pc[16];
                float cur[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) pc[j] = cb + h + j < vcols ? sh.col2pos[cb + h + j] : -1;
#pragma unroll
                for (int j = 0; j < 16; ++j) cur[j] = pc[j] >= 0 ? rr[pc[j]] : 0.0f;
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (pc[j] >= 0) rr[pc[j]] = cur[j] + __uint_as_float(d[h + j]);
            }
        }
    }
    __syncthreads();  // every base MMA complete, every copy landed: both rings are free
    // 2. push the per-token sums to the owners of their rows (receive slots
    //    [CK][kRows / CK rows][kRecvStride] in the base ring, free once every
    //    peer got here) as 16-byte stores, then each owner adds its slots in
    //    rank order.  Columns T..Tpad-1 carry unused values.
    constexpr int kRecvStride = Tpad + 4;           // 16-byte aligned rows
    constexpr int kQuads = Tpad / 4;                // float4 per row (a power of two)
    float* recv = reinterpret_cast<float*>(bring);
    const int nr = kRows / CK;                      // CK is a power of two up to 8
    const int lnr = 7 - (31 - __clz(CK));           // log2(nr)
    cluster.sync();
    for (int o = tid; o < kRows * kQuads; o += kThreads) {
        const int r = o / kQuads, c4 = 4 * (o % kQuads);
        const int owner = r >> lnr;
        const float* src = red + r * kRedStride + c4;
        const float4 v = make_float4(src[0], src[1], src[2], src[3]);
        float* dst = cluster.map_shared_rank(recv, owner);
        *reinterpret_cast<float4*>(dst + (rank * nr + (r - (owner << lnr))) * kRecvStride + c4) = v;
    }
    __syncthreads();  // red is read above before it is reused below
    // per-token corrections and per-row alphas of this rank's rows, staged in red
    float* corr_s = red;                       // [Tpad]
    float* alpha_s = red + Tpad;               // [n_act][nr]
    if (tid < T) {
        grid_dependency_wait();  // the corrections come from the prepare pass
        float c = 0.0f;
        for (int sp = 0; sp < p.nsplit; ++sp)
            if (bd_in(kBkMulti, static_cast<int64_t>(tid) * p.nsplit + sp, p.T * p.nsplit))
                c += p.corr[static_cast<int64_t>(tid) * p.nsplit + sp];
        corr_s[tid] = c;
    }
    for (int o = tid; o < n_act * nr; o += kThreads) {
        const int a = o >> lnr, r = o & (nr - 1);
        const int64_t row = row0 + rank * nr + r;
        alpha_s[o] = row < p.d_out && bd_in(kBkMulti, p.per_row ? row : 0, p.per_row ? p.d_out : 1)
                         ? p.alpha[rt.act[a]][p.per_row ? row : 0]
                         : 0.0f;
    }
    cluster.sync();
    for (int o = tid; o < nr * T; o += kThreads) {
        const int pos = o >> lnr, r = o & (nr - 1);
        const int64_t row = row0 + rank * nr + r;
        if (row >= p.d_out) continue;
        float y = 0.0f;
        for (int k = 0; k < CK; ++k) y += recv[(k * nr + r) * kRecvStride + pos];
        const int key = rt.keyp[pos];
        if (key >= 1) y = fmaf(-alpha_s[rt.slot_of_key[key] * nr + r], corr_s[pos], y);
        const int64_t idx = static_cast<int64_t>(rt.perm[pos]) * p.d_out + row;
        if (!bd_in(kBkMulti, idx, p.T * p.d_out)) continue;
        if (p.out_f32)
            static_cast<float*>(p.y)[idx] = y;
        else
            static_cast<__nv_bfloat16*>(p.y)[idx] = __float2bfloat16_rn(y);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kBaseWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int NT>
cudaError_t launch_nt(const MultiParams& prm, size_t smem, unsigned grid, cudaStream_t stream)
{
    auto kern = multi_kernel<NT>;
    static std::atomic<size_t> smem_set[kHostMaxDevices];
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem, smem_set);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(prm.CK);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // may start while the prepare pass runs (programmatic dependent launch):
    // the routing, the tensor-memory setup and the base phase overlap it
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, prm);
}

int tiles_for(int T) { return T <= 8 ? 1 : T <= 16 ? 2 : T <= 32 ? 4 : 8; }

// SM count of the current device (cached per device).
int sm_count()
{
    static std::atomic<int> sms[kHostMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kHostMaxDevices) return 1;
    int n = sms[dev].load(std::memory_order_relaxed);
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 1;
        sms[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

}  // namespace

int multi_max_ptiles(int T, int V)
{
    const int t = T < kMaxTok ? T : kMaxTok;
    const int a = t < V ? t : V;
    return (t + 7 * a) / 8;
}

int multi_group_tokens(int V)
{
    for (int g = kMaxTok; g > 8; g /= 2)
        if (multi_max_ptiles(g, V) <= kMaxVarTiles) return g;
    return 8;
}

int multi_corr_splits(int64_t d_in)
{
    const int64_t nc = d_in / kChunk;
    return static_cast<int>((nc + kPrepChunks - 1) / kPrepChunks);
}

cudaError_t launch_multi(const MultiArgs& a, cudaStream_t stream)
{
    const int T = static_cast<int>(a.T);
    if (T < 1 || T > kMaxTok || a.V < 1 || a.V > kMaxVariants) return cudaErrorInvalidValue;
    if (!a.xp || !a.corr) return cudaErrorInvalidValue;
    const int nt = tiles_for(T);
    const int npad = 8 * nt < 16 ? 16 : 8 * nt;
    const int nsplit = multi_corr_splits(a.d_in);
    static thread_local MultiParams prm;  // ~9 KB: kept off the stack
    prm.xp = a.xp;
    prm.xp_bytes = static_cast<int64_t>(multi_max_ptiles(T, a.V)) * 8 * a.d_in * 2;
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
    prm.nsplit = nsplit;
    prm.recode_const = kRecodeConst;
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
        !encode_tma_2d(&prm.x_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, static_cast<uint64_t>(a.d_in),
                       static_cast<uint64_t>(a.T), static_cast<uint64_t>(a.d_in) * 2, 64,
                       static_cast<uint32_t>(npad), CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    // K slices per cluster: one per 2048 columns of d_in, rounded down to a
    // power of two (1, 2 or 4) so that every slice owns kRows / CK rows; for
    // few row blocks (d_out = 1024: 8 blocks) doubled up to 8, the portable
    // cluster size, while the grid is smaller than the SM count and every
    // slice keeps at least 4 chunks
    const int nc = static_cast<int>(a.d_in / kChunk);
    int ck = nc >= 64 ? 4 : nc >= 32 ? 2 : 1;
    const int64_t row_blocks = (a.d_out + kRows - 1) / kRows;
    const int sms = sm_count();
    while (ck < 8 && row_blocks * ck < sms && nc / (2 * ck) >= 4) ck *= 2;
    prm.CK = ck;
    const size_t base_stage = static_cast<size_t>(kWTile) + static_cast<size_t>(npad) * kHalfRowBytes;
    const size_t red = static_cast<size_t>(kRows) * (8 * nt + 1) * sizeof(float);   // in the variant ring
    const size_t recv = static_cast<size_t>(kRows) * (8 * nt + 4) * sizeof(float);  // receive slots, base ring
    if (red > kVarStages * static_cast<size_t>(kVarSlot) || recv > kBaseStages * base_stage)
        return cudaErrorInvalidConfiguration;
    if (multi_max_ptiles(T, a.V) > kMaxVarTiles) return cudaErrorInvalidValue;
    const size_t smem = kBaseStages * base_stage + kVarStages * static_cast<size_t>(kVarSlot) + 1024;

    const dim3 prep_grid(static_cast<unsigned>(T + 7 * (T < a.V ? T : a.V)), static_cast<unsigned>(nsplit));
    multi_prepare_kernel<<<prep_grid, kPrepThreads, 0, stream>>>(a.x, a.vid, T, a.V, a.d_in, a.xp, a.corr, nsplit,
                                                                  prm.xp_bytes);
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

BD_BOUNDS_TAKE(bounds_take_multi)

}  // namespace bd
