// Prefill (T > 64) fused BitDelta linear on the 5th-generation tensor cores
// (section "Sunum mimarisi" of the BitDelta post: W_eff = W_base + alpha*s is
// rebuilt on chip, never in HBM, and the rebuild is fused with the matmul).
//
//   D[r][t] = sum_k W_eff[r][k] * x[t][k],   y[t][r] = D[r][t]
//
// A cluster of two CTAs computes 256-row x 256-token tiles of y^T over all
// of d_in with 2-SM MMAs (tcgen05 .cta_group::2, M = 256): each CTA owns 128
// rows (its tensor-memory lanes, for the A operand and the accumulator) and
// stages half of the tile's tokens, which the pair's MMAs read from both
// CTAs' shared memory.  So an SM takes in 34 KB per 64-column k-step (x half,
// W_base rows, signs) instead of the 50 KB a one-CTA 128 x 256 tile needs for
// the same FLOPs.  The pairs are persistent (one per two SMs that can hold
// one; pair c takes tiles c, c + C, ...), so each role runs ahead into the
// next tile while the current one drains.  Per CTA, through a 6-stage ring:
//   warp 0       TMA producer: x tile [128 tokens x 64] (128-byte swizzle),
//                W_base tile [128 x 64] (128-byte swizzle) and the sign words
//                of the tile's rows, all completing on one mbarrier per stage;
//   warps 2..9   transform: thread = one row of the tile (TMEM lane) and one
//                32-column half of the k-step (two warps per TMEM lane
//                quarter); reads its 32 W_base values from shared memory,
//                adds +alpha or -alpha per sign bit with packed bf16 adds
//                (W_eff rounded to bf16, the MMA's input precision), writes
//                them into the stage's A-operand columns of its CTA's tensor
//                memory with tcgen05.st and arrives on the even CTA's stage
//                barrier;
//   warp 1       in the even CTA, one thread issues the pair's tcgen05.mma
//                (kind::f16, M=256, N=256, K=16; A from tensor memory, B from
//                shared memory, fp32 accumulator in tensor memory) once both
//                CTAs' transforms of a stage are in, frees the stage in both
//                CTAs with a multicast tcgen05.commit, and starts a tile only
//                once both CTAs' epilogues have released the accumulator;
//   warps 10..17 epilogue: tcgen05.ld of the CTA's accumulator rows (two
//                warps per lane quarter, 128 token columns each), released as
//                soon as it is in registers (bf16 output), then the stores.
// So W_eff never goes through shared memory: per k-step the shared memory
// sees the W and x tiles written once by TMA, W read once by the transform
// and x read once by the tensor cores.
//
// Grouped form (multi-variant prefill, bd_linear_multi with large T): x is
// gathered into token order sorted by variant (key = vid + 1), and each
// 256-token block of the grid lies inside one key's segment, listed by a
// plan of {first token, segment end, key}.  A block builds W_eff with its
// key's signs and alpha (alpha = 0 for key 0, the base model: W_eff = W_base
// exactly) and writes only the rows of its own segment, in caller order.  A
// block of n < 256 tokens (a segment's tail) runs its MMAs with N = n rounded
// up to 16, the even CTA staging the first N/2 of its tokens and the odd CTA
// the next N/2.
//
// Every mbarrier wait is bounded; a timeout sets the error word, stops every
// role of the CTA at its next wait (the other CTA of the pair then times out
// on its own waits), drains the copies in flight, waits for the issued MMAs,
// and the pair frees its tensor memory together.
#include <algorithm>
#include <atomic>
#include <type_traits>

#include "bd_device.cuh"
#include "bd_tcgen05.cuh"
#include "bd_tma.h"

namespace bd {
namespace {

constexpr int BM = 128;        // W rows per CTA (tensor-memory lanes); a pair covers 2 * BM (MMA M)
constexpr int BN = 256;        // tokens per pair tile (MMA N)
constexpr int BNH = BN / 2;    // tokens staged per CTA
constexpr int BK = 64;         // k-step (one 128-byte swizzle atom of bf16)
constexpr int kStages = 6;
constexpr int kXBytes = BNH * BK * 2;                     // 16384
constexpr int kWBytes = BM * BK * 2;                      // 16384
constexpr int kSBytes = BM * 16;                          // 4 sign words per row (128 columns)
constexpr int kStageBytes = kXBytes + kWBytes + kSBytes;  // 34816 (multiple of 1024)
constexpr int kThreads = 576;                             // 18 warps
constexpr int kEpilogueWarp0 = 10;                        // warps 10..17: epilogue
constexpr int kTmemCols = 512;                            // D: 256 columns; A ring: 6 x 32 columns
constexpr int kDCol = 0;
constexpr int kACol = 256;
constexpr uint16_t kPairMask = 0x3;  // both CTAs of the cluster
static_assert(kACol + 32 * kStages <= kTmemCols, "tensor-memory columns");

struct PrefillParams {
    CUtensorMap x_map;  // [T][d_in] bf16, box 64 x 128, 128B swizzle
    CUtensorMap w_map;  // [d_out][d_in] bf16, box 64 x 128, 128B swizzle
    CUtensorMap s_map;  // [d_out][d_in/32] u32, box 4 x 128
    const float* alpha;
    void* y;
    uint32_t* err;
    int64_t T, d_out, d_in;
    int per_row, out_f32;
    int ntb;  // 256-token blocks (grouped: plan entries, some past the plan)
};

// Multi-variant prefill: the single-variant fields describe the gathered x
// (x_map over [T][d_in] in sorted order), W_base and y; the sign maps and
// alphas are per variant, the plan and the permutation come from the router.
struct GroupedPrefillParams : PrefillParams {
    const int4* plan;                     // [grid.x] {first token, segment end, key, valid}
    const int32_t* perm;                  // sorted position -> caller token
    const float* alphas[kMaxVariants];
    CUtensorMap s_maps[kMaxVariants];     // [d_out][d_in/32] u32 per variant, box 4 x 128
};

struct PrefillShared {
    uint64_t full[kStages];   // this CTA's TMA landed
    uint64_t afull[kStages];  // even CTA: both CTAs' transforms wrote the A stage (16 warp arrivals)
    uint64_t empty[kStages];  // the pair MMAs reading the stage finished (multicast tcgen05.commit)
    uint64_t accum;           // a tile's pair MMAs finished (multicast tcgen05.commit; one phase per tile)
    uint64_t dfree;           // even CTA: both CTAs' epilogues read the accumulator (16 warp arrivals)
    uint64_t mma_done;        // even CTA: every MMA it issued finished (teardown)
    uint32_t tmem_base;
    volatile int abort;
};

// Bounded wait; kCluster: acquire at cluster scope (a barrier that the other
// CTA of the pair arrives on).
template <bool kCluster = false>
__device__ __forceinline__ bool pwait(PrefillShared& sh, uint64_t* bar, uint32_t parity, uint32_t* err)
{
    auto poll = [&] { return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
    if (poll()) return true;
    const uint64_t t0 = global_timer_ns();
    while (!poll()) {
        if (sh.abort) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            sh.abort = 1;
            raise_error(err, kErrTimeout);
            return false;
        }
    }
    return true;
}

// The tile a CTA pair works on: tokens [tok0, tok_end) of a 256-token block
// (MMA N = nmma), this CTA's 128 rows from row0, its x rows from xtok, and
// the key's sign map and alpha.  Tiles are numbered row pair major, token
// block minor, so the clusters in flight share W_base rows in L2.
struct TileInfo {
    int64_t tok0, tok_end, xtok, row0;
    const CUtensorMap* s_map;
    const float* alpha;
    int nmma;
    bool valid;
};

constexpr int kRasterPairs = 8;  // grouped prefill: row pairs per raster group

template <class P>
__device__ __forceinline__ TileInfo tile_info(const P& p, int t, uint32_t rank)
{
    constexpr bool kGrouped = std::is_same<P, GroupedPrefillParams>::value;
    TileInfo ti;
    int tb = t % p.ntb, rp = t / p.ntb;
    if constexpr (kGrouped) {
        // groups of kRasterPairs row pairs x every block, block-major inside
        // a group: the group's W_base rows and the blocks' x stay in L2
        const int nrp = static_cast<int>((p.d_out + 2 * BM - 1) / (2 * BM));
        const int per = kRasterPairs * p.ntb;
        const int g = t / per, loc = t - g * per;
        const int gp = nrp - g * kRasterPairs < kRasterPairs ? nrp - g * kRasterPairs : kRasterPairs;
        tb = loc / gp;
        rp = g * kRasterPairs + (loc - tb * gp);
    }
    ti.row0 = (2 * static_cast<int64_t>(rp) + rank) * BM;
    ti.tok0 = static_cast<int64_t>(tb) * BN;
    ti.tok_end = p.T;
    ti.s_map = &p.s_map;
    ti.alpha = p.alpha;
    ti.nmma = BN;
    ti.valid = true;
    if constexpr (kGrouped) {
        const int4 b = bd_in(kBkPrefill, tb, p.ntb) ? p.plan[tb] : make_int4(0, 0, 0, 0);
        ti.valid = b.w != 0 && bd_in(kBkPrefill, b.z, kMaxVariants + 1);  // past the plan
        ti.tok0 = b.x;
        ti.tok_end = b.y;
        ti.s_map = &p.s_maps[b.z >= 1 ? b.z - 1 : 0];
        ti.alpha = b.z >= 1 ? p.alphas[b.z - 1] : nullptr;  // key 0: alpha = 0, W_eff = W_base
        // a segment's tail: N = its token count rounded up to 16
        const int n = ti.tok_end - ti.tok0 < BN ? static_cast<int>(ti.tok_end - ti.tok0) : BN;
        ti.nmma = (n + 15) / 16 * 16;
    }
    // this CTA stages tokens tok0 + rank * N/2 .. + N/2 - 1 (rows past N/2 of
    // the 128-token box are loaded but not multiplied)
    ti.xtok = ti.tok0 + static_cast<int64_t>(rank) * (ti.nmma / 2);
    return ti;
}

template <class P>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ P p)
{
    extern __shared__ uint8_t dyn_raw[];
    __shared__ PrefillShared sh;
    uint8_t* dyn = dyn_raw + ((1024u - (smem_u32(dyn_raw) & 1023u)) & 1023u);
    grid_dependency_wait();  // launched early (programmatic dependent launch): the previous kernel is done

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();  // 0: even CTA (rows 0..127 of the pair, issues the MMAs)
    // persistent pairs: cluster c takes tiles c, c + C, c + 2C, ... (pairs lie
    // along the cluster's x dimension: grid x = 2 * C)
    const int cid = static_cast<int>(blockIdx.x >> 1), ncl = static_cast<int>(gridDim.x >> 1);
    const int ntiles = p.ntb * static_cast<int>((p.d_out + 2 * BM - 1) / (2 * BM));
    const int nk = static_cast<int>(p.d_in / BK);

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.afull[s], 16);
            mbar_init(&sh.empty[s], 1);
        }
        mbar_init(&sh.accum, 1);
        mbar_init(&sh.dfree, 16);
        mbar_init(&sh.mma_done, 1);
        sh.abort = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) tmem_alloc_pair(&sh.tmem_base, kTmemCols);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers are initialised before any remote arrival
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;

    // Every role walks the same tiles and k-steps; g counts k-steps over all
    // of them (ring slot g % kStages, phase g / kStages), j counts tiles
    // (accumulator phase j).
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            uint32_t g = 0;
            bool ok = true;
            for (int t = cid; t < ntiles && ok; t += ncl) {
                const TileInfo ti = tile_info(p, t, rank);
                if (!ti.valid) continue;
                for (int i = 0; i < nk; ++i, ++g) {
                    const int s = static_cast<int>(g % kStages);
                    if (g >= kStages && !pwait(sh, &sh.empty[s], (g / kStages - 1) & 1u, p.err)) {
                        ok = false;
                        break;
                    }
                    uint8_t* st = dyn + s * kStageBytes;
                    mbar_arrive_expect_tx(&sh.full[s], kStageBytes);
                    tma_load_2d(st, &p.x_map, i * BK, static_cast<int>(ti.xtok), &sh.full[s]);
                    tma_load_2d(st + kXBytes, &p.w_map, i * BK, static_cast<int>(ti.row0), &sh.full[s]);
                    tma_load_2d(st + kXBytes + kWBytes, ti.s_map, 4 * (i / 2), static_cast<int>(ti.row0),
                                &sh.full[s]);
                }
            }
            // copies still in flight must land before the CTA ends
            for (uint32_t u = g > kStages ? g - kStages : 0; u < g; ++u) {
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(&sh.full[u % kStages], (u / kStages) & 1u) &&
                       global_timer_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (even CTA)
        if (lane == 0 && rank == 0) {
            uint32_t g = 0, j = 0;
            bool ok = true;
            for (int t = cid; t < ntiles && ok; t += ncl) {
                const TileInfo ti = tile_info(p, t, rank);
                if (!ti.valid) continue;
                // the accumulator is free once both CTAs' epilogues have read the previous tile
                if (j > 0 && !pwait<true>(sh, &sh.dfree, (j - 1) & 1u, p.err)) break;
                tc_fence_after();
                const uint32_t idesc = idesc_bf16_f32(2 * BM, ti.nmma);
                for (int i = 0; i < nk; ++i, ++g) {
                    const int s = static_cast<int>(g % kStages);
                    if (!pwait<true>(sh, &sh.afull[s], (g / kStages) & 1u, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bdesc = smem_desc_sw128(smem_u32(dyn + s * kStageBytes));
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        mma_ts_pair(tmem + kDCol, tmem + kACol + 32 * s + 8 * kk,
                                    bdesc + static_cast<uint64_t>(2 * kk), idesc, (i | kk) != 0 ? 1u : 0u);
                    mma_commit_pair(&sh.empty[s], kPairMask);
                }
                if (ok) {
                    mma_commit_pair(&sh.accum, kPairMask);  // the tile's accumulator is complete
                    ++j;
                }
            }
            // tensor memory is freed below only after every MMA issued above is done
            mma_commit_pair(&sh.mma_done, 0x1);
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(&sh.mma_done, 0u) && global_timer_ns() - t0 < kWaitLimitNs) {
            }
        }
    } else if (warp < kEpilogueWarp0) {
        // ------------------------------------------------------------ transform
        const int quarter = warp & 3;     // TMEM lanes 32*quarter .. +31
        const int ch = (warp - 2) >> 2;   // column half of the k-step (warps 2..5 -> 0, 6..9 -> 1)
        const int rl = 32 * quarter + lane;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * quarter) << 16);
        uint32_t g = 0;
        bool ok = true;
        for (int t = cid; t < ntiles && ok; t += ncl) {
            const TileInfo ti = tile_info(p, t, rank);
            if (!ti.valid) continue;
            const int64_t row = ti.row0 + rl;
            float a = 0.0f;
            if (ti.alpha && row < p.d_out && bd_in(kBkPrefill, p.per_row ? row : 0, p.per_row ? p.d_out : 1))
                a = ti.alpha[p.per_row ? row : 0];
            const uint32_t ab = static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(a)));
            const uint32_t neg = ((ab << 16) | ab) ^ 0x80008000u;  // (-alpha, -alpha) as bf16x2
            for (int i = 0; i < nk; ++i, ++g) {
                const int s = static_cast<int>(g % kStages);
                if (!__all_sync(0xffffffffu, pwait(sh, &sh.full[s], (g / kStages) & 1u, p.err))) {
                    ok = false;
                    break;
                }
                const uint8_t* st = dyn + s * kStageBytes;
                const uint8_t* wrow = st + kXBytes + rl * 128;
                const uint32_t* srow = reinterpret_cast<const uint32_t*>(st + kXBytes + kWBytes + rl * 16);
                const uint32_t word = srow[2 * (i & 1) + ch];  // sign bits of this warp's 32 columns
                uint32_t v[16];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int cc = 4 * ch + c;  // 16-byte chunk within the 128-byte row
                    const uint4 u = *reinterpret_cast<const uint4*>(wrow + ((cc ^ (rl & 7)) << 4));
                    v[4 * c + 0] = u.x;
                    v[4 * c + 1] = u.y;
                    v[4 * c + 2] = u.z;
                    v[4 * c + 3] = u.w;
                }
#pragma unroll
                for (int hw = 0; hw < 2; ++hw) {  // 16 columns per sign half-word
                    const uint32_t h = (word >> (16 * hw)) & 0xFFFFu;
                    const uint32_t z = (h | (h << 15)) & 0x55555555u;
#pragma unroll
                    for (int pp = 0; pp < 8; ++pp) {
                        const uint32_t add = neg ^ ((z << (15 - 2 * pp)) & 0x80008000u);  // +alpha where bit = 1
                        __nv_bfloat162 w2 = *reinterpret_cast<__nv_bfloat162*>(&v[8 * hw + pp]);
                        const __nv_bfloat162 a2 = *reinterpret_cast<const __nv_bfloat162*>(&add);
                        w2 = __hadd2(w2, a2);
                        v[8 * hw + pp] = *reinterpret_cast<uint32_t*>(&w2);
                    }
                }
                tmem_st16(lane_addr + kACol + 32 * s + 16 * ch, v);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(&sh.afull[s], 0);
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue
        // warps 10..17: lane quarter warp % 4, token columns 128 * half ..
        // +127 of the accumulator.  bf16 output: the columns are read into
        // registers as packed bf16 and the accumulator is released before
        // the stores, which then overlap the next tile's MMAs; fp32 output
        // releases it after the stores.
        const int quarter = warp & 3;
        const int half = (warp - kEpilogueWarp0) >> 2;
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * quarter) << 16);
        uint32_t j = 0;
        for (int t = cid; t < ntiles; t += ncl) {
            const TileInfo ti = tile_info(p, t, rank);
            if (!ti.valid) continue;
            if (!__all_sync(0xffffffffu, pwait(sh, &sh.accum, j & 1u, p.err))) break;
            tc_fence_after();
            const int64_t row = ti.row0 + 32 * quarter + lane;
            const int c0 = 128 * half;
            auto store = [&](int col, float val) {
                int64_t tk = ti.tok0 + col;
                if (tk >= ti.tok_end || row >= p.d_out) return;
                if constexpr (std::is_same<P, GroupedPrefillParams>::value) {
                    if (!bd_in(kBkPrefill, tk, p.T)) return;
                    tk = p.perm[tk];
                }
                if (!bd_in(kBkPrefill, tk * p.d_out + row, p.T * p.d_out)) return;
                if (p.out_f32)
                    static_cast<float*>(p.y)[tk * p.d_out + row] = val;
                else
                    static_cast<__nv_bfloat16*>(p.y)[tk * p.d_out + row] = __float2bfloat16_rn(val);
            };
            if (p.out_f32) {
                for (int cb = 0; cb < 4 && c0 + 32 * cb < ti.nmma; ++cb) {
                    uint32_t d[32];
                    tmem_ld32(lane_addr + kDCol + c0 + 32 * cb, d);
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) store(c0 + 32 * cb + jj, __uint_as_float(d[jj]));
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(&sh.dfree, 0);
            } else {
                uint32_t pk[64];  // bf16 pairs of columns c0 + 2q, c0 + 2q + 1
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    pk[8 * c] = pk[8 * c + 1] = pk[8 * c + 2] = pk[8 * c + 3] = 0u;
                    pk[8 * c + 4] = pk[8 * c + 5] = pk[8 * c + 6] = pk[8 * c + 7] = 0u;
                    if (c0 + 16 * c < ti.nmma) {
                        uint32_t d[16];
                        tmem_ld16(lane_addr + kDCol + c0 + 16 * c, d);
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const __nv_bfloat162 h2 =
                                __floats2bfloat162_rn(__uint_as_float(d[2 * q]), __uint_as_float(d[2 * q + 1]));
                            pk[8 * c + q] = *reinterpret_cast<const uint32_t*>(&h2);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(&sh.dfree, 0);
                const int64_t nvalid = ti.tok_end - ti.tok0 - c0;  // columns of this half with a token
                uint16_t* yb = static_cast<uint16_t*>(p.y);
#pragma unroll
                for (int q = 0; q < 64; ++q) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        if (row < p.d_out && 2 * q + e < nvalid) {
                            int64_t tk = ti.tok0 + c0 + 2 * q + e;
                            if constexpr (std::is_same<P, GroupedPrefillParams>::value) {
                                if (!bd_in(kBkPrefill, tk, p.T)) continue;
                                tk = p.perm[tk];
                            }
                            if (bd_in(kBkPrefill, tk * p.d_out + row, p.T * p.d_out))
                                yb[tk * p.d_out + row] = static_cast<uint16_t>(e ? (pk[q] >> 16) : (pk[q] & 0xFFFFu));
                        }
                    }
                }
            }
            ++j;
        }
    }

    // the pair's MMAs read both CTAs' shared and tensor memory: neither CTA
    // frees tensor memory or ends before the even CTA's issuer has seen them
    // finish (or given up)
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

// Clusters of prefill_kernel<P> resident on the current device at once with
// this shared-memory size (cached per device): the persistent grid.
template <class P>
int resident_clusters(size_t smem)
{
    static std::atomic<int> cached[kHostMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kHostMaxDevices) return 1;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    if (cudaOccupancyMaxActiveClusters(&n, prefill_kernel<P>, &cfg) != cudaSuccess || n < 1) {
        (void)cudaGetLastError();
        int sms = 0;
        (void)cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        n = sms >= 4 ? sms / 2 : 1;
    }
    cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

int row_pairs(int64_t d_out) { return static_cast<int>((d_out + 2 * BM - 1) / (2 * BM)); }

}  // namespace

bool prefill_available() { return true; }

cudaError_t launch_prefill(const PrefillArgs& a, int /*sm_count*/, cudaStream_t stream)
{
    static thread_local PrefillParams prm;
    if (!encode_tma_2d(&prm.x_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, static_cast<uint64_t>(a.d_in),
                       static_cast<uint64_t>(a.T), static_cast<uint64_t>(a.d_in) * 2, BK, BNH,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tma_2d(&prm.w_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.w_base, static_cast<uint64_t>(a.d_in),
                       static_cast<uint64_t>(a.d_out), static_cast<uint64_t>(a.d_in) * 2, BK, BM,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tma_2d(&prm.s_map, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.signs, static_cast<uint64_t>(a.d_in / 32),
                       static_cast<uint64_t>(a.d_out), static_cast<uint64_t>(a.d_in / 8), 4, BM,
                       CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    prm.alpha = a.alpha;
    prm.y = a.y;
    prm.err = a.err;
    prm.T = a.T;
    prm.d_out = a.d_out;
    prm.d_in = a.d_in;
    prm.per_row = a.per_row;
    prm.out_f32 = a.out_f32;
    prm.ntb = static_cast<int>((a.T + BN - 1) / BN);
    const size_t smem = static_cast<size_t>(kStages) * kStageBytes + 1024;
    static std::atomic<size_t> smem_set[kHostMaxDevices];
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(prefill_kernel<PrefillParams>), smem, smem_set);
    if (e != cudaSuccess) return e;
    const int64_t tiles = static_cast<int64_t>(prm.ntb) * row_pairs(a.d_out);
    const int64_t ncl = std::min<int64_t>(tiles, resident_clusters<PrefillParams>(smem));
    e = cudaSuccess;
    launch_dep(e, prefill_kernel<PrefillParams>, dim3(static_cast<unsigned>(2 * ncl)), dim3(kThreads), smem, stream, prm);
    return e != cudaSuccess ? e : cudaGetLastError();
}

namespace {

// One thread: the plan of 256-token blocks, each inside one key's segment
// [seg_off[k], seg_off[k + 1]) of the sorted tokens; entries past the plan
// are marked invalid (their CTAs leave at once).
__global__ void prefill_plan_kernel(const int32_t* __restrict__ seg_off, int V, int nblk, int4* __restrict__ plan)
{
    grid_launch_dependents();  // the gather may start launching
    grid_dependency_wait();    // the router's seg_off is visible
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    int n = 0;
    for (int k = 0; k <= V; ++k) {
        if (!bd_in(kBkPrefillPlan, k + 1, V + 2)) break;
        const int a = seg_off[k], e = seg_off[k + 1];
        for (int t = a; t < e && n < nblk; t += BN) plan[n++] = make_int4(t, e, k, 1);
    }
    for (; n < nblk; ++n) plan[n] = make_int4(0, 0, 0, 0);
}

// xs[i] = x[perm[i]]: one block per sorted row, 16-byte copies (d_in % 8 == 0).
__global__ void gather_rows_kernel(const uint16_t* __restrict__ x, const int32_t* __restrict__ perm, int64_t d_in,
                                   uint16_t* __restrict__ xs)
{
    grid_launch_dependents();  // the prefill may start launching
    grid_dependency_wait();    // the router's perm is visible (the plan kernel before this one waited for it)
    const int64_t i = blockIdx.x;  // grid = T rows
    if (!bd_in(kBkGather, perm[i], gridDim.x)) return;
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(perm[i]) * d_in);
    uint4* dst = reinterpret_cast<uint4*>(xs + i * d_in);
    for (int64_t c = threadIdx.x; c < d_in / 8; c += blockDim.x) dst[c] = src[c];
}

}  // namespace

int grouped_prefill_blocks(int64_t T, int V) { return static_cast<int>((T + BN - 1) / BN) + V + 1; }

cudaError_t launch_prefill_grouped(const GroupedPrefillArgs& a, cudaStream_t stream)
{
    if (a.V < 1 || a.V > kMaxVariants || a.T < 1) return cudaErrorInvalidValue;
    static thread_local GroupedPrefillParams prm;  // ~9 KB: kept off the stack
    if (!encode_tma_2d(&prm.x_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.xs, static_cast<uint64_t>(a.d_in),
                       static_cast<uint64_t>(a.T), static_cast<uint64_t>(a.d_in) * 2, BK, BNH,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tma_2d(&prm.w_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.w_base, static_cast<uint64_t>(a.d_in),
                       static_cast<uint64_t>(a.d_out), static_cast<uint64_t>(a.d_in) * 2, BK, BM,
                       CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    for (int v = 0; v < a.V; ++v) {
        prm.alphas[v] = a.alpha[v];
        if (!encode_tma_2d(&prm.s_maps[v], CU_TENSOR_MAP_DATA_TYPE_UINT32, a.signs[v],
                           static_cast<uint64_t>(a.d_in / 32), static_cast<uint64_t>(a.d_out),
                           static_cast<uint64_t>(a.d_in / 8), 4, BM, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    prm.s_map = prm.s_maps[0];
    prm.alpha = nullptr;
    prm.y = a.y;
    prm.err = a.err;
    prm.T = a.T;
    prm.d_out = a.d_out;
    prm.d_in = a.d_in;
    prm.per_row = a.per_row;
    prm.out_f32 = a.out_f32;
    prm.plan = a.plan;
    prm.perm = a.perm;
    const int nblk = grouped_prefill_blocks(a.T, a.V);
    prm.ntb = nblk;
    cudaError_t e = cudaSuccess;
    launch_dep(e, prefill_plan_kernel, dim3(1), dim3(32), 0, stream, a.seg_off, a.V, nblk, a.plan);
    launch_dep(e, gather_rows_kernel, dim3(static_cast<unsigned>(a.T)), dim3(256), 0, stream, a.x, a.perm, a.d_in,
               a.xs);
    if (e != cudaSuccess) return e;
    const size_t smem = static_cast<size_t>(kStages) * kStageBytes + 1024;
    static std::atomic<size_t> smem_set[kHostMaxDevices];
    e = ensure_dynamic_smem(reinterpret_cast<const void*>(prefill_kernel<GroupedPrefillParams>), smem, smem_set);
    if (e != cudaSuccess) return e;
    const int64_t tiles = static_cast<int64_t>(nblk) * row_pairs(a.d_out);
    const int64_t ncl = std::min<int64_t>(tiles, resident_clusters<GroupedPrefillParams>(smem));
    launch_dep(e, prefill_kernel<GroupedPrefillParams>, dim3(static_cast<unsigned>(2 * ncl)), dim3(kThreads), smem,
               stream, prm);
    return e != cudaSuccess ? e : cudaGetLastError();
}

BD_BOUNDS_TAKE(bounds_take_prefill)

}  // namespace bd
