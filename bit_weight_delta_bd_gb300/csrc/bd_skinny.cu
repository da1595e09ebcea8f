// Fused BitDelta linear for decode-sized token counts (T <= 64) of one variant
// (section "Sunum mimarisi" of the BitDelta post: the fused
// reconstruct+matmul kernel that reads W_base and the packed bits together).
//
//   y[t][r] = sum_j x[t][j] * W_base[r][j]  +  alpha[r] * sum_j x[t][j] * s[r][j]
//
// which is exactly x . (W_base + alpha*s)^T with no rounding of W_eff: the
// base and the sign contraction are separate bf16 MMAs (s in {-1,+1} is exact
// in bf16) that share the x operand, accumulated in fp32.
//
// Work split.  A thread-block cluster of CK CTAs covers all of d_in (CTA
// rank k takes the k-th of CK equal slices; CK depends on d_in only, never on
// d_out, so a row's arithmetic does not change when the rows are sharded) and
// is persistent: it takes the blocks of 16*kConsumers output rows numbered
// c, c + C, c + 2C, ... (C clusters resident), reducing each block's partial
// outputs (base + alpha * sign over the CTA's slice, one fma per value, so
// that one buffer holds them) through distributed shared memory, in rank
// order.  Inside the CTA one
// producer thread streams 128-column stages into a ring of shared-memory
// buffers with a handful of 2-D TMA boxes per stage, one running stage count
// across the blocks, and the consumer warps (16 rows each) run the MMAs:
//   - W_base: two boxes [block rows x 64 columns], 128-byte swizzle;
//   - x: two boxes [8*NT tokens x 64 columns], 128-byte swizzle;
//   - sign bits: one box [block rows x 4 words];
//   - full/empty mbarriers between producer and consumers, all waits bounded.
// Between two row blocks the producer first fills the ring with the next
// block's stages and then joins the block's cluster barrier, so the stream
// from device memory does not stop while the consumers reduce and store the
// finished block.  The reduction buffers are double-buffered by block parity
// (one cluster barrier per block: a CTA reuses a buffer only after its peers
// passed the next block's barrier, i.e. after they read it).
// The swizzle puts 16-byte chunk c of a 128-byte row r at chunk c ^ (r % 8),
// so the fragment loads below are bank-conflict free.
//
// Fragments.  mma.m16n8k16 wants, per thread (g = lane/4, q = lane%4), A
// elements (row g / g+8, k = 2q,2q+1,2q+8,2q+9) and B elements (token g,
// same k).  Any permutation of k applied to both operands leaves the sum
// unchanged, so logical k {2q,2q+1,2q+8,2q+9} of MMA step m is mapped to
// physical columns 16q+4m+{0,1,2,3} of a 64-column half-stage: every thread
// then reads 16 consecutive columns (two 16-byte loads) of its rows and of
// its token, and the 16 sign bits of those columns are one half-word.  Bits
// become bf16 +-1 pairs with 2 integer ops per register.
#include <cooperative_groups.h>

#include "bd_device.cuh"
#include "bd_tma.h"

namespace cg = cooperative_groups;

namespace bd {
namespace {

constexpr int kChunk = 128;        // columns per pipeline stage
constexpr int kHalfRowBytes = 128;  // one 64-column half of a staged row (one swizzle atom)
constexpr int kSignRowBytes = 16;  // 4 sign words per row per stage
constexpr int kMaxStages = 4;
constexpr int kConsumers = 4;      // 64 rows per CTA, up to three CTAs per SM
constexpr int kRows = 16 * kConsumers;
constexpr int kThreads = 32 * (kConsumers + 1);
constexpr size_t kSmemBudget = 74u * 1024u;  // three CTAs per SM

struct SkinnyParams {
    CUtensorMap sign_map;   // [d_out][d_in/32] uint32, box 4 x 64 rows
    CUtensorMap w_map;      // [d_out][d_in] bf16, box 64 x 64 rows, 128B swizzle
    CUtensorMap x_map;      // [T][d_in] bf16, box 64 x 8*NT, 128B swizzle
    const float* alpha;
    void* y;
    uint32_t* err;
    int64_t T, d_out, d_in;
    int per_row, out_f32;
    int CK, stages;
    int n_blocks;     // row blocks of kRows rows
    int n_clusters;   // clusters launched (each takes every n_clusters-th block)
};

struct SkinnyShared {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    volatile int abort;
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

// Bounded wait that also gives up as soon as another warp of the CTA has
// timed out (sets the CTA-wide abort flag and the error word on timeout).
__device__ __forceinline__ bool wait_or_abort(SkinnyShared& sh, uint64_t* bar, uint32_t parity, uint32_t* err)
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

template <int NT>
__global__ void __launch_bounds__(kThreads, 2) skinny_kernel(const __grid_constant__ SkinnyParams p)
{
    constexpr int Tpad = 8 * NT;

    extern __shared__ uint8_t dyn_raw[];
    __shared__ SkinnyShared sh;
    // 1024-byte aligned base for the stage ring (the allocation has the slack)
    uint8_t* dyn = dyn_raw + ((1024u - (smem_u32(dyn_raw) & 1023u)) & 1023u);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, q = lane & 3;
    const int T = static_cast<int>(p.T);
    const int64_t d_in = p.d_in;
    const int CK = p.CK;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const int cl = static_cast<int>(blockIdx.x) / CK;  // cluster index

    grid_launch_dependents();  // a kernel launched after this one with programmatic dependent launch may start
    if (tid == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], kConsumers);
        }
        sh.abort = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    grid_dependency_wait();  // the previous kernel's results (x, the signs, alpha) are visible

    // ---------------------------------------------------------------- pipeline
    // stage layout: [W half 0 | W half 1 | x half 0 | x half 1 | sign tile], 1024-byte aligned;
    // after the ring: two reduction buffers of the CTA's partial outputs
    // base + alpha * sign, [kRows][Tpad] fp32 each
    const int stages = p.stages;
    constexpr int kWHalf = kRows * kHalfRowBytes;
    constexpr int kXHalf = Tpad * kHalfRowBytes;
    constexpr int kSignOff = 2 * kWHalf + 2 * kXHalf;
    constexpr int kSignTile = kRows * kSignRowBytes;
    constexpr int kStageBytes = (kSignOff + kSignTile + 1023) & ~1023;
    constexpr int kRedFloats = kRows * Tpad;  // one buffer
    float* red_all = reinterpret_cast<float*>(dyn + static_cast<size_t>(stages) * kStageBytes);
    const int nc = static_cast<int>(d_in / kChunk);
    const int c_begin = static_cast<int>(static_cast<int64_t>(rank) * nc / CK);
    const int c_end = static_cast<int>(static_cast<int64_t>(rank + 1) * nc / CK);
    const int n_chunks = c_end - c_begin;
    const int n_mine = cl < p.n_blocks ? (p.n_blocks - 1 - cl) / p.n_clusters + 1 : 0;  // blocks of this cluster
    const uint32_t tx = static_cast<uint32_t>(2 * kWHalf + 2 * kXHalf + kSignTile);

    // Producer: stage k (running count over this cluster's blocks) is chunk
    // k % n_chunks of the block k / n_chunks.  Issues stages up to `target`;
    // waits only for ring slots whose previous stage precedes `target` - the
    // stages slots back, which the consumers release without waiting for
    // anything the producer does later.
    int pk = 0;
    auto produce_until = [&](int target) {
        for (; pk < target; ++pk) {
            const int s = pk % stages;
            if (pk >= stages &&
                !__all_sync(0xffffffffu, wait_or_abort(sh, &sh.empty[s], static_cast<uint32_t>(pk / stages - 1) & 1u,
                                                       p.err)))
                return false;
            uint8_t* st = dyn + static_cast<size_t>(s) * kStageBytes;
            const int col = (c_begin + pk % n_chunks) * kChunk;
            const int rb = (cl + (pk / n_chunks) * p.n_clusters) * kRows;
            if (lane == 0) {
                mbar_arrive_expect_tx(&sh.full[s], tx);
                tma_load_2d(st, &p.w_map, col, rb, &sh.full[s]);
                tma_load_2d(st + kWHalf, &p.w_map, col + 64, rb, &sh.full[s]);
                tma_load_2d(st + 2 * kWHalf, &p.x_map, col, 0, &sh.full[s]);
                tma_load_2d(st + 2 * kWHalf + kXHalf, &p.x_map, col + 64, 0, &sh.full[s]);
                tma_load_2d(st + kSignOff, &p.sign_map, col / 32, rb, &sh.full[s]);
            }
            __syncwarp();
        }
        return true;
    };
    bool p_ok = true;
    const int rl0 = 16 * warp + g;  // consumer rows rl0 and rl0 + 8 (both = g mod 8)
    const int c0 = ((2 * q) ^ g) << 4, c1 = ((2 * q + 1) ^ g) << 4;  // swizzled chunk offsets

    for (int u = 0; u < n_mine; ++u) {
        const int64_t row0 = static_cast<int64_t>(cl + u * p.n_clusters) * kRows;
        const int valid_rows = static_cast<int>(p.d_out - row0 < kRows ? p.d_out - row0 : kRows);
        float* red = red_all + (u & 1) * kRedFloats;
        if (warp == kConsumers) {
            // ------------------------------------------------------------ producer warp
            // the rest of this block, then the first `stages` stages of the next one (their slots
            // held this block's last stages), before the block's cluster barrier
            int target = (u + 1) * n_chunks;
            if (u + 1 < n_mine) target += n_chunks < stages ? n_chunks : stages;
            if (p_ok && !sh.abort) p_ok = produce_until(target);
        } else {
            // ------------------------------------------------------------ consumer warps
            float accb[NT][4], accs[NT][4];
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) accb[j][e] = accs[j][e] = 0.0f;
            for (int i = 0; i < n_chunks; ++i) {
                const int kst = u * n_chunks + i;
                const int s = kst % stages;
                if (!__all_sync(0xffffffffu, wait_or_abort(sh, &sh.full[s], static_cast<uint32_t>(kst / stages) & 1u,
                                                           p.err)))
                    break;
                const uint8_t* st = dyn + static_cast<size_t>(s) * kStageBytes;
                const uint32_t* sgn = reinterpret_cast<const uint32_t*>(st + kSignOff);
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
                    const int sign_word = 2 * h + (q >> 1);
                    const uint32_t sign_shift = 16u * (q & 1);
                    uint32_t S0[8], S1[8];
                    expand_signs((sgn[rl0 * 4 + sign_word] >> sign_shift) & 0xFFFFu, S0);
                    expand_signs((sgn[(rl0 + 8) * 4 + sign_word] >> sign_shift) & 0xFFFFu, S1);
#pragma unroll
                    for (int j = 0; j < NT; ++j) {
                        const uint8_t* xr = xst + (8 * j + g) * kHalfRowBytes;
                        const uint4 xa = *reinterpret_cast<const uint4*>(xr + c0);
                        const uint4 xb = *reinterpret_cast<const uint4*>(xr + c1);
                        mma4(accb[j], W0, W1, xa, xb);
                        mma4(accs[j], S0, S1, xa, xb);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.empty[s]);
            }
            // this block's partial outputs base + alpha * sign (alpha of the row) into
            // this CTA's reduction buffer of the block's parity
            float a0 = 0.0f, a1 = 0.0f;
            if (rl0 < valid_rows && bd_in(kBkSkinny, p.per_row ? row0 + rl0 : 0, p.per_row ? p.d_out : 1))
                a0 = p.alpha[p.per_row ? row0 + rl0 : 0];
            if (rl0 + 8 < valid_rows && bd_in(kBkSkinny, p.per_row ? row0 + rl0 + 8 : 0, p.per_row ? p.d_out : 1))
                a1 = p.alpha[p.per_row ? row0 + rl0 + 8 : 0];
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                const int pos = 8 * j + 2 * q;
                red[rl0 * Tpad + pos] = fmaf(a0, accs[j][0], accb[j][0]);
                red[rl0 * Tpad + pos + 1] = fmaf(a0, accs[j][1], accb[j][1]);
                red[(rl0 + 8) * Tpad + pos] = fmaf(a1, accs[j][2], accb[j][2]);
                red[(rl0 + 8) * Tpad + pos + 1] = fmaf(a1, accs[j][3], accb[j][3]);
            }
        }
        // ---------------------------------------------------------------- cluster K reduction of block u
        cluster.sync();
        if (warp < kConsumers) {
            const int r_lo = rank * kRows / CK, r_hi = (rank + 1) * kRows / CK;
            const int nr = r_hi - r_lo;
            for (int o = tid; o < nr * T; o += 32 * kConsumers) {
                const int t = o / nr, r = r_lo + o % nr;
                if (r >= valid_rows) continue;
                float y = cluster.map_shared_rank(red, 0)[r * Tpad + t];
                for (int k = 1; k < CK; ++k) y += cluster.map_shared_rank(red, k)[r * Tpad + t];
                const int64_t row = row0 + r;
                const int64_t idx = static_cast<int64_t>(t) * p.d_out + row;
                if (!bd_in(kBkSkinny, idx, p.T * p.d_out)) continue;
                if (p.out_f32)
                    static_cast<float*>(p.y)[idx] = y;
                else
                    static_cast<__nv_bfloat16*>(p.y)[idx] = __float2bfloat16_rn(y);
            }
        }
    }
    if (warp == kConsumers) {
        // every issued stage must have landed before the CTA exits
        for (int i = (pk > stages ? pk - stages : 0); i < pk; ++i) {
            const int s = i % stages;
            const uint32_t par = static_cast<uint32_t>(i / stages) & 1u;
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(&sh.full[s], par) && global_timer_ns() - t0 < kWaitLimitNs) {
            }
        }
    }
    cluster.sync();  // peers may still read this CTA's last reduction buffer until here
}

template <int NT>
cudaError_t launch_nt(SkinnyParams& prm, size_t smem, cudaStream_t stream)
{
    auto kern = skinny_kernel<NT>;
    static std::atomic<size_t> smem_set[kHostMaxDevices];
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem, smem_set);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(prm.CK);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // programmatic dependent launch: the launch overlaps the end of the kernel before it
    // (the kernel waits for that kernel's results before its first global access)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // persistent clusters: as many as can be resident at once (cached per device,
    // cluster size and shared-memory size), each taking every n-th row block
    int dev = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if (dev < 0 || dev >= kHostMaxDevices) return cudaErrorInvalidDevice;
    static std::atomic<int> resident[kHostMaxDevices][4];
    static std::atomic<size_t> resident_smem[kHostMaxDevices][4];
    const int ci = prm.CK == 1 ? 0 : prm.CK == 2 ? 1 : prm.CK == 4 ? 2 : 3;
    int n_res = resident[dev][ci].load(std::memory_order_relaxed);
    if (n_res <= 0 || resident_smem[dev][ci].load(std::memory_order_relaxed) != smem) {
        cfg.gridDim = dim3(static_cast<unsigned>(prm.CK));
        if ((e = cudaOccupancyMaxActiveClusters(&n_res, kern, &cfg)) != cudaSuccess) return e;
        if (n_res < 1) n_res = 1;
        resident[dev][ci].store(n_res, std::memory_order_relaxed);
        resident_smem[dev][ci].store(smem, std::memory_order_relaxed);
    }
    prm.n_clusters = prm.n_blocks < n_res ? prm.n_blocks : n_res;
    cfg.gridDim = dim3(static_cast<unsigned>(prm.n_clusters * prm.CK));
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, prm);
}

int tiles_for(int T) { return T <= 8 ? 1 : T <= 16 ? 2 : T <= 32 ? 4 : 8; }

size_t stage_bytes_for(int nt)
{
    const size_t raw = 2u * kRows * kHalfRowBytes + 2u * (8u * nt) * kHalfRowBytes + kRows * kSignRowBytes;
    return (raw + 1023u) & ~static_cast<size_t>(1023u);
}

}  // namespace

cudaError_t launch_skinny(const SkinnyArgs& a, cudaStream_t stream)
{
    const int nc = static_cast<int>(a.d_in / kChunk);
    const int T = static_cast<int>(a.T);
    if (T < 1 || T > kSkinnyMaxTokens) return cudaErrorInvalidValue;
    const int nt = tiles_for(T);

    static thread_local SkinnyParams prm;
    prm.alpha = a.alpha;
    prm.y = a.y;
    prm.err = a.err;
    prm.T = a.T;
    prm.d_out = a.d_out;
    prm.d_in = a.d_in;
    prm.per_row = a.per_row;
    prm.out_f32 = a.out_f32;
    if (!encode_tma_2d(&prm.sign_map, CU_TENSOR_MAP_DATA_TYPE_UINT32, a.signs, static_cast<uint64_t>(a.d_in / 32),
                       static_cast<uint64_t>(a.d_out), static_cast<uint64_t>(a.d_in / 8), 4,
                       static_cast<uint32_t>(kRows), CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_tma_2d(&prm.w_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.w_base, static_cast<uint64_t>(a.d_in),
                       static_cast<uint64_t>(a.d_out), static_cast<uint64_t>(a.d_in) * 2, 64,
                       static_cast<uint32_t>(kRows), CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tma_2d(&prm.x_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.x, static_cast<uint64_t>(a.d_in),
                       static_cast<uint64_t>(a.T), static_cast<uint64_t>(a.d_in) * 2, 64,
                       static_cast<uint32_t>(8 * nt), CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    // K slices per cluster: a function of d_in only (one per 4096 columns, at
    // most 4; measured best on GB300 for d_in = 8192).
    int ck = nc / 32;
    ck = ck < 1 ? 1 : ck > 4 ? 4 : ck;
    prm.CK = ck;
    const size_t stage_bytes = stage_bytes_for(nt);
    const size_t red = 2u * (kRows * (8u * nt) * sizeof(float));  // two buffers of partial outputs
    int stages = kMaxStages;
    while (stages > 2 && stages * stage_bytes + red + 1024 > kSmemBudget) --stages;
    prm.stages = stages;
    prm.n_blocks = static_cast<int>((a.d_out + kRows - 1) / kRows);
    const size_t smem = stages * stage_bytes + red + 1024;
    if (smem > 227u * 1024u) return cudaErrorInvalidConfiguration;
    switch (nt) {
        case 1: return launch_nt<1>(prm, smem, stream);
        case 2: return launch_nt<2>(prm, smem, stream);
        case 4: return launch_nt<4>(prm, smem, stream);
        default: return launch_nt<8>(prm, smem, stream);
    }
}

BD_BOUNDS_TAKE(bounds_take_skinny)

}  // namespace bd
