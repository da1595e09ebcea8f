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
//   B B^T = U_B Lambda U_B^T   (l x l symmetric eigenproblem: tridiagonalisation,
//                               bisection, inverse iteration)
//   tau = (Q U_r) (U_r^T B)    (U_r: the r leading eigenvectors)
// which is U_r S_r V_r^T of the rank-l approximation Q Q^T Delta.  Every pass
// over Delta reads W_i and W_base (bf16) and forms Delta in fp32 on the fly.
// Orthonormalisation is CholeskyQR: the Gram matrix is accumulated and
// factored in float-float (one CTA per checkpoint), and Y <- Y R^-1 applied by
// forward substitution (twice, CholeskyQR2, for the final basis); directions
// whose pivot falls below 1e-12 of the largest are dropped (rank-deficient
// sketches).
// The merge is one pass: W_base + (1/k) [L_1 .. L_k][R_1 .. R_k]^T with
// L_i = Q_i U_r, R_i = B_i^T U_r, rounded once to the output type.
//
// The products with Delta (l <= 32) and the merge run on the tcgen05 tensor
// cores on exact three-piece bf16 splits of their fp32 operands, with fp32
// accumulation; wider sketches (l <= 64) use fp32 CUDA-core products.  The
// Gram matrices and Cholesky factors are float-float on the fp32 units, the
// eigenproblem fp32.  Up to kMaxBatch checkpoints go through every step
// together (one launch per step, the checkpoint in a grid dimension).  No
// kernel waits on another CTA; the passes are stream-ordered launches, each
// allowed to start launching while the kernel before it finishes
// (programmatic dependent launch).
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include <atomic>

#include "bd_device.cuh"
#include "bd_tcgen05.cuh"
#include "bd_tma.h"

namespace bd {
namespace {

constexpr int kMaxL = 64;        // sketch width l (columns of Y, Q, B^T)
constexpr int kGramParts = 304;   // CTAs of one Gram pass (fixed-order float-float partials)
constexpr int kGramThreads = 1024;
constexpr int kSlices = 16;       // partial results of one product pass (over the checkpoints of a batch)
constexpr int kMaxBatch = 8;      // checkpoints that go through the steps together

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// acc += (a, a) * m on a pair of fp32 lanes: one paired FMA instruction
// (two independent fma.rn, the same results as two fmaf calls) issues two
// FMAs in one instruction slot.
__device__ __forceinline__ void ffma2(float2& acc, float a, float mx, float my)
{
    uint64_t ac, aa, mm;
    asm("mov.b64 %0, {%1, %2};" : "=l"(ac) : "f"(acc.x), "f"(acc.y));
    asm("mov.b64 %0, {%1, %1};" : "=l"(aa) : "f"(a));
    asm("mov.b64 %0, {%1, %2};" : "=l"(mm) : "f"(mx), "f"(my));
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(ac) : "l"(aa), "l"(mm));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(acc.x), "=f"(acc.y) : "l"(ac));
}

// The two products with Delta on the CUDA cores (fp32 FMA).  Products
// accurate to fp32 are needed (the subspace of the final basis moves with
// the products' relative error, amplified by the spectral spread): a bf16
// tensor-core form accurate to fp32 takes six bf16 MMAs per 256 products
// (three pieces of each operand), which at GB300's legacy MMA rate equals its
// fp32 FMA rate, and tcgen05 MMAs with N = l <= 64 are bound by their issue
// rate.  Both products stream the same tiles through one kernel:
//   - a producer warp issues, per 64 x 64 tile of Delta's index space, TMA
//     loads of W_i and W_base (128-byte swizzle) and a bulk copy of the 64
//     rows of the small operand that the tile meets (Omega / Z for the
//     sketch: rows = Delta's columns; Q for the transpose product: rows =
//     Delta's rows) into a ring of prod_stages<L4>() stages;
//   - eight FMA warps, as four pairs that split each stage 4 ways along its
//     reduction index; every lane owns RPL rows (sketch) or 2 columns
//     (transpose product) of Delta, the two warps of a pair one half each of
//     the l output columns; Delta values come from the swizzled tile
//     (conflict-free), the small operand as broadcasts (every lane of a warp
//     reads the same row).
// The warps' partial sums are added in warp order at the end and written as
// one of gridDim.y partial results (summed in slice order by the next Gram
// pass, gram_kernel with nslice > 1).

constexpr int kPWarps = 8;       // FMA warps per product CTA
constexpr int kPTile = 64;       // Delta tile per stage: 64 x 64
// ring stages and resident CTAs per SM: l <= 32 takes three CTAs of three
// stages (six FMA warps per scheduler), l <= 64 two CTAs of four stages
template <int L4>
constexpr int prod_stages() { return L4 <= 8 ? 3 : 4; }
template <int L4>
constexpr int prod_ctas() { return L4 <= 8 ? 3 : 2; }
constexpr int kPThreads = 32 * (kPWarps + 1);

struct ProdParams {
    CUtensorMap b_map;               // W_base [d_out][d_in] bf16, box 64 x 64, 128-byte swizzle
    CUtensorMap w_map[kMaxBatch];    // W_i of checkpoint blockIdx.z, same
    CUtensorMap s_map[kMaxBatch];    // its small operand, fp32 [rows][l], box 4 L4 x 64 (zero past l and
                                     // past the rows): Omega / Z [d_in][l] (sketch) or Q [d_out][l]
    float* part;         // [gridDim.z][gridDim.y][out rows][l]
    uint32_t* err;
    int64_t d_out, d_in;
    int l;
    int64_t k_per;       // reduction indices per slice (a multiple of 64)
};

// Checkpoint z = blockIdx.z of the batch:
// MODE 0: part[z][s][row][c] = sum over slice s of j of Delta[row][j] small[j][c]
//         (CTA: 32 RPL rows of Delta; lane: rows lane + 32 h, h < RPL; warp
//         pair cg = warp / 2 takes columns 16 cg .. 16 cg + 15 of each tile)
// MODE 1: part[z][s][j][c] = sum over slice s of rows of Delta[row][j] small[row][c]
//         (CTA: 64 columns of Delta; lane: columns 2 lane, 2 lane + 1; warp
//         pair rg = warp / 2 takes rows 16 rg .. 16 rg + 15 of each tile)
// The two warps of a pair hold the two halves of the l output columns
// (LH = L4 / 2 float4 each), so that a lane keeps 2 x 4 LH accumulators.
template <int MODE, int L4>
__global__ void __launch_bounds__(kPThreads, prod_ctas<L4>()) dprod_kernel(const __grid_constant__ ProdParams p)
{
    grid_launch_dependents();  // the next kernel of the merge may start launching
    grid_dependency_wait();    // the previous kernel's results are visible
    constexpr int LH = L4 / 2;                                // float4 output columns per warp
    constexpr int RPL = MODE == 0 ? (L4 <= 8 ? 2 : 1) : 2;  // Delta rows (columns) per lane
    constexpr int kOut = MODE == 0 ? 32 * RPL : kPTile;      // output rows of one CTA
    constexpr int kBoxRows = MODE == 0 ? 32 * RPL : kPTile;  // Delta rows per tile
    constexpr int kWTile = kBoxRows * 128;                  // one bf16 tile: kBoxRows x 64
    constexpr int kSTile = kPTile * 4 * L4 * 4;              // 64 rows of the small operand (fp32, 4 L4 wide)
    constexpr int kStage = 2 * kWTile + kSTile;
    constexpr int kPStages = prod_stages<L4>();
    extern __shared__ uint8_t dyn_raw[];
    __shared__ uint64_t full[kPStages], empty[kPStages];
    __shared__ volatile int abort;
    uint8_t* ring = dyn_raw + ((1024u - (smem_u32(dyn_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int l = p.l;
    const int grp = warp >> 1, half = warp & 1;
    const int c0 = half * LH;  // first float4 output column of this warp
    const int64_t o0 = static_cast<int64_t>(blockIdx.x) * kOut;  // first output row of this CTA
    const int64_t kb = static_cast<int64_t>(blockIdx.y) * p.k_per;
    const int64_t klen = MODE == 0 ? p.d_in : p.d_out;
    const int64_t ke = kb + p.k_per < klen ? kb + p.k_per : klen;
    const int nt = static_cast<int>((ke - kb + kPTile - 1) / kPTile);  // tiles of this CTA
    if (tid == 0) {
        for (int s = 0; s < kPStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kPWarps);
        }
        abort = 0;
        fence_mbarrier_init();
    }
    __syncthreads();
    auto wait = [&](uint64_t* bar, uint32_t par) {
        if (mbar_try_wait(bar, par)) return true;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(bar, par)) {
            if (abort) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                abort = 1;
                raise_error(p.err, kErrTimeout);
                return false;
            }
        }
        return true;
    };
    float2 acc[RPL][2 * LH];
#pragma unroll
    for (int h = 0; h < RPL; ++h)
#pragma unroll
        for (int c = 0; c < 2 * LH; ++c) acc[h][c] = make_float2(0.0f, 0.0f);
    // acc += d[h] * small row (this warp's float4 columns c0 .. c0 + LH; the
    // staged rows are 4 L4 floats, zero past l)
    auto fma_row = [&](const float* row, const float (&d)[RPL]) {
        const float4* r4 = reinterpret_cast<const float4*>(row) + c0;
#pragma unroll
        for (int c = 0; c < LH; ++c) {
            const float4 m = r4[c];
#pragma unroll
            for (int h = 0; h < RPL; ++h) {
                ffma2(acc[h][2 * c], d[h], m.x, m.y);
                ffma2(acc[h][2 * c + 1], d[h], m.z, m.w);
            }
        }
    };

    if (warp == kPWarps) {
        // ---------------------------------------------------------------- producer
        int t = 0;
        for (; t < nt; ++t) {
            const int s = t % kPStages;
            if (t >= kPStages && !__all_sync(0xffffffffu, wait(&empty[s], static_cast<uint32_t>(t / kPStages - 1) & 1u)))
                break;
            uint8_t* st = ring + static_cast<size_t>(s) * kStage;
            const int64_t k0 = kb + static_cast<int64_t>(t) * kPTile;  // first reduction index of the tile
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(kStage));
                const int cx = static_cast<int>(MODE == 0 ? k0 : o0), cy = static_cast<int>(MODE == 0 ? o0 : k0);
                tma_load_2d(st, &p.w_map[blockIdx.z], cx, cy, &full[s]);
                tma_load_2d(st + kWTile, &p.b_map, cx, cy, &full[s]);
                tma_load_2d(st + 2 * kWTile, &p.s_map[blockIdx.z], 0, static_cast<int>(k0), &full[s]);
            }
            __syncwarp();
        }
        for (int i = (t > kPStages ? t - kPStages : 0); i < t; ++i) {  // every issued copy lands before exit
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(&full[i % kPStages], static_cast<uint32_t>(i / kPStages) & 1u) &&
                   global_timer_ns() - t0 < kWaitLimitNs) {
            }
        }
    } else {
        // ---------------------------------------------------------------- FMA warps
        for (int t = 0; t < nt; ++t) {
            const int s = t % kPStages;
            if (!__all_sync(0xffffffffu, wait(&full[s], static_cast<uint32_t>(t / kPStages) & 1u))) break;
            const uint8_t* st = ring + static_cast<size_t>(s) * kStage;
            const int64_t k0 = kb + static_cast<int64_t>(t) * kPTile;
            const int kn = static_cast<int>(ke - k0 < kPTile ? ke - k0 : kPTile);
            const float* sm = reinterpret_cast<const float*>(st + 2 * kWTile);  // [64][4 L4]
            if (MODE == 0) {
                // pair grp: columns 16 grp .. 16 grp + 15 of the tile (16-byte chunks 2 grp, 2 grp + 1)
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    const int chunk = 2 * grp + ch, jj0 = 8 * chunk;
                    if (jj0 >= kn) break;
                    float d[RPL][8];
#pragma unroll
                    for (int h = 0; h < RPL; ++h) {
                        const int r = lane + 32 * h;
                        const int off = r * 128 + ((chunk ^ (r & 7)) << 4);
                        const uint4 a = *reinterpret_cast<const uint4*>(st + off);
                        const uint4 b = *reinterpret_cast<const uint4*>(st + kWTile + off);
                        const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            d[h][2 * q] = bf16_bits_to_float(av[q] & 0xFFFFu) - bf16_bits_to_float(bv[q] & 0xFFFFu);
                            d[h][2 * q + 1] = bf16_bits_to_float(av[q] >> 16) - bf16_bits_to_float(bv[q] >> 16);
                        }
                    }
                    const int qn = kn - jj0 < 8 ? kn - jj0 : 8;
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        if (q >= qn) break;
                        float dq[RPL];
#pragma unroll
                        for (int h = 0; h < RPL; ++h) dq[h] = d[h][q];
                        fma_row(sm + (jj0 + q) * 4 * L4, dq);
                    }
                }
            } else {
                // pair grp: rows 16 grp .. 16 grp + 15 of the tile; lane: columns 2 lane, 2 lane + 1
#pragma unroll 4
                for (int q = 0; q < 16; ++q) {
                    const int r = 16 * grp + q;
                    if (r >= kn) break;
                    const int off = r * 128 + (((lane >> 2) ^ (r & 7)) << 4) + ((lane & 3) << 2);
                    const uint32_t a = *reinterpret_cast<const uint32_t*>(st + off);
                    const uint32_t b = *reinterpret_cast<const uint32_t*>(st + kWTile + off);
                    float d[RPL];
                    d[0] = bf16_bits_to_float(a & 0xFFFFu) - bf16_bits_to_float(b & 0xFFFFu);
                    d[RPL - 1] = bf16_bits_to_float(a >> 16) - bf16_bits_to_float(b >> 16);
                    fma_row(sm + r * 4 * L4, d);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
    }
    // ---------------------------------------------------------------- the warps' partials, in warp order
    __syncthreads();  // the ring is drained: it becomes the reduction buffer [kOut][4 L4 + 1]
    float* red = reinterpret_cast<float*>(ring);
    constexpr int kRS = 4 * L4 + 1;
    for (int wv = 0; wv < kPWarps; ++wv) {
        if (warp == wv) {
#pragma unroll
            for (int h = 0; h < RPL; ++h) {
                const int row = MODE == 0 ? lane + 32 * h : 2 * lane + h;
#pragma unroll
                for (int c = 0; c < 2 * LH; ++c) {
                    const float v[2] = {acc[h][c].x, acc[h][c].y};
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        float* dst = &red[row * kRS + 4 * c0 + 2 * c + e];
                        *dst = wv < 2 ? v[e] : *dst + v[e];  // warps 0 and 1 start the two halves
                    }
                }
            }
        }
        __syncthreads();
    }
    const int64_t nrows = MODE == 0 ? p.d_out : p.d_in;
    float* out = p.part + (static_cast<int64_t>(blockIdx.z) * gridDim.y + blockIdx.y) * nrows * l;
    for (int e = tid; e < kOut * l; e += kPThreads) {
        const int rr = e / l, c = e - rr * l;
        if (o0 + rr < nrows &&
            bd_in(kBkMsProd, (static_cast<int64_t>(blockIdx.z) * gridDim.y + blockIdx.y) * nrows * l + (o0 + rr) * l + c,
                  static_cast<int64_t>(gridDim.z) * gridDim.y * nrows * l))
            out[(o0 + rr) * l + c] = red[rr * kRS + c];
    }
}

template <int MODE, int L4>
size_t dprod_smem()
{
    constexpr int RPL = MODE == 0 ? (L4 <= 8 ? 2 : 1) : 2;
    constexpr int kBoxRows = MODE == 0 ? 32 * RPL : kPTile;
    const size_t stage = 2u * kBoxRows * 128 + static_cast<size_t>(kPTile) * 4 * L4 * 4;
    const size_t red = static_cast<size_t>(MODE == 0 ? 32 * RPL : kPTile) * (4 * L4 + 1) * 4;
    constexpr int kPStages = prod_stages<L4>();
    return (kPStages * stage > red ? kPStages * stage : red) + 1024;
}

// ---------------------------------------------------------------- tensor-core products (l <= 32)
// The same two products on the tcgen05 tensor cores with exact splits: an
// fp32 value v is v1 + v2 + v3 with v1 = v with the low 16 bits of its
// encoding cleared, v2 the same of v - v1 and v3 = v - v1 - v2 (each
// subtraction exact, each piece a bf16 value), so that Delta S is the sum of
// the products of pieces, each bf16 x bf16 product exact and the sums in
// fp32 in the tensor core; the six products of pieces a, b with a + b <= 2
// are kept (the other three are below the fp32 rounding of the sums).
//   A = a piece of Delta (M = 128 rows of Delta for the sketch, 128 columns
//       for the transpose product; K = its other index), formed by the
//       piece warps from the W_i and W_base tiles and written to tensor
//       memory (one lane per row of A, a bf16 pair per column);
//   B = the pieces of the small operand stacked along N: row 32 b + c =
//       piece b of column c (N = 96, rows c >= l zero), K-major in shared
//       memory (split_small_kernel writes them, a TMA box brings 64 K);
//   D[m][32 b + c] (+)= sum over the k-step of A_a B_b^T, b < 3 - a, for the
//       three pieces a of Delta (MMAs of M = 128, N = 96, 64 and 32, K = 16
//       per k-step) in tensor memory; the result is
//       D[m][c] + D[m][32 + c] + D[m][64 + c].
// A stage holds only the W_i and W_base tiles and the B tile (44 KB), so four
// stages keep four tiles of Delta in flight per SM.  The W tiles of a stage
// are free as soon as the piece warps hold their values (wfree), the B tile
// when the stage's MMAs finish (empty).  The CTAs are persistent, one per
// SM: CTA c takes the units (row block, checkpoint, slice of the reduction
// dimension) c, c + gridDim.x, ... and its ring runs on across them (a new
// CTA per unit spent ~4 us per unit on its ramp and on the switch).  The
// checkpoint varies fastest along the units, so the CTAs that read the same
// W_base tiles run side by side and share them in L2.  Warp 0 issues the
// TMA loads, warp 1 allocates tensor memory and issues the MMAs, warps 2..9
// form the pieces (lane quarter warp % 4, K half (warp - 2) / 4), warps
// 10..13 read each unit's accumulator, one row per thread (the next unit's
// MMAs wait for those loads).
constexpr int kTM = 128;                     // MMA M: Delta rows (MODE 0) or columns (MODE 1) of a CTA
constexpr int kTK = 64;                      // reduction indices per stage
constexpr int kTNB = 96;                     // MMA N: three pieces x 32 columns of the small operand
constexpr int kTStages = 4;
constexpr int kTWTile = kTM * kTK * 2;       // one bf16 tile of W: 16 KB
constexpr int kTBTile = kTNB * kTK * 2;      // the B tile: 12 KB
constexpr int kTStage = 2 * kTWTile + kTBTile;
constexpr int kTConvWarps = 8;
constexpr int kTEpiWarp = 2 + kTConvWarps;         // warps kTEpiWarp .. + 3 drain the accumulator
constexpr int kTThreads = 32 * (2 + kTConvWarps + 4);
constexpr uint32_t kTTmemCols = 512;
constexpr uint32_t kTDCol = 0;                // D: 96 columns
constexpr uint32_t kTACol = 128;              // A ring: 3 pieces x 32 columns per stage
static_assert(kTACol + 3 * 32 * kTStages <= kTTmemCols, "tensor-memory columns");
static_assert(kTStage % 1024 == 0, "1024-byte aligned stages");

struct TProdParams {
    CUtensorMap b_map;             // W_base [d_out][d_in] bf16, box 64 x 128 (MODE 0) or 64 x 64 (MODE 1), 128-byte swizzle
    CUtensorMap w_map[kMaxBatch];  // W_i of checkpoint blockIdx.x % nz, same
    CUtensorMap s_map[kMaxBatch];  // its split small operand [128][Kp] bf16, box 64 x 96, 128-byte swizzle
    float* part;                   // [checkpoints][ns][out rows][l]
    uint32_t* err;                 // the error word: a wait that timed out sets kErrTimeout
    int64_t d_out, d_in;
    int l;
    int nz;                        // checkpoints of the batch
    int ns;                        // slices of the reduction dimension
    int tiles;                     // row blocks x checkpoints
    int64_t k_per;                 // reduction indices per slice (a multiple of 64)
};

// The three pieces of the two Delta values of a bf16 pair (W_i word wi,
// W_base word wb), each packed as a bf16 pair.
__device__ __forceinline__ void split_pair(uint32_t wi, uint32_t wb, uint32_t& o1, uint32_t& o2, uint32_t& o3)
{
    const float dl = __fsub_rn(__uint_as_float(wi << 16), __uint_as_float(wb << 16));
    const float dh = __fsub_rn(__uint_as_float(wi & 0xFFFF0000u), __uint_as_float(wb & 0xFFFF0000u));
    const uint32_t l1 = __float_as_uint(dl) & 0xFFFF0000u, h1 = __float_as_uint(dh) & 0xFFFF0000u;
    const float rl = __fsub_rn(dl, __uint_as_float(l1)), rh = __fsub_rn(dh, __uint_as_float(h1));
    const uint32_t l2 = __float_as_uint(rl) & 0xFFFF0000u, h2 = __float_as_uint(rh) & 0xFFFF0000u;
    const float sl = __fsub_rn(rl, __uint_as_float(l2)), sh = __fsub_rn(rh, __uint_as_float(h2));
    o1 = __byte_perm(l1, h1, 0x7632);
    o2 = __byte_perm(l2, h2, 0x7632);
    o3 = __byte_perm(__float_as_uint(sl), __float_as_uint(sh), 0x7632);
}

// Sp[z][32 b + c][k] = piece b of S_z[k][c] (c < l, b < 3, k < K), zero for
// c >= l and in the columns K .. Kp - 1 (rows of Kp elements, Kp = K rounded
// up to 64; rows 96 .. 127 are not read); S_z = S + z zstride ([K][l] fp32,
// l a multiple of 4), z = blockIdx.y.  Thread: 8 consecutive k (lane: k
// group 32 blockIdx.x + lane) and 4 columns (warp w: columns 4 w .. 4 w + 3),
// one 16-byte store per row; 256 threads.
__global__ void __launch_bounds__(256) split_small_kernel(const float* __restrict__ S, int64_t zstride, int64_t K,
                                                          int64_t Kp, int l, uint16_t* __restrict__ Sp)
{
    grid_launch_dependents();  // the next kernel of the merge may start launching
    grid_dependency_wait();    // the previous kernel's results are visible
    const int64_t g = static_cast<int64_t>(blockIdx.x) * 32 + (threadIdx.x & 31);
    if (8 * g >= Kp) return;
    const float* src = S + blockIdx.y * zstride;
    uint16_t* o = Sp + static_cast<int64_t>(blockIdx.y) * 128 * Kp + 8 * g;
    {
        const int c0 = 4 * static_cast<int>(threadIdx.x >> 5);
        float v[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int64_t k = 8 * g + j;
            const float4 f = (k < K && c0 < l &&
                              bd_in_range(kBkMsSplit, blockIdx.y * zstride + k * l + c0, 4,
                                          (gridDim.y - 1) * zstride + K * l))
                                 ? *reinterpret_cast<const float4*>(src + k * l + c0)
                                               : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            v[j][0] = f.x;
            v[j][1] = f.y;
            v[j][2] = f.z;
            v[j][3] = f.w;
        }
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            uint32_t w1[4], w2[4], w3[4];
#pragma unroll
            for (int j = 0; j < 8; j += 2) {
                uint32_t p1[2], p2[2], p3[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float x = v[j + e][cc];
                    const uint32_t b1 = __float_as_uint(x) & 0xFFFF0000u;
                    const float r1 = __fsub_rn(x, __uint_as_float(b1));
                    const uint32_t b2 = __float_as_uint(r1) & 0xFFFF0000u;
                    const float r2 = __fsub_rn(r1, __uint_as_float(b2));
                    p1[e] = b1;
                    p2[e] = b2;
                    p3[e] = __float_as_uint(r2);
                }
                w1[j / 2] = __byte_perm(p1[0], p1[1], 0x7632);
                w2[j / 2] = __byte_perm(p2[0], p2[1], 0x7632);
                w3[j / 2] = __byte_perm(p3[0], p3[1], 0x7632);
            }
            const int c = c0 + cc;
            const int64_t ob = static_cast<int64_t>(blockIdx.y) * 128 * Kp + 8 * g, on = gridDim.y * 128 * Kp;
            if (!bd_in_range(kBkMsSplit, ob + c * Kp, 8, on) || !bd_in_range(kBkMsSplit, ob + (64 + c) * Kp, 8, on))
                continue;
            *reinterpret_cast<uint4*>(o + static_cast<int64_t>(c) * Kp) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
            *reinterpret_cast<uint4*>(o + static_cast<int64_t>(32 + c) * Kp) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
            *reinterpret_cast<uint4*>(o + static_cast<int64_t>(64 + c) * Kp) = make_uint4(w3[0], w3[1], w3[2], w3[3]);
        }
    }
}

__device__ __forceinline__ void tmem_st16_nowait(uint32_t taddr, const uint32_t (&v)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

template <int MODE>
__global__ void __launch_bounds__(kTThreads, 1) tprod_kernel(const __grid_constant__ TProdParams p)
{
    extern __shared__ uint8_t dyn_raw[];
    __shared__ uint64_t full[kTStages], afull[kTStages], empty[kTStages];
    __shared__ uint64_t wfree[kTStages];  // the piece warps hold the stage's W values (W slots free)
    __shared__ uint64_t accfull, accempty;  // a unit's MMAs are done / the epilogue holds its accumulator
    __shared__ uint64_t done;               // every MMA issued has finished (before tensor memory is freed)
    __shared__ uint32_t tmem_base;
    __shared__ volatile int abort;
    uint8_t* ring = dyn_raw + ((1024u - (smem_u32(dyn_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nz = p.nz;
    const int64_t klen = MODE == 0 ? p.d_in : p.d_out;
    const int units = p.tiles * p.ns;
    // unit u (this CTA takes u = blockIdx.x, blockIdx.x + gridDim.x, ...): slice u / tiles, row block
    // (u % tiles) / nz, checkpoint u % nz -- the checkpoint varies fastest, so the CTAs that read the
    // same W_base tiles run side by side
    struct Unit {
        int z, slice, nt;
        int64_t o0, kb;
    };
    auto unit = [&](int u) {
        Unit x;
        const int tile = u % p.tiles;
        x.slice = u / p.tiles;
        x.z = tile % nz;
        x.o0 = static_cast<int64_t>(tile / nz) * kTM;
        x.kb = static_cast<int64_t>(x.slice) * p.k_per;
        const int64_t ke = x.kb + p.k_per < klen ? x.kb + p.k_per : klen;
        x.nt = ke > x.kb ? static_cast<int>((ke - x.kb + kTK - 1) / kTK) : 0;
        return x;
    };
    if (tid == 0) {
        for (int st = 0; st < kTStages; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&afull[st], kTConvWarps);
            mbar_init(&empty[st], 1);
            mbar_init(&wfree[st], kTConvWarps);
        }
        mbar_init(&accfull, 1);
        mbar_init(&accempty, 4);
        mbar_init(&done, 1);
        abort = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) tmem_alloc(&tmem_base, kTTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    grid_launch_dependents();  // the next kernel of the merge may start launching
    grid_dependency_wait();    // the previous kernel's results are visible
    const uint32_t tmem = tmem_base;
    auto wait = [&](uint64_t* bar, uint32_t par) {
        if (mbar_try_wait(bar, par)) return true;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(bar, par)) {
            if (abort) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                abort = 1;
                raise_error(p.err, kErrTimeout);
                return false;
            }
        }
        return true;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int g = 0;  // stages issued, over all units of this CTA
            bool ok = true;
            for (int u = blockIdx.x; ok && u < units; u += gridDim.x) {
                const Unit x = unit(u);
                for (int t = 0; t < x.nt; ++t, ++g) {
                    const int st = g % kTStages;
                    const uint32_t prev = static_cast<uint32_t>(g / kTStages - 1) & 1u;
                    if (g >= kTStages && !wait(&wfree[st], prev)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sb = ring + static_cast<size_t>(st) * kTStage;
                    const int k0 = static_cast<int>(x.kb + static_cast<int64_t>(t) * kTK);
                    mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(kTStage));
                    if (MODE == 0) {
                        tma_load_2d(sb, &p.w_map[x.z], k0, static_cast<int>(x.o0), &full[st]);
                        tma_load_2d(sb + kTWTile, &p.b_map, k0, static_cast<int>(x.o0), &full[st]);
                    } else {
#pragma unroll
                        for (int hb = 0; hb < 2; ++hb) {
                            const int cx = static_cast<int>(x.o0) + 64 * hb;
                            tma_load_2d(sb + hb * (kTWTile / 2), &p.w_map[x.z], cx, k0, &full[st]);
                            tma_load_2d(sb + kTWTile + hb * (kTWTile / 2), &p.b_map, cx, k0, &full[st]);
                        }
                    }
                    // the B tile once the stage's MMAs are done with it
                    if (g >= kTStages && !wait(&empty[st], prev)) {
                        ok = false;
                        break;
                    }
                    tma_load_2d(sb + 2 * kTWTile, &p.s_map[x.z], k0, 0, &full[st]);
                }
            }
            for (int i = (g > kTStages ? g - kTStages : 0); i < g; ++i) {  // every issued copy lands before exit
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(&full[i % kTStages], static_cast<uint32_t>(i / kTStages) & 1u) &&
                       global_timer_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            // piece a of Delta times the first 3 - a pieces of the small operand (B rows
            // 0 .. 32 (3 - a) - 1): the products of pieces a, b with a + b <= 2, as in
            // the merge.  Piece b + 1 is below 2^-7 of the value that piece b was cut
            // from, so the dropped products (a + b >= 3) of one term add up to less
            // than 2^-20 |Delta_j S_j|, below the fp32 accumulation error over K.
            constexpr uint32_t idesc_a[3] = {idesc_bf16_f32(kTM, 96), idesc_bf16_f32(kTM, 64),
                                             idesc_bf16_f32(kTM, 32)};
            int g = 0, j = 0;  // stages and units done by this CTA
            bool ok = true;
            for (int u = blockIdx.x; ok && u < units; u += gridDim.x, ++j) {
                const Unit x = unit(u);
                // the accumulator: free once the epilogue holds the previous unit's values
                if (j > 0 && !wait(&accempty, static_cast<uint32_t>(j - 1) & 1u)) break;
                tc_fence_after();
                for (int t = 0; t < x.nt; ++t, ++g) {
                    const int st = g % kTStages;
                    if (!wait(&afull[st], static_cast<uint32_t>(g / kTStages) & 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bdesc =
                        smem_desc_sw128(smem_u32(ring + static_cast<size_t>(st) * kTStage + 2 * kTWTile));
                    const uint32_t acol = tmem + kTACol + 96u * static_cast<uint32_t>(st);
#pragma unroll
                    for (int kk = 0; kk < kTK / 16; ++kk) {
#pragma unroll
                        for (int a = 0; a < 3; ++a)
                            mma_ts(tmem + kTDCol, acol + 32u * a + 8u * kk, bdesc + static_cast<uint64_t>(2 * kk),
                                   idesc_a[a], (t | kk | a) != 0 ? 1u : 0u);
                    }
                    mma_commit(&empty[st]);
                }
                if (ok) mma_commit(&accfull);  // every MMA of the unit has finished when this arrives
            }
            mma_commit(&done);  // also after a wait gave up: no MMA may be in flight when tensor memory is freed
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(&done, 0u) && global_timer_ns() - t0 < kWaitLimitNs) {
            }
        }
    } else if (warp < kTEpiWarp) {
        // ------------------------------------------------------------ pieces of Delta -> tensor memory
        const int q = warp & 3;                  // lane quarter: rows 32 q .. 32 q + 31 of A
        const int kh = (warp - 2) >> 2;          // K half: 32 reduction indices (16 columns) of each stage
        const int rl = 32 * q + lane;            // this thread's row of A
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(32 * q) << 16);
        int total = 0;  // stages of all units of this CTA
        for (int u = blockIdx.x; u < units; u += gridDim.x) total += unit(u).nt;
        for (int g = 0; g < total; ++g) {
            const int st = g % kTStages;
            if (!__all_sync(0xffffffffu, wait(&full[st], static_cast<uint32_t>(g / kTStages) & 1u))) break;
            const uint8_t* sb = ring + static_cast<size_t>(st) * kTStage;
            uint32_t v1[16], v2[16], v3[16];
            if (MODE == 0) {
                // row rl of the tiles, 16-byte chunks 4 kh .. 4 kh + 3 (swizzled)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int off = rl * 128 + (((4 * kh + c) ^ (rl & 7)) << 4);
                    const uint4 wi = *reinterpret_cast<const uint4*>(sb + off);
                    const uint4 wb = *reinterpret_cast<const uint4*>(sb + kTWTile + off);
                    split_pair(wi.x, wb.x, v1[4 * c + 0], v2[4 * c + 0], v3[4 * c + 0]);
                    split_pair(wi.y, wb.y, v1[4 * c + 1], v2[4 * c + 1], v3[4 * c + 1]);
                    split_pair(wi.z, wb.z, v1[4 * c + 2], v2[4 * c + 2], v3[4 * c + 2]);
                    split_pair(wi.w, wb.w, v1[4 * c + 3], v2[4 * c + 3], v3[4 * c + 3]);
                }
            } else {
                // column rl of the tile (box rl / 64, column rl % 64), rows 32 kh .. 32 kh + 31
                const int bx = rl >> 6, cb = rl & 63;
                const uint8_t* base = sb + bx * (kTWTile / 2) + (cb & 7) * 2;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int r0 = 32 * kh + 2 * j, r1 = r0 + 1;
                    const int off0 = r0 * 128 + (((cb >> 3) ^ (r0 & 7)) << 4);
                    const int off1 = r1 * 128 + (((cb >> 3) ^ (r1 & 7)) << 4);
                    const uint32_t wi = static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(base + off0)) |
                                        (static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(base + off1)) << 16);
                    const uint32_t wb =
                        static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(base + kTWTile + off0)) |
                        (static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(base + kTWTile + off1)) << 16);
                    split_pair(wi, wb, v1[j], v2[j], v3[j]);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&wfree[st]);  // the W values are in registers
            const uint32_t acol = lane_addr + kTACol + 96u * static_cast<uint32_t>(st) + 16u * kh;
            tmem_st16_nowait(acol, v1);
            tmem_st16_nowait(acol + 32, v2);
            tmem_st16_nowait(acol + 64, v3);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&afull[st]);
        }
    } else {
        // ------------------------------------------------------------ epilogue: one row of D per thread, per unit
        const int q = warp & 3;
        const int rl = 32 * q + lane;
        const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) + kTDCol;
        const int64_t nrows = MODE == 0 ? p.d_out : p.d_in;
        int j = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x, ++j) {
            const Unit x = unit(u);
            if (!__all_sync(0xffffffffu, wait(&accfull, static_cast<uint32_t>(j) & 1u))) break;
            tc_fence_after();
            // D[m][c] + D[m][32 + c] + D[m][64 + c], added in that order (64 registers live)
            uint32_t d0[32], d1[32];
            tmem_ld32(taddr, d0);
            tmem_ld32(taddr + 32, d1);
#pragma unroll
            for (int c = 0; c < 32; ++c) d0[c] = __float_as_uint(__uint_as_float(d0[c]) + __uint_as_float(d1[c]));
            tmem_ld32(taddr + 64, d1);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&accempty);  // the next unit's MMAs may overwrite D
#pragma unroll
            for (int c = 0; c < 32; ++c) d0[c] = __float_as_uint(__uint_as_float(d0[c]) + __uint_as_float(d1[c]));
            const int64_t row = x.o0 + rl;
            if (row < nrows) {
                const int64_t ob = ((static_cast<int64_t>(x.z) * p.ns + x.slice) * nrows + row) * p.l;
                float* out = p.part + ob;
#pragma unroll
                for (int c = 0; c < 32; c += 4) {
                    if (c >= p.l) break;
                    const float4 y = make_float4(__uint_as_float(d0[c]), __uint_as_float(d0[c + 1]),
                                                 __uint_as_float(d0[c + 2]), __uint_as_float(d0[c + 3]));
                    if (bd_in_range(kBkMsProd, ob + c, 4, static_cast<int64_t>(nz) * p.ns * nrows * p.l))
                        *reinterpret_cast<float4*>(out + c) = y;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTTmemCols);
    }
}

// ---------------------------------------------------------------- small-matrix steps
// GB300 has few fp64 units (about 2 fp64 FMAs per cycle per SM, with long
// latencies), so the Gram matrices and their Cholesky factors are computed in
// float-float arithmetic on the fp32 units (each product split exactly with
// an FMA, each sum with TwoSum; about 2^-44 relative, like fp64 for this
// purpose).

// s + t = a + b exactly (Knuth's TwoSum; explicit _rn intrinsics so that no
// operation is contracted or reordered).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& t)
{
    s = __fadd_rn(a, b);
    const float z = __fsub_rn(s, a);
    t = __fadd_rn(__fsub_rn(a, __fsub_rn(s, z)), __fsub_rn(b, z));
}

// (s, c) += a * b in float-float: the rounded product and its exact error
// (fma), the sum by TwoSum, the errors gathered in c.
__device__ __forceinline__ void ff_madd(float& s, float& c, float a, float b)
{
    const float p = __fmul_rn(a, b);
    const float pe = __fmaf_rn(a, b, -p);
    float t, e;
    two_sum(s, p, t, e);
    s = t;
    c = __fadd_rn(c, __fadd_rn(e, pe));
}

// (s, c) += (x, y) in float-float.
__device__ __forceinline__ void ff_add(float& s, float& c, float x, float y)
{
    float t, e;
    two_sum(s, x, t, e);
    s = t;
    c = __fadd_rn(c, __fadd_rn(e, y));
}

// Partial Gram matrices of A_z [n][l] (checkpoint z = blockIdx.y, the A_z
// consecutive): CTA b sums A_z^T A_z over its contiguous row range in
// float-float into part[z][b][l * l] (entry i * l + j as (hi, lo)).  Only the
// l (l + 1) / 2 entries i <= j are summed (ENT per thread, blockDim.x threads
// of consecutive entries; ENT = 1 takes at most kGramThreads1 threads and
// runs two CTAs per SM); each is stored at (i, j) and (j, i).  Rows come in
// chunks of kGramRows (one chunk for the usual 8192-row operands over about
// a hundred CTAs per checkpoint), l columns per row, coalesced.  With
// nslice > 1 the operand is the sum of a product's K slices (slice s of
// checkpoint z at a_all + (z nslice + s) n l, added in slice order) and the
// kernel also writes that sum to sum_all[z][n][l]: the CTAs' row ranges cover
// every row once, so no separate pass sums the slices.
constexpr int kGramThreads1 = 576;
constexpr int kGramRows = 96;
template <int ENT>
__global__ void __launch_bounds__(ENT == 1 ? kGramThreads1 : kGramThreads, ENT == 1 ? 2 : 1)
    gram_kernel(const float* __restrict__ a_all, int nslice, int64_t n, int l, float2* __restrict__ part_all,
                float* __restrict__ sum_all)
{
    grid_launch_dependents();  // the next kernel of the merge may start launching
    grid_dependency_wait();    // the previous kernel's results are visible
    __shared__ float sa[kGramRows][kMaxL + 1];
    const int tid = threadIdx.x, nt = blockDim.x;
    const float* a = a_all + static_cast<int64_t>(blockIdx.y) * nslice * n * l;
    float2* part = part_all + static_cast<int64_t>(blockIdx.y) * gridDim.x * l * l;
    const int64_t per = (n + gridDim.x - 1) / gridDim.x;
    const int64_t b0 = static_cast<int64_t>(blockIdx.x) * per;
    const int64_t b1 = b0 + per < n ? b0 + per : n;
    const int np = l * (l + 1) / 2;
    int pi[ENT], pj[ENT];
    float s[ENT], c[ENT];
#pragma unroll
    for (int m = 0; m < ENT; ++m) {
        int u = tid + nt * m;
        int i = 0;
        if (u < np) {
            while (u >= l - i) {  // u -> (i, j), i <= j, row-major over the upper triangle
                u -= l - i;
                ++i;
            }
        }
        pi[m] = u < np ? i : 0;  // past the triangle: a dummy entry, never stored
        pj[m] = u < np ? i + u : 0;
        s[m] = c[m] = 0.0f;
    }
    for (int64_t r0 = b0; r0 < b1; r0 += kGramRows) {
        const int nr = b1 - r0 < kGramRows ? static_cast<int>(b1 - r0) : kGramRows;
        for (int e = tid; e < nr * l; e += nt) {
            const int rr = e / l, cc = e - rr * l;
            const int64_t row = r0 + rr;
            const int64_t ext = static_cast<int64_t>(gridDim.y) * nslice * n * l;
            const int64_t at = static_cast<int64_t>(blockIdx.y) * nslice * n * l + row * l + cc;
            float v = bd_in(kBkMsGram, at, ext) ? a[row * l + cc] : 0.0f;
            for (int sl = 1; sl < nslice; ++sl)
                if (bd_in(kBkMsGram, at + sl * n * l, ext)) v += a[sl * n * l + row * l + cc];
            sa[rr][cc] = v;
            if (sum_all && bd_in(kBkMsGram, blockIdx.y * n * l + row * l + cc, static_cast<int64_t>(gridDim.y) * n * l))
                sum_all[static_cast<int64_t>(blockIdx.y) * n * l + row * l + cc] = v;
        }
        __syncthreads();
        for (int rr = 0; rr < nr; ++rr) {
#pragma unroll
            for (int m = 0; m < ENT; ++m) ff_madd(s[m], c[m], sa[rr][pi[m]], sa[rr][pj[m]]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int m = 0; m < ENT; ++m) {
        if (tid + nt * m < np) {
            float hi, lo;
            two_sum(s[m], c[m], hi, lo);
            const int64_t pb = static_cast<int64_t>(blockIdx.x) * l * l;
            const int64_t zb = static_cast<int64_t>(blockIdx.y) * gridDim.x * l * l,
                          np = static_cast<int64_t>(gridDim.y) * gridDim.x * l * l;
            if (bd_in(kBkMsGram, zb + pb + pi[m] * l + pj[m], np) && bd_in(kBkMsGram, zb + pb + pj[m] * l + pi[m], np)) {
                part[pb + pi[m] * l + pj[m]] = make_float2(hi, lo);
                part[pb + pj[m] * l + pi[m]] = make_float2(hi, lo);
            }
        }
    }
}

// G[z][e] = sum_b part[z][b][e], b < nb (float-float, normalised to
// (hi, lo) with |lo| <= ulp(hi) / 2), checkpoint z = blockIdx.y, one warp per
// entry: lane L takes partials L, L + 32, ... in order, then a fixed
// butterfly; the result does not depend on timing.
__global__ void __launch_bounds__(256) gram_sum_kernel(const float2* __restrict__ part_all, int nb, int l,
                                                       float2* __restrict__ G_all)
{
    grid_launch_dependents();  // the next kernel of the merge may start launching
    grid_dependency_wait();    // the previous kernel's results are visible
    const int e = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    const int ll = l * l;
    if (e >= ll) return;
    const float2* part = part_all + static_cast<int64_t>(blockIdx.y) * nb * ll;
    // four independent float-float chains per lane (partials lane + 32 (4 i + u)), then fixed combines
    float s[4] = {0.0f, 0.0f, 0.0f, 0.0f}, c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int b = lane; b < nb; b += 128) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int bb = b + 32 * u;
            if (bb < nb) {
                if (!bd_in(kBkMsGramSum, (static_cast<int64_t>(blockIdx.y) * nb + bb) * ll + e,
                           static_cast<int64_t>(gridDim.y) * nb * ll))
                    continue;
                const float2 v = part[static_cast<int64_t>(bb) * ll + e];
                ff_add(s[u], c[u], v.x, v.y);
            }
        }
    }
    ff_add(s[0], c[0], s[1], c[1]);
    ff_add(s[2], c[2], s[3], c[3]);
    ff_add(s[0], c[0], s[2], c[2]);
    float sv = s[0], cv = c[0];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float os = __shfl_xor_sync(0xffffffffu, sv, o), oc = __shfl_xor_sync(0xffffffffu, cv, o);
        ff_add(sv, cv, os, oc);  // fixed butterfly: lane 0's sum does not depend on timing
    }
    if (lane == 0) {
        float hi, lo;
        two_sum(sv, cv, hi, lo);
        if (bd_in(kBkMsGramSum, static_cast<int64_t>(blockIdx.y) * ll + e, static_cast<int64_t>(gridDim.y) * ll))
            G_all[static_cast<int64_t>(blockIdx.y) * ll + e] = make_float2(hi, lo);
    }
}

// s + t = a + b exactly when |a| >= |b| or a = 0 (Dekker's Fast2Sum).
__device__ __forceinline__ void fast_two_sum(float a, float b, float& s, float& t)
{
    s = __fadd_rn(a, b);
    t = __fsub_rn(b, __fsub_rn(s, a));
}

// (ph, pl) = (ah + al) (bh + bl) in float-float (the al bl term, below
// 2^-48 of the product, is left out), normalised.
__device__ __forceinline__ void ff_mul(float ah, float al, float bh, float bl, float& ph, float& pl)
{
    const float p = __fmul_rn(ah, bh);
    float e = __fmaf_rn(ah, bh, -p);
    e = __fmaf_rn(ah, bl, e);
    e = __fmaf_rn(al, bh, e);
    fast_two_sum(p, e, ph, pl);
}

// (h, l) += (xh, xl) in float-float, normalised.
__device__ __forceinline__ void ff_add_norm(float& h, float& l, float xh, float xl)
{
    float s, e;
    two_sum(h, xh, s, e);
    fast_two_sum(s, __fadd_rn(e, __fadd_rn(l, xl)), h, l);
}

// One CTA per checkpoint (blockIdx.x): G = R^T R (Cholesky, R upper) in
// float-float, right-looking; R written as fp32 [l][l] (zero below the
// diagonal) with the reciprocals of its diagonal in rinv (Rf of checkpoint z
// at Rf_all + z (kMaxL^2 + kMaxL), rinv right after its kMaxL^2 floats).
// Pivot d: y = rsqrt(d_hi) (fp32, about 2^-22), s0 = d_hi y, one Newton step
// s = s0 + (d - s0^2) y / 2 with d - s0^2 formed exactly (Sterbenz and an
// FMA), then 1/s by one Newton step from y; both within about 2^-42.  Warp 0 takes the pivot (every lane the same
// values) and scales row k by 1/s; the CTA then updates the trailing upper
// triangle.  A pivot below 1e-12 of the largest diagonal entry drops its
// direction (its row of R and its reciprocal are zero).
__global__ void __launch_bounds__(256) chol_kernel(const float2* __restrict__ G_all, int l, float* __restrict__ Rf_all)
{
    grid_launch_dependents();  // the next kernel of the merge may start launching
    grid_dependency_wait();    // the previous kernel's results are visible
    __shared__ float2 g[kMaxL][kMaxL + 1];
    __shared__ float rdiag[kMaxL];
    __shared__ int live[kMaxL];
    __shared__ float dmax;
    const float2* G = G_all + static_cast<int64_t>(blockIdx.x) * l * l;
    float* Rf = Rf_all + static_cast<int64_t>(blockIdx.x) * (kMaxL * kMaxL + kMaxL);
    float* rinv = Rf + kMaxL * kMaxL;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ti = tid >> 4, tj = tid & 15;
    for (int e = tid; e < l * l; e += 256)
        g[e / l][e % l] = bd_in(kBkMsChol, static_cast<int64_t>(blockIdx.x) * l * l + e,
                                static_cast<int64_t>(gridDim.x) * l * l)
                              ? G[e]
                              : make_float2(0.0f, 0.0f);
    __syncthreads();
    if (warp == 0) {
        float m = 0.0f;
        for (int i = lane; i < l; i += 32) m = fmaxf(m, g[i][i].x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) dmax = m;
    }
    __syncthreads();
    const float tol = 1e-12f * dmax;
    for (int k = 0; k < l; ++k) {
        if (warp == 0) {
            const float dh = g[k][k].x, dl = g[k][k].y;
            const bool ok = dh > tol && dh > 0.0f;
            float sh = 0.0f, sl = 0.0f, ih = 0.0f, il = 0.0f;
            if (ok) {
                const float y = rsqrtf(dh);
                const float s0 = __fmul_rn(dh, y);
                const float p = __fmul_rn(s0, s0), pe = __fmaf_rn(s0, s0, -p);
                const float res = __fadd_rn(__fsub_rn(__fsub_rn(dh, p), pe), dl);  // d - s0^2
                fast_two_sum(s0, __fmul_rn(__fmul_rn(0.5f, res), y), sh, sl);
                float t = __fmaf_rn(-sh, y, 1.0f);  // 1 - s y
                t = __fmaf_rn(-sl, y, t);
                fast_two_sum(y, __fmul_rn(y, t), ih, il);
            }
            for (int j = k + 1 + lane; j < l; j += 32) {
                float2 v = g[k][j];
                ff_mul(v.x, v.y, ih, il, v.x, v.y);
                g[k][j] = v;
            }
            if (lane == 0) {
                g[k][k] = make_float2(sh, sl);
                rdiag[k] = ih;
                live[k] = ok ? 1 : 0;
            }
        }
        __syncthreads();
        for (int i = k + 1 + ti; i < l; i += 16) {
            const float2 a = g[k][i];
            for (int j = i + ((tj - i) & 15); j < l; j += 16) {
                const float2 b = g[k][j];
                float ph, pl;
                ff_mul(a.x, a.y, b.x, b.y, ph, pl);
                float2 v = g[i][j];
                ff_add_norm(v.x, v.y, -ph, -pl);
                g[i][j] = v;
            }
        }
        __syncthreads();
    }
    for (int e = tid; e < l * l; e += 256) {
        const int i = e / l, j = e % l;
        if (bd_in(kBkMsChol, e, kMaxL * kMaxL)) Rf[e] = (j >= i && live[i]) ? g[i][j].x : 0.0f;
    }
    for (int i = tid; i < l; i += 256)
        if (bd_in(kBkMsChol, i, kMaxL)) rinv[i] = live[i] ? rdiag[i] : 0.0f;
}

// The r leading eigenvectors of the symmetric l x l matrix G of each
// checkpoint (one CTA of 256 threads per checkpoint, fp32; G arrives as
// float-float pairs and is rounded to fp32):
//   1. Householder tridiagonalisation Q^T G Q = T (reflector k, for
//      k < l - 2, zeroes column k below the subdiagonal; its vector and 2 /
//      (v^T v) are kept for step 4): per reflector one warp forms it, the CTA
//      forms p = tau S v, w = p - (tau v^T p / 2) v and the rank-2 update of
//      the trailing block S -= v w^T + w v^T;
//   2. a half-warp finds the m-th largest eigenvalue of T (m < r) by
//      multisection of the Gershgorin interval on the Sturm count (the number
//      of negative pivots of T - x I): 16 points per round, at most 12 rounds
//      or until the interval is two ulps wide;
//   3. thread m then takes two steps of inverse iteration with T - lambda_m I
//      (tridiagonal elimination, tiny pivots replaced by a floor) from a fixed
//      start vector, and one warp orthonormalises the r vectors in order of
//      decreasing eigenvalue (Gram-Schmidt, twice, within clusters of close
//      eigenvalues, which keeps the vectors of close eigenvalues apart; then
//      one Newton-Schulz step over all r vectors);
//   4. each vector is carried back to G's basis by the reflectors in reverse
//      order (a warp takes two vectors at a time, in registers).
// ur[i][m] = entry i of the unit eigenvector of the m-th largest eigenvalue,
// m < r.  Standard dense symmetric eigensolver steps (Householder
// tridiagonalisation, Sturm bisection, inverse iteration), as in Golub and
// Van Loan, "Matrix Computations", sections 8.3-8.4.
constexpr int kEigThreads = 256;
constexpr int kEigLd = kMaxL + 1;  // row stride of A and of the vectors
constexpr int kEigLuLd = 2 * kMaxL + 1;  // row stride of the per-vector pivots (odd: no bank conflicts)
constexpr size_t kEigSmem =
    static_cast<size_t>(kMaxL * kEigLd + kMaxL * kMaxL + kMaxL * kEigLuLd + kMaxL * kEigLd + 12 * kMaxL) * 4;

__global__ void __launch_bounds__(kEigThreads) eig_kernel(const float2* __restrict__ G_all, int l, int r,
                                                          float* __restrict__ ur_all)
{
    grid_launch_dependents();  // the next kernel of the merge may start launching
    grid_dependency_wait();    // the previous kernel's results are visible
    extern __shared__ float esm[];
    float* A = esm;                                   // [kMaxL][kEigLd]
    float* HV = A + kMaxL * kEigLd;                   // [kMaxL][kMaxL]: reflector k, entries 0 .. l - k - 2
    float* LU = HV + kMaxL * kMaxL;                   // [kMaxL][kEigLuLd]: per vector m, u_i then l_i
    float* Y = LU + kMaxL * kEigLuLd;                 // [kMaxL][kEigLd]: vector m, entry i
    float* tau = Y + kMaxL * kEigLd;
    float* dd = tau + kMaxL;
    float* ee = dd + kMaxL;
    float* e2 = ee + kMaxL;
    float* pv = e2 + kMaxL;
    float* wv = pv + kMaxL;
    float* red = wv + kMaxL;  // 4 kMaxL floats of scratch
    const float2* G = G_all + static_cast<size_t>(blockIdx.x) * l * l;
    float* ur = ur_all + static_cast<size_t>(blockIdx.x) * l * r;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < l * l; e += kEigThreads)
        A[(e / l) * kEigLd + e % l] =
            bd_in(kBkMsEig, static_cast<int64_t>(blockIdx.x) * l * l + e, static_cast<int64_t>(gridDim.x) * l * l)
                ? __fadd_rn(G[e].x, G[e].y)
                : 0.0f;
    __syncthreads();

    // ---------------------------------------------------------------- 1. tridiagonalisation
    // Every warp forms reflector k itself (its vector in registers: entries
    // lane and lane + 32) and the p entries of its rows; after a barrier every
    // warp forms K and w for itself and updates its rows of S; a second
    // barrier ends the step.  Warp 0 keeps the reflectors for step 4.
    for (int k = 0; k + 2 < l; ++k) {
        const int m = l - k - 1;  // the trailing block S = A[k+1..][k+1..] is m x m
        const float x0 = A[(k + 1) * kEigLd + k];
        const float xa = lane < m ? A[(k + 1 + lane) * kEigLd + k] : 0.0f;
        const float xb = lane + 32 < m ? A[(k + 33 + lane) * kEigLd + k] : 0.0f;
        float sg = fmaf(xa, xa, xb * xb);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sg += __shfl_xor_sync(0xffffffffu, sg, o);
        float alpha = 0.0f, t = 0.0f, v0 = x0;
        if (sg > 0.0f) {
            alpha = -copysignf(sqrtf(sg), x0);
            v0 = x0 - alpha;
            const float vtv = sg - x0 * x0 + v0 * v0;
            t = vtv > 0.0f ? 2.0f / vtv : 0.0f;
        }
        const float va = lane == 0 ? v0 : xa, vb = xb;  // v_i, i = lane and lane + 32
        if (warp == 0) {
            if (lane < m) HV[k * kMaxL + lane] = va;
            if (lane + 32 < m) HV[k * kMaxL + 32 + lane] = vb;
            if (lane == 0) {
                tau[k] = t;
                ee[k] = t > 0.0f ? alpha : x0;  // the subdiagonal entry this reflector leaves
            }
        }
        if (t != 0.0f) {
            // p_i = tau (S v)_i for this warp's rows i = warp, warp + 8, ...
            for (int i = warp; i < m; i += kEigThreads / 32) {
                const float* srow = &A[(k + 1 + i) * kEigLd + k + 1];
                float sv = (lane < m ? srow[lane] * va : 0.0f) + (lane + 32 < m ? srow[lane + 32] * vb : 0.0f);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) sv += __shfl_xor_sync(0xffffffffu, sv, o);
                if (lane == 0) pv[i] = t * sv;
            }
        }
        __syncthreads();
        if (t != 0.0f) {
            const float pa = lane < m ? pv[lane] : 0.0f, pb = lane + 32 < m ? pv[lane + 32] : 0.0f;
            float kp = fmaf(pa, va, pb * vb);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) kp += __shfl_xor_sync(0xffffffffu, kp, o);
            const float K = 0.5f * t * kp;
            const float wa = fmaf(-K, va, pa), wb = fmaf(-K, vb, pb);  // w_i, i = lane and lane + 32
            for (int i = warp; i < m; i += kEigThreads / 32) {
                // this warp's row i: S[i][j] -= v_i w_j + w_i v_j
                const float vi = __shfl_sync(0xffffffffu, i < 32 ? va : vb, i & 31);
                const float wi = __shfl_sync(0xffffffffu, i < 32 ? wa : wb, i & 31);
                float* srow = &A[(k + 1 + i) * kEigLd + k + 1];
                if (lane < m) srow[lane] = fmaf(-vi, wa, fmaf(-wi, va, srow[lane]));
                if (lane + 32 < m) srow[lane + 32] = fmaf(-vi, wb, fmaf(-wi, vb, srow[lane + 32]));
            }
        }
        __syncthreads();
    }
    for (int i = tid; i < l; i += kEigThreads) {
        dd[i] = A[i * kEigLd + i];
        if (i + 2 == l) ee[i] = A[(i + 1) * kEigLd + i];  // the last subdiagonal entry (no reflector)
    }
    __syncthreads();
    for (int i = tid; i + 1 < l; i += kEigThreads) e2[i] = ee[i] * ee[i];
    __syncthreads();

    // ---------------------------------------------------------------- 2. eigenvalues by multisection
    // A half-warp per eigenvalue (m = half-warp index, then + 16, ...): each of
    // its 16 lanes counts the eigenvalues below one of 16 interior points of
    // the interval, and the interval shrinks to the 1/17 that holds the
    // eigenvalue; at most 12 rounds, or until the interval is two ulps wide.
    float scale, pivmin, ufl;
    {
        float lo = dd[0], hi = dd[0], emax2 = 0.0f;
        for (int i = 0; i < l; ++i) {
            const float rad = (i > 0 ? fabsf(ee[i - 1]) : 0.0f) + (i + 1 < l ? fabsf(ee[i]) : 0.0f);
            lo = fminf(lo, dd[i] - rad);
            hi = fmaxf(hi, dd[i] + rad);
            if (i + 1 < l) emax2 = fmaxf(emax2, e2[i]);
        }
        scale = fmaxf(fabsf(lo), fabsf(hi));
        pivmin = fmaxf(1e-30f, 0x1p-60f * fmaxf(emax2, scale * scale));
        ufl = fmaxf(pivmin, 0x1p-23f * scale);
        const int hw = tid >> 4, g = tid & 15;
        for (int mb = 0; mb < r; mb += kEigThreads / 16) {  // trip count uniform over the CTA
            const int mm = mb + hw;
            const bool act = mm < r;
            float a = lo - (0x1p-22f * scale + pivmin), b = hi + (0x1p-22f * scale + pivmin);
            const int target = act ? l - 1 - mm : 0;  // index of the eigenvalue in ascending order
            for (int it = 0; it < 12; ++it) {
                const float step = (b - a) * (1.0f / 17.0f);
                const float x = g == 15 ? b - step : a + static_cast<float>(g + 1) * step;
                int cnt = 0;
                float q = dd[0] - x;
                if (fabsf(q) < pivmin) q = -pivmin;
                cnt += q < 0.0f ? 1 : 0;
                for (int i = 1; i < l; ++i) {
                    q = (dd[i] - x) - __fdividef(e2[i - 1], q);
                    if (fabsf(q) < pivmin) q = -pivmin;
                    cnt += q < 0.0f ? 1 : 0;
                }
                // the first point above the eigenvalue (count > target) bounds it from above
                const unsigned above = __ballot_sync(0xffffffffu, cnt > target) >> (tid & 16);
                const unsigned mine = above & 0xFFFFu;
                const int gf = mine ? __ffs(mine) - 1 : 16;
                const float xl = __shfl_sync(0xffffffffu, x, ((tid & 16) | (gf > 0 ? gf - 1 : 0)));
                const float xh = __shfl_sync(0xffffffffu, x, ((tid & 16) | (gf < 16 ? gf : 15)));
                const float na = gf > 0 ? xl : a, nb = gf < 16 ? xh : b;
                const bool done = !(na < nb) || (nb - na) <= 2.0f * (fabsf(na) + fabsf(nb)) * 0x1p-24f;
                a = na;
                b = nb;
                if (__all_sync(0xffffffffu, done)) break;
            }
            if (act && g == 0) red[mm] = 0.5f * (a + b);
        }
    }
    __syncthreads();

    // ---------------------------------------------------------------- 3. inverse iteration, then Gram-Schmidt
    if (tid < r) {
        const int mm = tid;
        const float lam = red[mm];
        // T - lam I = L U (no pivoting; a pivot below the floor is replaced by it)
        float* U = LU + mm * kEigLuLd;
        float* Lf = U + kMaxL;
        float u = dd[0] - lam;
        if (fabsf(u) < ufl) u = u < 0.0f ? -ufl : ufl;
        U[0] = u;
        for (int i = 1; i < l; ++i) {
            const float lf = __fdividef(ee[i - 1], u);
            u = (dd[i] - lam) - lf * ee[i - 1];
            if (fabsf(u) < ufl) u = u < 0.0f ? -ufl : ufl;
            Lf[i] = lf;
            U[i] = u;
        }
        float* y = Y + mm * kEigLd;
        for (int i = 0; i < l; ++i) y[i] = 1.0f + 0.125f * static_cast<float>((i * 7 + mm * 3) % 11);  // start vector
        for (int pass = 0; pass < 2; ++pass) {
            for (int i = 1; i < l; ++i) y[i] = fmaf(-Lf[i], y[i - 1], y[i]);
            y[l - 1] = __fdividef(y[l - 1], U[l - 1]);
            for (int i = l - 2; i >= 0; --i) y[i] = __fdividef(fmaf(-ee[i], y[i + 1], y[i]), U[i]);
            // scale by the largest entry first (the solve can grow large), then normalise;
            // a vector that is not finite or zero becomes the unit vector e_mm
            float mx = 0.0f;
            for (int i = 0; i < l; ++i) mx = fmaxf(mx, fabsf(y[i]));
            if (!(mx > 0.0f) || !isfinite(mx)) {
                for (int i = 0; i < l; ++i) y[i] = i == mm ? 1.0f : 0.0f;
                continue;
            }
            const float inv = 1.0f / mx;
            float nn = 0.0f;
            for (int i = 0; i < l; ++i) {
                y[i] *= inv;
                nn = fmaf(y[i], y[i], nn);
            }
            const float sc = rsqrtf(nn);
            for (int i = 0; i < l; ++i) y[i] *= sc;
        }
    }
    __syncthreads();
    // Gram-Schmidt in order of decreasing eigenvalue, twice, by warp 0 alone,
    // within clusters: a vector is projected off the earlier vectors whose
    // eigenvalues lie within 2^-10 of the spectrum's scale of its own (the
    // vectors of eigenvalues further apart are orthogonal to about
    // 2^-23 scale / gap after inverse iteration)
    if (warp == 0) {
        for (int rep = 0; rep < 2; ++rep) {
            int c0 = 0;  // first vector of the current cluster
            for (int mm = 0; mm < r; ++mm) {
                if (mm > 0 && red[c0] - red[mm] > 0x1p-10f * scale) {
                    c0 = mm;
                    while (c0 > 0 && red[c0 - 1] - red[mm] <= 0x1p-10f * scale) --c0;
                }
                if (c0 == mm) continue;  // no earlier vector in its cluster: already a unit vector
                float ya = lane < l ? Y[mm * kEigLd + lane] : 0.0f;
                float yb = lane + 32 < l ? Y[mm * kEigLd + lane + 32] : 0.0f;
                for (int i0 = c0; i0 < mm; ++i0) {
                    const float ua = lane < l ? Y[i0 * kEigLd + lane] : 0.0f;
                    const float ub = lane + 32 < l ? Y[i0 * kEigLd + lane + 32] : 0.0f;
                    float d = fmaf(ua, ya, ub * yb);
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
                    ya = fmaf(-d, ua, ya);
                    yb = fmaf(-d, ub, yb);
                }
                float nn = fmaf(ya, ya, yb * yb);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) nn += __shfl_xor_sync(0xffffffffu, nn, o);
                if (nn > 0x1p-40f) {
                    const float sc = rsqrtf(nn);
                    ya *= sc;
                    yb *= sc;
                } else {  // nothing left after the projection: a unit vector, orthogonalised by the next pass
                    ya = lane == mm ? 1.0f : 0.0f;
                    yb = lane + 32 == mm ? 1.0f : 0.0f;
                }
                if (lane < l) Y[mm * kEigLd + lane] = ya;
                if (lane + 32 < l) Y[mm * kEigLd + lane + 32] = yb;
                __syncwarp();
            }
        }
    }
    __syncthreads();
    // One Newton-Schulz step over all r vectors (the rows of Y):
    // Y <- (3 I - Y Y^T) Y / 2 keeps their span and takes an orthonormality
    // error e to about 1.5 e^2 (plus fp32 dot-product rounding).  It covers
    // the pairs that Gram-Schmidt leaves alone: inverse iteration makes the
    // vectors of eigenvalues g apart orthogonal only to about 2^-23 scale / g,
    // 2^-13 at the cluster threshold.  C = (3 I - Y Y^T) / 2 takes the
    // pivots' space, the result A's (both free by now).
    {
        float* C = LU;
        for (int e = tid; e < r * r; e += kEigThreads) {
            const int a = e / r, b = e - a * r;
            const float* ya = Y + a * kEigLd;
            const float* yb = Y + b * kEigLd;
            float d = 0.0f;
            for (int i = 0; i < l; ++i) d = fmaf(ya[i], yb[i], d);
            C[e] = (a == b ? 1.5f : 0.0f) - 0.5f * d;
        }
        __syncthreads();
        for (int e = tid; e < r * l; e += kEigThreads) {
            const int mm = e / l, i = e - mm * l;
            const float* c = C + mm * r;
            float s = 0.0f;
            for (int b = 0; b < r; ++b) s = fmaf(c[b], Y[b * kEigLd + i], s);
            A[mm * kEigLd + i] = s;
        }
        __syncthreads();
    }

    // ---------------------------------------------------------------- 4. back to G's basis
    // Warp w carries vectors w + 8 j (two at a time, entries lane and
    // lane + 32 in registers) through the reflectors in reverse order:
    // y <- y - tau (v^T y) v, v_i at entry k + 1 + i.
    for (int j0 = warp; j0 < r; j0 += 2 * (kEigThreads / 32)) {
        const int mA = j0, mB = j0 + kEigThreads / 32;
        const bool hasB = mB < r;
        float ya0 = lane < l ? A[mA * kEigLd + lane] : 0.0f;
        float ya1 = lane + 32 < l ? A[mA * kEigLd + lane + 32] : 0.0f;
        float yb0 = hasB && lane < l ? A[mB * kEigLd + lane] : 0.0f;
        float yb1 = hasB && lane + 32 < l ? A[mB * kEigLd + lane + 32] : 0.0f;
        for (int k = l - 3; k >= 0; --k) {
            const float t = tau[k];
            if (t == 0.0f) continue;
            const int m = l - k - 1;
            const int i0 = lane - (k + 1), i1 = lane + 32 - (k + 1);
            const float v0 = (i0 >= 0 && i0 < m) ? HV[k * kMaxL + i0] : 0.0f;
            const float v1 = (i1 >= 0 && i1 < m) ? HV[k * kMaxL + i1] : 0.0f;
            float sa = fmaf(v0, ya0, v1 * ya1), sb = fmaf(v0, yb0, v1 * yb1);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                sa += __shfl_xor_sync(0xffffffffu, sa, o);
                sb += __shfl_xor_sync(0xffffffffu, sb, o);
            }
            sa *= t;
            sb *= t;
            ya0 = fmaf(-sa, v0, ya0);
            ya1 = fmaf(-sa, v1, ya1);
            yb0 = fmaf(-sb, v0, yb0);
            yb1 = fmaf(-sb, v1, yb1);
        }
        if (lane < l) A[mA * kEigLd + lane] = ya0;
        if (lane + 32 < l) A[mA * kEigLd + lane + 32] = ya1;
        if (hasB && lane < l) A[mB * kEigLd + lane] = yb0;
        if (hasB && lane + 32 < l) A[mB * kEigLd + lane + 32] = yb1;
    }
    __syncthreads();
    for (int e = tid; e < l * r; e += kEigThreads) {
        const int i = e / r, mm = e - i * r;
        if (bd_in(kBkMsEig, static_cast<int64_t>(blockIdx.x) * l * r + e, static_cast<int64_t>(gridDim.x) * l * r))
            ur[e] = A[mm * kEigLd + i];
    }
}

// A_z <- A_z R_z^-1 in place (R_z from chol_kernel, checkpoint z =
// blockIdx.y): per row the forward substitution x_j = (a_j - sum_{m<j} x_m
// R[m][j]) / R[j][j] (the sum in order m = 0, 1, ...), a dropped direction
// giving x_j = 0; one row per thread (16-byte row loads and stores), R
// staged transposed so that four coefficients of column j come with one
// 16-byte broadcast load.  With sp_all (l <= 32, the last CholeskyQR pass
// before a tensor-core product) the kernel also writes the small operand's
// bf16 pieces as split_small_kernel does, Sp[z][32 b + c][row] for every
// row < kp (zero past n and for c >= l), so that pass needs no split
// launch.
constexpr int kTriThreads = 128;
constexpr int kTriStride = kMaxL + 4;  // floats per row of R^T in shared memory (16-byte multiple)

__global__ void __launch_bounds__(kTriThreads) tri_solve_kernel(float* a_all, int64_t n, int l,
                                                                const float* __restrict__ Rf_all,
                                                                uint16_t* __restrict__ sp_all, int64_t kp)
{
    grid_launch_dependents();  // the next kernel of the merge may start launching
    grid_dependency_wait();    // the previous kernel's results are visible
    float* a = a_all + static_cast<int64_t>(blockIdx.y) * n * l;
    const float* Rf = Rf_all + static_cast<int64_t>(blockIdx.y) * (kMaxL * kMaxL + kMaxL);
    const float* rinv = Rf + kMaxL * kMaxL;
    __shared__ __align__(16) float srt[kMaxL][kTriStride];  // srt[j][m] = R[m][j]
    __shared__ float sd[kMaxL];
    for (int e = threadIdx.x; e < kMaxL * kTriStride; e += blockDim.x) {
        const int j = e / kTriStride, m = e - j * kTriStride;
        srt[j][m] = (j < l && m < l && bd_in(kBkMsTri, m * l + j, kMaxL * kMaxL)) ? Rf[m * l + j] : 0.0f;
    }
    for (int i = threadIdx.x; i < kMaxL; i += blockDim.x) sd[i] = i < l ? rinv[i] : 0.0f;
    __syncthreads();
    const int64_t row = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const bool live = row < n &&
                      bd_in_range(kBkMsTri, blockIdx.y * n * l + row * l, l, static_cast<int64_t>(gridDim.y) * n * l);
    if (!live && (sp_all == nullptr || row >= kp)) return;
    float x[kMaxL];
    float4* ar = reinterpret_cast<float4*>(a + row * l);  // l is a multiple of 4
#pragma unroll
    for (int j4 = 0; j4 < kMaxL / 4; ++j4) {
        const float4 v = live && 4 * j4 < l ? ar[j4] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        x[4 * j4] = v.x;
        x[4 * j4 + 1] = v.y;
        x[4 * j4 + 2] = v.z;
        x[4 * j4 + 3] = v.w;
    }
#pragma unroll
    for (int j = 0; j < kMaxL; ++j) {
        if (j >= l) break;
        float s = x[j];
#pragma unroll
        for (int m4 = 0; m4 < (j + 3) / 4; ++m4) {
            const float4 r = *reinterpret_cast<const float4*>(&srt[j][4 * m4]);
            const float rv[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (4 * m4 + u < j) s = fmaf(-x[4 * m4 + u], rv[u], s);
        }
        x[j] = s * sd[j];
    }
    if (live) {
#pragma unroll
        for (int j4 = 0; j4 < kMaxL / 4; ++j4)
            if (4 * j4 < l) ar[j4] = make_float4(x[4 * j4], x[4 * j4 + 1], x[4 * j4 + 2], x[4 * j4 + 3]);
    }
    if (sp_all != nullptr && row < kp) {
        // the three bf16 pieces of each x_c (c < 32; zero for c >= l and past n)
        uint16_t* o = sp_all + static_cast<int64_t>(blockIdx.y) * 128 * kp + row;
        const int64_t ne = static_cast<int64_t>(gridDim.y) * 128 * kp;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            const float v = c < l ? x[c] : 0.0f;
            const uint32_t b1 = __float_as_uint(v) & 0xFFFF0000u;
            const float r1 = __fsub_rn(v, __uint_as_float(b1));
            const uint32_t b2 = __float_as_uint(r1) & 0xFFFF0000u;
            const float r2 = __fsub_rn(r1, __uint_as_float(b2));
            const int64_t base = static_cast<int64_t>(blockIdx.y) * 128 * kp + row;
            if (bd_in(kBkMsTri, base + static_cast<int64_t>(64 + c) * kp, ne)) {
                o[static_cast<int64_t>(c) * kp] = static_cast<uint16_t>(b1 >> 16);
                o[static_cast<int64_t>(32 + c) * kp] = static_cast<uint16_t>(b2 >> 16);
                o[static_cast<int64_t>(64 + c) * kp] = static_cast<uint16_t>(__float_as_uint(r2) >> 16);
            }
        }
    }
}

// ---------------------------------------------------------------- the merge on the tensor cores
// out[row][j] = W_base[row][j] + inv_k * sum_e L[e][row] R[e][j], e over the
// K = k r factor columns, rounded once to the output type.  Every factor
// value is split into three bf16 pieces (as for the products) and the six
// piece pairs (1,1), (1,2), (2,1), (1,3), (2,2), (3,1) are stacked along the
// reduction: Ls[row][p K + e] = piece a_p of L[e][row], Rs[j][p K + e] =
// piece b_p of R[e][j] (factor_split_kernel forms the factors and writes
// them so; a piece after the first is below 2^-7 of the
// value's magnitude and the third below 2^-15, so the three pairs left out
// add up to less than 2^-21 |L[e][row] R[e][j]|), zero-padded to Kp = 6 K
// rounded up to 64.  Persistent CTAs (one per SM) walk the 128-row x
// 256-column output tiles c, c + G, c + 2G, ... (row-major tile order): per
// tile D = Ls Rs^T in tensor memory (M = 128, N = 256, K = 16 MMAs; A and B
// K-major in shared memory, a ring of three 48 KB stages shared by all the
// CTA's tiles), with two accumulators of 256 columns, so that the MMAs of
// the next tile run while warps 2..9 add W_base to this one row by row (lane
// quarter warp % 4, column half (warp - 2) / 4).  Warp 10 loads each tile's
// W_base block by TMA (four 64-column boxes, 128-byte swizzle, 64 KB) into
// one of two buffers as soon as the epilogue has finished with the tile two
// back, so the epilogue reads W_base from shared memory and the next block
// is in flight while it works.  Two operand stages (48 KB each) leave room
// for the two W_base buffers.
constexpr int kMgM = 128;
constexpr int kMgN = 256;
constexpr int kMgStages = 2;
constexpr int kMgWBufs = 2;                   // W_base blocks in flight
constexpr int kMgATile = kMgM * 128;          // 64 reduction indices x 128 rows, bf16: 16 KB
constexpr int kMgBTile = kMgN * 128;          // 64 x 256: 32 KB
constexpr int kMgStage = kMgATile + kMgBTile;
constexpr int kMgWTile = kMgM * kMgN * 2;     // a tile's W_base block: 64 KB
constexpr int kMgThreads = 352;               // warp 0 TMA, warp 1 MMA, warps 2..9 epilogue, warp 10 W_base
constexpr uint32_t kMgTmemCols = 2 * kMgN;    // two accumulators
constexpr int kMgPairs = 6;

__device__ __forceinline__ int merge_piece(int p, int side)
{
    // piece index (0, 1, 2) of the L side (side 0) or the R side (side 1) in pair p
    const int a = p == 2 ? 1 : (p == 4 ? 1 : (p == 5 ? 2 : 0));
    const int b = p == 1 ? 1 : (p == 3 ? 2 : (p == 4 ? 1 : 0));
    return side == 0 ? a : b;
}

// The merge's factor operands straight from the bases and the eigenvectors:
// row n of side 0 holds L_z[n][e] = sum_c Q_z[n][c] U_z[c][e] (Q_z the
// d_out x l basis of checkpoint z), row n of side 1 holds R_z[n][e] =
// sum_c Bt_z[n][c] U_z[c][e] (Bt_z = Delta_z^T Q_z, d_in x l), for every
// checkpoint z < k and e < r (factor index E = z r + e, K = k r of them).
// Each value is split into three bf16 pieces and stored as the stacked piece
// pairs merge_tc_kernel reads: dst[n][p K + E] = piece merge_piece(p, side)
// of it (p < 6), zero for p K + E >= 6 K up to Kp.  A warp takes one row at
// a time (rows numbered with the d_out rows of side 0 first, the warps of
// the grid striding over them), lane L taking E = L, L + 32, ...: the stores
// of a warp are consecutive; the sum over c runs in order c = 0, 1, ...
constexpr int kFsStageFloats = 12288;  // U of all checkpoints staged in shared memory up to 48 KB

__global__ void __launch_bounds__(256) factor_split_kernel(const float* __restrict__ Yall,
                                                           const float* __restrict__ Zall, int64_t d_out,
                                                           int64_t d_in, int l, int k, int r,
                                                           const float* __restrict__ Uk, int K, int Kp,
                                                           uint16_t* __restrict__ Ls, uint16_t* __restrict__ Rs)
{
    extern __shared__ float su[];  // U when k l r <= kFsStageFloats
    grid_launch_dependents();  // the next kernel of the merge may start launching
    grid_dependency_wait();    // the previous kernel's results are visible
    const int64_t nu = static_cast<int64_t>(k) * l * r;
    const bool staged = nu <= kFsStageFloats;
    if (staged) {
        for (int e = threadIdx.x; e < nu; e += blockDim.x) su[e] = bd_in(kBkMsApply, e, nu) ? Uk[e] : 0.0f;
        __syncthreads();
    }
    const float* U = staged ? su : Uk;
    const int lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    for (int64_t gr = static_cast<int64_t>(blockIdx.x) * wpb + (threadIdx.x >> 5); gr < d_out + d_in;
         gr += static_cast<int64_t>(gridDim.x) * wpb) {
        const int side = gr < d_out ? 0 : 1;
        const int64_t n = side ? gr - d_out : gr;
        const int64_t rows = side ? d_in : d_out;
        const float* src = side ? Zall : Yall;
        uint16_t* dst = side ? Rs : Ls;
        const int64_t nsrc = static_cast<int64_t>(k) * rows * l, ndst = rows * Kp;
        for (int E = lane; E < K; E += 32) {
            const int z = E / r, e = E - z * r;
            const int64_t so = (static_cast<int64_t>(z) * rows + n) * l;
            const int64_t uo = static_cast<int64_t>(z) * l * r + e;
            float sv[kMaxL];  // the row of the basis, l <= kMaxL values (l is a multiple of 4)
#pragma unroll
            for (int c4 = 0; c4 < kMaxL / 4; ++c4) {
                const float4 v = 4 * c4 < l && bd_in_range(kBkMsApply, so + 4 * c4, 4, nsrc)
                                     ? *reinterpret_cast<const float4*>(src + so + 4 * c4)
                                     : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                sv[4 * c4] = v.x;
                sv[4 * c4 + 1] = v.y;
                sv[4 * c4 + 2] = v.z;
                sv[4 * c4 + 3] = v.w;
            }
            float acc = 0.0f;
#pragma unroll
            for (int c = 0; c < kMaxL; ++c) {
                if (c >= l) break;
                const int64_t ui = uo + static_cast<int64_t>(c) * r;
                acc = fmaf(sv[c], bd_in(kBkMsApply, ui, nu) ? U[ui] : 0.0f, acc);
            }
            const uint32_t b1 = __float_as_uint(acc) & 0xFFFF0000u;
            const float r1 = __fsub_rn(acc, __uint_as_float(b1));
            const uint32_t b2 = __float_as_uint(r1) & 0xFFFF0000u;
            const float r2 = __fsub_rn(r1, __uint_as_float(b2));
            const uint16_t p0 = static_cast<uint16_t>(b1 >> 16), p1 = static_cast<uint16_t>(b2 >> 16),
                           p2 = static_cast<uint16_t>(__float_as_uint(r2) >> 16);
#pragma unroll
            for (int pr = 0; pr < kMgPairs; ++pr) {
                const int64_t di = n * Kp + static_cast<int64_t>(pr) * K + E;
                const int mp = merge_piece(pr, side);
                if (bd_in(kBkMsSplit, di, ndst)) dst[di] = mp == 0 ? p0 : (mp == 1 ? p1 : p2);
            }
        }
        for (int kk = kMgPairs * K + lane; kk < Kp; kk += 32)
            if (bd_in(kBkMsSplit, n * Kp + kk, ndst)) dst[n * Kp + kk] = 0;
    }
}

struct MergeParams {
    CUtensorMap a_map;  // Ls [d_out][Kp] bf16, box 64 x 128, 128-byte swizzle
    CUtensorMap b_map;  // Rs [d_in][Kp] bf16, box 64 x 256, 128-byte swizzle
    CUtensorMap w_map;  // W_base [d_out][d_in] bf16, box 64 x 128, 128-byte swizzle
    const uint16_t* wb;
    void* out;
    uint32_t* err;      // the error word: a wait that timed out sets kErrTimeout
    int64_t d_out, d_in;
    int nk;             // Kp / 64 (0: rank 0, out = W_base)
    int ncb, ntiles;    // column tiles, tiles
    float inv_k;
    int out_f32;
};

__global__ void __launch_bounds__(kMgThreads, 1) merge_tc_kernel(const __grid_constant__ MergeParams p)
{
    extern __shared__ uint8_t dyn_raw[];
    __shared__ uint64_t full[kMgStages], empty[kMgStages];
    __shared__ uint64_t accfull[2], accempty[2], done;
    __shared__ uint64_t wfull[kMgWBufs], wfree[kMgWBufs];  // a tile's W_base block landed / the epilogue is done with it
    __shared__ uint32_t tmem_base;
    __shared__ volatile int abort;
    uint8_t* ring = dyn_raw + ((1024u - (smem_u32(dyn_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nk = p.nk;
    const int c0 = static_cast<int>(blockIdx.x), G = static_cast<int>(gridDim.x);
    if (tid == 0) {
        for (int st = 0; st < kMgStages; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&accfull[b], 1);
            mbar_init(&accempty[b], 8);  // the eight epilogue warps
        }
        mbar_init(&done, 1);
        for (int b = 0; b < kMgWBufs; ++b) {
            mbar_init(&wfull[b], 1);
            mbar_init(&wfree[b], 8);  // the eight epilogue warps
        }
        abort = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) tmem_alloc(&tmem_base, kMgTmemCols);
    uint8_t* wtiles = ring + static_cast<size_t>(kMgStages) * kMgStage;  // [kMgWBufs][4 boxes][128 rows][128 B]
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    grid_launch_dependents();
    grid_dependency_wait();    // the factors split by the previous kernels are visible
    const uint32_t tmem = tmem_base;
    auto wait = [&](uint64_t* bar, uint32_t par) {
        if (mbar_try_wait(bar, par)) return true;
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(bar, par)) {
            if (abort) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                abort = 1;
                raise_error(p.err, kErrTimeout);
                return false;
            }
        }
        return true;
    };
    if (warp == 10) {
        // ------------------------------------------------------------ W_base blocks, two buffers
        if (lane == 0) {
            int j = 0;
            for (int tile = c0; tile < p.ntiles; tile += G, ++j) {
                const int wb = j % kMgWBufs;
                // buffer wb is free once the epilogue is done with tile j - kMgWBufs
                if (j >= kMgWBufs && !wait(&wfree[wb], static_cast<uint32_t>(j / kMgWBufs - 1) & 1u)) break;
                const int rb = tile / p.ncb, cb = tile - rb * p.ncb;
                uint8_t* wt = wtiles + static_cast<size_t>(wb) * kMgWTile;
                mbar_arrive_expect_tx(&wfull[wb], static_cast<uint32_t>(kMgWTile));
#pragma unroll
                for (int bx = 0; bx < kMgN / 64; ++bx)  // columns past d_in read the fill value, never stored
                    tma_load_2d(wt + bx * (kMgWTile / 4), &p.w_map, cb * kMgN + 64 * bx, rb * kMgM, &wfull[wb]);
            }
            for (int i = (j > kMgWBufs ? j - kMgWBufs : 0); i < j; ++i) {  // the last blocks land before the CTA ends
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(&wfull[i % kMgWBufs], static_cast<uint32_t>(i / kMgWBufs) & 1u) &&
                       global_timer_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
    } else if (warp == 0) {
        // ------------------------------------------------------------ TMA producer (one k-step counter g over all tiles)
        if (lane == 0) {
            int g = 0;
            bool ok = true;
            for (int tile = c0; tile < p.ntiles && ok; tile += G) {
                const int rb = tile / p.ncb, cb = tile - rb * p.ncb;
                for (int t = 0; t < nk; ++t, ++g) {
                    const int st = g % kMgStages;
                    if (g >= kMgStages && !wait(&empty[st], static_cast<uint32_t>(g / kMgStages - 1) & 1u)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sb = ring + static_cast<size_t>(st) * kMgStage;
                    mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(kMgStage));
                    tma_load_2d(sb, &p.a_map, 64 * t, rb * kMgM, &full[st]);
                    tma_load_2d(sb + kMgATile, &p.b_map, 64 * t, cb * kMgN, &full[st]);
                }
            }
            for (int i = (g > kMgStages ? g - kMgStages : 0); i < g; ++i) {  // every issued copy lands before exit
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(&full[i % kMgStages], static_cast<uint32_t>(i / kMgStages) & 1u) &&
                       global_timer_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(kMgM, kMgN);
            int g = 0, j = 0;
            bool ok = true;
            for (int tile = c0; tile < p.ntiles && ok; tile += G, ++j) {
                const int b = j & 1;
                // accumulator b is free once the epilogue has read tile j - 2
                if (j >= 2 && !wait(&accempty[b], static_cast<uint32_t>(j / 2 - 1) & 1u)) break;
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(b * kMgN);
                for (int t = 0; t < nk; ++t, ++g) {
                    const int st = g % kMgStages;
                    if (!wait(&full[st], static_cast<uint32_t>(g / kMgStages) & 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sb = smem_u32(ring + static_cast<size_t>(st) * kMgStage);
                    const uint64_t adesc = smem_desc_sw128(sb), bdesc = smem_desc_sw128(sb + kMgATile);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_ss(d, adesc + static_cast<uint64_t>(2 * kk), bdesc + static_cast<uint64_t>(2 * kk), idesc,
                               (t | kk) != 0 ? 1u : 0u);
                    mma_commit(&empty[st]);
                }
                if (ok) mma_commit(&accfull[b]);  // tile j's accumulator is complete
            }
            mma_commit(&done);  // every MMA issued above has finished when this arrives
        }
    } else if (warp < 10) {
        // ------------------------------------------------------------ epilogue: one row per thread, columns
        // 128 hc .. 128 hc + 127 of the tile in chunks of 32
        const int q = warp & 3, hc = (warp - 2) >> 2;
        const int rl = 32 * q + lane;
        int j = 0;
        for (int tile = c0; tile < p.ntiles; tile += G, ++j) {
            const int b = j & 1;
            const int wb = j % kMgWBufs;
            if (!__all_sync(0xffffffffu, wait(&accfull[b], static_cast<uint32_t>(j / 2) & 1u) &&
                                             wait(&wfull[wb], static_cast<uint32_t>(j / kMgWBufs) & 1u)))
                break;
            const uint8_t* wtile = wtiles + static_cast<size_t>(wb) * kMgWTile;
            tc_fence_after();
            const int rb = tile / p.ncb, cb = tile - rb * p.ncb;
            const int64_t row = static_cast<int64_t>(rb) * kMgM + rl;
            const bool live = row < p.d_out;
            const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(b * kMgN) +
                                   128u * hc;
            const int64_t cbase = static_cast<int64_t>(cb) * kMgN + 128 * hc;
            const int nch =
                cbase >= p.d_in ? 0 : static_cast<int>((p.d_in - cbase < 128 ? p.d_in - cbase : 128) / 32);
#pragma unroll 1
            for (int ch = 0; ch < nch; ++ch) {
                uint32_t v[32];
                tmem_ld32(taddr + 32 * ch, v);
                if (!live) continue;
                const int64_t col = cbase + 32 * ch;
                const int cl = 128 * hc + 32 * ch;  // column within the tile
                const uint8_t* wbox = wtile + (cl >> 6) * (kMgWTile / 4) + rl * 128;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int chunk = ((cl & 63) >> 3) + c;  // 16-byte chunk of the 128-byte box row
                    const uint4 w = *reinterpret_cast<const uint4*>(wbox + ((chunk ^ (rl & 7)) << 4));
                    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
                    float o[8];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float a0 = nk > 0 ? __uint_as_float(v[8 * c + 2 * u]) : 0.0f;
                        const float a1 = nk > 0 ? __uint_as_float(v[8 * c + 2 * u + 1]) : 0.0f;
                        o[2 * u] = bf16_bits_to_float(wv[u] & 0xFFFFu) + p.inv_k * a0;
                        o[2 * u + 1] = bf16_bits_to_float(wv[u] >> 16) + p.inv_k * a1;
                    }
                    if (!bd_in_range(kBkMsMerge, row * p.d_in + col + 8 * c, 8, p.d_out * p.d_in)) continue;
                    if (p.out_f32) {
                        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + row * p.d_in + col + 8 * c);
                        dst[0] = make_float4(o[0], o[1], o[2], o[3]);
                        dst[1] = make_float4(o[4], o[5], o[6], o[7]);
                    } else {
                        uint32_t ob[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const __nv_bfloat162 h = __floats2bfloat162_rn(o[2 * u], o[2 * u + 1]);
                            ob[u] = *reinterpret_cast<const uint32_t*>(&h);
                        }
                        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + row * p.d_in + col + 8 * c) =
                            make_uint4(ob[0], ob[1], ob[2], ob[3]);
                    }
                }
            }
            // this warp has read its part of accumulator b and of the W_base block
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&accempty[b]);
                mbar_arrive(&wfree[wb]);
            }
        }
    }
    // tensor memory is freed only after every MMA issued has finished
    if (warp == 1 && lane == 0) {
        const uint64_t t0 = global_timer_ns();
        while (!mbar_try_wait(&done, 0u) && global_timer_ns() - t0 < kWaitLimitNs) {
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kMgTmemCols);
    }
}

size_t up256(size_t b) { return (b + 255) / 256 * 256; }

struct MonoSoupWs {
    size_t y, z, ypart, zpart, part, g, gk, m, uk, L, Rt, sp, ls, rs, total;
};

MonoSoupWs ws_layout(int64_t d_out, int64_t d_in, int k, int r, int l)
{
    MonoSoupWs w{};
    size_t off = 256;  // the asynchronous error word (a product or merge wait that timed out)
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += up256(bytes);
        return at;
    };
    w.y = take(static_cast<size_t>(k) * d_out * l * 4);  // Q_i of every checkpoint
    w.z = take(static_cast<size_t>(k) * d_in * l * 4);   // B_i^T of every checkpoint
    w.ypart = take(static_cast<size_t>(kSlices) * d_out * l * 4);
    w.zpart = take(static_cast<size_t>(kSlices) * d_in * l * 4);
    w.part = take(static_cast<size_t>(kGramParts) * l * l * 8);   // Gram partials of a batch (float2)
    w.g = take(static_cast<size_t>(kMaxBatch) * l * l * 8);       // Gram matrices of a batch (float2)
    w.gk = take(static_cast<size_t>(k) * l * l * 8);              // B_i B_i^T of every checkpoint (float2)
    w.m = take(static_cast<size_t>(kMaxBatch) * (kMaxL * kMaxL + kMaxL) * 4);  // R and 1/diag(R) of a batch
    w.uk = take(static_cast<size_t>(k) * l * (r > 0 ? r : 1) * 4);
    w.L = take(static_cast<size_t>(k) * d_out * (r > 0 ? r : 1) * 4);
    w.Rt = take(static_cast<size_t>(k) * d_in * (r > 0 ? r : 1) * 4);
    // split small operands of a batch for the tensor-core products (l <= 32)
    const size_t kp = static_cast<size_t>(((d_in > d_out ? d_in : d_out) + 63) / 64 * 64);
    w.sp = take(l <= 32 ? static_cast<size_t>(kMaxBatch) * 128 * kp * 2 : 0);
    // the split factors of the merge: [rows][Kp] bf16, Kp = 6 k r rounded up to 64
    const size_t kpm = static_cast<size_t>((kMgPairs * k * (r > 0 ? r : 1) + 63) / 64 * 64);
    w.ls = take(static_cast<size_t>(d_out) * kpm * 2);
    w.rs = take(static_cast<size_t>(d_in) * kpm * 2);
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
    static std::atomic<size_t> s00[kHostMaxDevices], s01[kHostMaxDevices], s10[kHostMaxDevices], s11[kHostMaxDevices];
    cudaError_t e0 = ensure_dynamic_smem(reinterpret_cast<const void*>(dprod_kernel<0, 8>), dprod_smem<0, 8>(), s00);
    if (e0 == cudaSuccess)
        e0 = ensure_dynamic_smem(reinterpret_cast<const void*>(dprod_kernel<0, 16>), dprod_smem<0, 16>(), s01);
    if (e0 == cudaSuccess)
        e0 = ensure_dynamic_smem(reinterpret_cast<const void*>(dprod_kernel<1, 8>), dprod_smem<1, 8>(), s10);
    if (e0 == cudaSuccess)
        e0 = ensure_dynamic_smem(reinterpret_cast<const void*>(dprod_kernel<1, 16>), dprod_smem<1, 16>(), s11);
    static std::atomic<size_t> t0c[kHostMaxDevices], t1c[kHostMaxDevices];
    constexpr size_t kTSmem = static_cast<size_t>(kTStages) * kTStage + 1024;
    if (e0 == cudaSuccess) e0 = ensure_dynamic_smem(reinterpret_cast<const void*>(tprod_kernel<0>), kTSmem, t0c);
    if (e0 == cudaSuccess) e0 = ensure_dynamic_smem(reinterpret_cast<const void*>(tprod_kernel<1>), kTSmem, t1c);
    static std::atomic<size_t> mgc[kHostMaxDevices];
    constexpr size_t kMgSmem = static_cast<size_t>(kMgStages) * kMgStage + kMgWBufs * kMgWTile + 1024;
    static_assert(kMgSmem <= 227 * 1024, "merge shared memory");
    if (e0 == cudaSuccess) e0 = ensure_dynamic_smem(reinterpret_cast<const void*>(merge_tc_kernel), kMgSmem, mgc);
    static std::atomic<size_t> eic[kHostMaxDevices];
    if (e0 == cudaSuccess) e0 = ensure_dynamic_smem(reinterpret_cast<const void*>(eig_kernel), kEigSmem, eic);
    if (e0 != cudaSuccess) return e0;
    const MonoSoupWs lay = ws_layout(a.d_out, a.d_in, a.k, a.rank, a.l);
    char* w = static_cast<char*>(a.ws);
    float* Yall = reinterpret_cast<float*>(w + lay.y);
    float* Zall = reinterpret_cast<float*>(w + lay.z);
    float2* Gk = reinterpret_cast<float2*>(w + lay.gk);
    float* Uk = reinterpret_cast<float*>(w + lay.uk);
    float* Yp = reinterpret_cast<float*>(w + lay.ypart);
    float* Zp = reinterpret_cast<float*>(w + lay.zpart);
    float2* part = reinterpret_cast<float2*>(w + lay.part);
    float2* G = reinterpret_cast<float2*>(w + lay.g);
    float* M = reinterpret_cast<float*>(w + lay.m);
    float* L = reinterpret_cast<float*>(w + lay.L);
    float* Rt = reinterpret_cast<float*>(w + lay.Rt);
    uint16_t* Sp = reinterpret_cast<uint16_t*>(w + lay.sp);
    const int l = a.l, r = a.rank;
    const bool tc = l <= 32;  // tensor-core products
    const int64_t ll = static_cast<int64_t>(l) * l;
    // the two products with Delta: CTAs of 64 rows (or 32, l > 32) / 64
    // columns of Delta for each checkpoint of the batch, the reduction
    // dimension split in gridDim.y slices (so that every SM gets its resident
    // CTAs), the slices summed in order
    const int sms = a.sm_count > 0 ? a.sm_count : 152;
    static thread_local ProdParams pp_sk, pp_lf;
    const int sk_rows = l <= 32 ? 64 : 32;
    const int64_t rblocks = (a.d_out + sk_rows - 1) / sk_rows, cblocks = a.d_in / kPTile;
    // slices: the smallest count whose CTAs fill whole waves of resident CTAs
    // to within an eighth (else the count nearest three waves), at most
    // kSlices / nb over the nb checkpoints of a batch
    auto slices = [&](int64_t blocks, int64_t klen, int nb, int64_t* per) {
        const int64_t wave = tc ? static_cast<int64_t>(sms) : static_cast<int64_t>(prod_ctas<16>()) * sms;
        const int cap = kSlices / nb;
        int ns = 1;
        for (int c = 1; c <= cap; ++c) {
            const int64_t ctas = blocks * nb * c;
            const int64_t full = (ctas + wave - 1) / wave;
            if (ctas * 8 >= full * wave * 7 && ctas >= wave) {
                ns = c;
                break;
            }
            if (std::llabs(ctas - 3 * wave) < std::llabs(blocks * nb * ns - 3 * wave)) ns = c;
        }
        *per = ((klen + ns - 1) / ns + kPTile - 1) / kPTile * kPTile;
        return static_cast<int>((klen + *per - 1) / *per);
    };
    cudaError_t perr = cudaSuccess;
    // tensor maps of checkpoints i0 .. i0 + nb - 1; small(z) = the small operand of checkpoint z
    auto prep = [&](ProdParams& pr, int i0, int nb, auto small, int64_t small_rows, float* part, int64_t per,
                    int box_rows) {
        auto enc_w = [&](CUtensorMap* m, const uint16_t* src) {
            return encode_tma_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, src, static_cast<uint64_t>(a.d_in),
                                 static_cast<uint64_t>(a.d_out), static_cast<uint64_t>(a.d_in) * 2, kPTile,
                                 static_cast<uint32_t>(box_rows), CU_TENSOR_MAP_SWIZZLE_128B);
        };
        if (!enc_w(&pr.b_map, a.w_base)) return false;
        for (int z = 0; z < nb; ++z) {
            if (!enc_w(&pr.w_map[z], a.w_ft[i0 + z])) return false;
            if (!encode_tma_2d(&pr.s_map[z], CU_TENSOR_MAP_DATA_TYPE_FLOAT32, small(z), static_cast<uint64_t>(l),
                               static_cast<uint64_t>(small_rows), static_cast<uint64_t>(l) * 4,
                               static_cast<uint32_t>(l <= 32 ? 32 : 64), kPTile, CU_TENSOR_MAP_SWIZZLE_NONE))
                return false;
        }
        pr.part = part;
        pr.err = a.err;
        pr.d_out = a.d_out;
        pr.d_in = a.d_in;
        pr.l = l;
        pr.k_per = per;
        return true;
    };
    // tensor-core form: A = the split small operands (Sp), B = the pieces of Delta
    static thread_local TProdParams tp_sk, tp_lf;
    auto tprep = [&](TProdParams& pr, int i0, int nb, int64_t Kp, float* part, int64_t per, int box_rows) {
        auto enc_w = [&](CUtensorMap* m, const uint16_t* src) {
            return encode_tma_2d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, src, static_cast<uint64_t>(a.d_in),
                                 static_cast<uint64_t>(a.d_out), static_cast<uint64_t>(a.d_in) * 2, kTK,
                                 static_cast<uint32_t>(box_rows), CU_TENSOR_MAP_SWIZZLE_128B);
        };
        if (!enc_w(&pr.b_map, a.w_base)) return false;
        for (int z = 0; z < nb; ++z) {
            if (!enc_w(&pr.w_map[z], a.w_ft[i0 + z])) return false;
            if (!encode_tma_2d(&pr.s_map[z], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Sp + static_cast<size_t>(z) * 128 * Kp,
                               static_cast<uint64_t>(Kp), 128, static_cast<uint64_t>(Kp) * 2, kTK, kTNB,
                               CU_TENSOR_MAP_SWIZZLE_128B))
                return false;
        }
        pr.part = part;
        pr.err = a.err;
        pr.d_out = a.d_out;
        pr.d_in = a.d_in;
        pr.l = l;
        pr.k_per = per;
        return true;
    };
    // a product's output still in K slices, summed by the next Gram pass over dst
    struct PendingSlices {
        const float* src = nullptr;
        int ns = 1;
        float* dst = nullptr;
    } pend;
    bool sp_ready = false;  // the last CholeskyQR pass wrote the next product's split operand
    const int64_t tr_blocks = (a.d_out + kTM - 1) / kTM, tc_blocks = a.d_in / kTM;
    // the tensor-core products run one persistent CTA per SM over their units
    auto persistent_ctas = [&](int64_t units) {
        return static_cast<unsigned>(units < sms ? units : sms);
    };
    // Y_z = Delta_z S_z for the batch (S_z = Omega, or Z_z with zs)
    auto sketch = [&](int i0, int nb, bool zs) {
        if (perr != cudaSuccess) return;
        int64_t per = 0;
        if (tc) {
            const int ns = slices(tr_blocks, a.d_in, nb, &per);
            const int64_t kp = (a.d_in + 63) / 64 * 64;
            if (!zs || !sp_ready)  // after a CholeskyQR pass the split is already written
                launch_dep(perr, split_small_kernel, dim3(static_cast<unsigned>((kp / 8 + 31) / 32), static_cast<unsigned>(nb)), 256, 0, st, zs ? Zall + static_cast<size_t>(i0) * a.d_in * l : a.omega,
                zs ? static_cast<int64_t>(a.d_in) * l : 0, a.d_in, kp, l, Sp);
            if (!tprep(tp_sk, i0, nb, kp, Yp, per, kTM)) {
                perr = cudaErrorInvalidValue;
                return;
            }
            tp_sk.nz = nb;
            tp_sk.ns = ns;
            tp_sk.tiles = static_cast<int>(tr_blocks * nb);
            launch_dep(perr, tprod_kernel<0>, dim3(persistent_ctas(tr_blocks * nb * ns)), kTThreads, kTSmem, st, tp_sk);
            pend = {Yp, ns, Yall + static_cast<size_t>(i0) * a.d_out * l};  // summed by the next Gram pass
            sp_ready = false;
            return;
        }
        const int ns = slices(rblocks, a.d_in, nb, &per);
        auto small = [&](int z) -> const float* {
            return zs ? Zall + static_cast<size_t>(i0 + z) * a.d_in * l : a.omega;
        };
        if (!prep(pp_sk, i0, nb, small, a.d_in, Yp, per, sk_rows)) {
            perr = cudaErrorInvalidValue;
            return;
        }
        const dim3 g(static_cast<unsigned>(rblocks), static_cast<unsigned>(ns), static_cast<unsigned>(nb));
        if (l <= 32)
            launch_dep(perr, dprod_kernel<0, 8>, g, kPThreads, dprod_smem<0, 8>(), st, pp_sk);
        else
            launch_dep(perr, dprod_kernel<0, 16>, g, kPThreads, dprod_smem<0, 16>(), st, pp_sk);
        pend = {Yp, ns, Yall + static_cast<size_t>(i0) * a.d_out * l};
    };
    // Z_z = Delta_z^T Y_z for the batch
    auto left = [&](int i0, int nb) {
        if (perr != cudaSuccess) return;
        int64_t per = 0;
        if (tc) {
            const int ns = slices(tc_blocks, a.d_out, nb, &per);
            const int64_t kp = (a.d_out + 63) / 64 * 64;
            if (!sp_ready)  // after a CholeskyQR pass the split is already written
                launch_dep(perr, split_small_kernel, dim3(static_cast<unsigned>((kp / 8 + 31) / 32), static_cast<unsigned>(nb)), 256, 0, st, Yall + static_cast<size_t>(i0) * a.d_out * l, static_cast<int64_t>(a.d_out) * l, a.d_out, kp, l, Sp);
            if (!tprep(tp_lf, i0, nb, kp, Zp, per, 64)) {
                perr = cudaErrorInvalidValue;
                return;
            }
            tp_lf.nz = nb;
            tp_lf.ns = ns;
            tp_lf.tiles = static_cast<int>(tc_blocks * nb);
            launch_dep(perr, tprod_kernel<1>, dim3(persistent_ctas(tc_blocks * nb * ns)), kTThreads, kTSmem, st, tp_lf);
            pend = {Zp, ns, Zall + static_cast<size_t>(i0) * a.d_in * l};
            sp_ready = false;
            return;
        }
        const int ns = slices(cblocks, a.d_out, nb, &per);
        auto small = [&](int z) -> const float* { return Yall + static_cast<size_t>(i0 + z) * a.d_out * l; };
        if (!prep(pp_lf, i0, nb, small, a.d_out, Zp, per, kPTile)) {
            perr = cudaErrorInvalidValue;
            return;
        }
        const dim3 g(static_cast<unsigned>(cblocks), static_cast<unsigned>(ns), static_cast<unsigned>(nb));
        if (l <= 32)
            launch_dep(perr, dprod_kernel<1, 8>, g, kPThreads, dprod_smem<1, 8>(), st, pp_lf);
        else
            launch_dep(perr, dprod_kernel<1, 16>, g, kPThreads, dprod_smem<1, 16>(), st, pp_lf);
        pend = {Zp, ns, Zall + static_cast<size_t>(i0) * a.d_in * l};
    };
    // out_z = A_z^T A_z for the nb consecutive A_z [n][l]
    // the upper triangle's l (l + 1) / 2 entries: one per thread up to
    // kGramThreads1 threads (two CTAs per SM), else 2 or 3 per thread
    const int npairs = l * (l + 1) / 2;
    const int gent = npairs <= kGramThreads1 ? 1 : (npairs <= 2 * kGramThreads ? 2 : 3);
    const int gthreads = ((npairs + gent - 1) / gent + 31) / 32 * 32;
    // (a product's output still in K slices is summed by its first Gram pass,
    // which writes the sum to A)
    auto gram = [&](float* A, int64_t n, int nb, float2* out) {
        const int gb = kGramParts / nb;
        const dim3 g(static_cast<unsigned>(gb), static_cast<unsigned>(nb));
        const float* src = A;
        int nsl = 1;
        float* sum = nullptr;
        if (pend.dst == A) {
            src = pend.src;
            nsl = pend.ns;
            sum = A;
            pend = {};
        }
        if (gent == 1)
            launch_dep(perr, gram_kernel<1>, g, gthreads, 0, st, src, nsl, n, l, part, sum);
        else if (gent == 2)
            launch_dep(perr, gram_kernel<2>, g, gthreads, 0, st, src, nsl, n, l, part, sum);
        else
            launch_dep(perr, gram_kernel<3>, g, gthreads, 0, st, src, nsl, n, l, part, sum);
        launch_dep(perr, gram_sum_kernel, dim3(blocks_for(32 * ll), static_cast<unsigned>(nb)), 256, 0, st, part, gb, l, out);
    };
    // A_z <- A_z R_z^-1 (CholeskyQR), `passes` times: two (CholeskyQR2) for
    // the Q that B is projected on, one for the intermediate bases of the
    // power iterations, where only the spanned subspace matters
    // (on the tensor-core path the last pass also writes the split small
    // operand of the product that follows it)
    auto orth = [&](float* A, int64_t n, int nb, int passes) {
        for (int pass = 0; pass < passes; ++pass) {
            gram(A, n, nb, G);
            launch_dep(perr, chol_kernel, static_cast<unsigned>(nb), 256, 0, st, G, l, M);
            const bool split = tc && pass + 1 == passes;
            const int64_t kp = (n + 63) / 64 * 64, rows = split ? kp : n;
            launch_dep(perr, tri_solve_kernel, dim3(static_cast<unsigned>((rows + kTriThreads - 1) / kTriThreads), static_cast<unsigned>(nb)), kTriThreads, 0, st, A, n, l, static_cast<const float*>(M), split ? Sp : nullptr, kp);
            sp_ready = split;
        }
    };
    if (r > 0) {
        for (int i0 = 0; i0 < a.k; i0 += kMaxBatch) {
            const int nb = a.k - i0 < kMaxBatch ? a.k - i0 : kMaxBatch;
            float* Y = Yall + static_cast<size_t>(i0) * a.d_out * l;
            float* Z = Zall + static_cast<size_t>(i0) * a.d_in * l;
            sketch(i0, nb, false);
            orth(Y, a.d_out, nb, a.power_iters > 0 ? 1 : 2);
            for (int it = 0; it < a.power_iters; ++it) {
                left(i0, nb);
                orth(Z, a.d_in, nb, 1);
                sketch(i0, nb, true);
                orth(Y, a.d_out, nb, it + 1 == a.power_iters ? 2 : 1);
            }
            left(i0, nb);                                          // Z = B^T
            gram(Z, a.d_in, nb, Gk + static_cast<size_t>(i0) * ll);  // B B^T
        }
        // the k projected eigenproblems at once, one CTA each
        launch_dep(perr, eig_kernel, static_cast<unsigned>(a.k), kEigThreads, kEigSmem, st, static_cast<const float2*>(Gk), l, r, Uk);  // U_r [l][r]
    }
    if (perr != cudaSuccess) return perr;
    // the merge: split factors, then D = Ls Rs^T + W_base on the tensor cores
    const int K = r > 0 ? a.k * r : 0;
    const int Kp = (kMgPairs * (K > 0 ? K : 1) + 63) / 64 * 64;
    uint16_t* Ls = reinterpret_cast<uint16_t*>(w + lay.ls);
    uint16_t* Rs = reinterpret_cast<uint16_t*>(w + lay.rs);
    static thread_local MergeParams mp;
    if (K > 0) {
        const int64_t nu = static_cast<int64_t>(a.k) * l * r;
        const size_t fs_smem = nu <= kFsStageFloats ? static_cast<size_t>(nu) * 4 : 0;
        const int64_t fs_ctas = (a.d_out + a.d_in + 7) / 8;  // eight warps, each striding over the rows
        launch_dep(perr, factor_split_kernel, static_cast<unsigned>(fs_ctas < 2 * sms ? fs_ctas : 2 * sms), 256, fs_smem, st,
                   static_cast<const float*>(Yall), static_cast<const float*>(Zall), a.d_out, a.d_in, l, a.k, r,
                   static_cast<const float*>(Uk), K, Kp, Ls, Rs);
    }
    if (!encode_tma_2d(&mp.a_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Ls, static_cast<uint64_t>(Kp),
                       static_cast<uint64_t>(a.d_out), static_cast<uint64_t>(Kp) * 2, 64, kMgM,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tma_2d(&mp.b_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Rs, static_cast<uint64_t>(Kp),
                       static_cast<uint64_t>(a.d_in), static_cast<uint64_t>(Kp) * 2, 64, kMgN,
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tma_2d(&mp.w_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.w_base, static_cast<uint64_t>(a.d_in),
                       static_cast<uint64_t>(a.d_out), static_cast<uint64_t>(a.d_in) * 2, 64, kMgM,
                       CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    mp.wb = a.w_base;
    mp.out = a.out;
    mp.err = a.err;
    mp.d_out = a.d_out;
    mp.d_in = a.d_in;
    mp.nk = K > 0 ? Kp / 64 : 0;
    mp.inv_k = 1.0f / static_cast<float>(a.k);
    mp.out_f32 = a.out_f32;
    mp.ncb = static_cast<int>((a.d_in + kMgN - 1) / kMgN);
    mp.ntiles = mp.ncb * static_cast<int>((a.d_out + kMgM - 1) / kMgM);
    const int mg_grid = mp.ntiles < sms ? mp.ntiles : sms;  // persistent: one CTA per SM
    launch_dep(perr, merge_tc_kernel, mg_grid, kMgThreads, kMgSmem, st, mp);
    return perr != cudaSuccess ? perr : cudaGetLastError();
}

BD_BOUNDS_TAKE(bounds_take_monosoup)

}  // namespace bd
