// Internal interface between the C ABI (bd_api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#ifndef BD_NO_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

namespace bd {

constexpr int kMaxVariants = 64;

// Launches a kernel with programmatic dependent launch: it may start
// launching while the previous kernel of the stream finishes.  The kernel
// must wait for that kernel (griddepcontrol.wait) before it touches device
// memory; kernels that also let their dependents launch at their start
// (griddepcontrol.launch_dependents) overlap the launch latency of the next
// kernel of a chain.  The first error is kept in err and no later kernel is
// launched.
template <typename... KArgs, typename... Args>
void launch_dep(cudaError_t& err, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                Args&&... args)
{
    if (err != cudaSuccess) return;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}


// An NVTX range around each compute entry point of the C ABI, named after
// the entry point, so that a profiler's timeline (or ncu --nvtx-include)
// groups the launches of one call.  NVTX v3 is header-only: with no tool
// attached a push or a pop tests one function pointer.  -DBD_NO_NVTX leaves
// the ranges out.
#ifndef BD_NO_NVTX
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};
#define BD_NVTX_RANGE(name) const ::bd::NvtxRange bd_nvtx_range_(name)
#else
#define BD_NVTX_RANGE(name) static_cast<void>(0)
#endif

// Maps a CUDA runtime result to a library status: cudaSuccess -> 0
// (BD_OK), anything else -> BD_ERR_CUDA, with the code kept as the calling
// thread's last CUDA error (bd_last_cuda_error).
int cuda_status(cudaError_t e);

// ---- compression (bd_compress.cu) -------------------------------------------------------------

// Rows handled by one compression CTA (one warp per row).
constexpr int kCompressRowsPerCta = 4;

cudaError_t launch_compress(const uint16_t* w_base, const uint16_t* w_ft, int64_t d_out, int64_t d_in, bool per_row,
                            uint32_t* signs, float* alpha, double* partials, uint32_t* err, cudaStream_t stream);

cudaError_t launch_debug_reconstruct(const uint16_t* w_base, const uint32_t* signs, const float* alpha, bool per_row,
                                     int64_t d_out, int64_t d_in, float* w_eff, cudaStream_t stream);

// ---- decode linear, one variant (bd_skinny.cu) ------------------------------------------------

// Tokens one decode launch covers (8 MMA n-tiles of 8 tokens); also the
// token group of the multi-variant linear.
constexpr int kSkinnyMaxTokens = 64;

struct SkinnyArgs {
    const uint16_t* x;        // [T][d_in] bf16 bits
    const uint16_t* w_base;   // [d_out][d_in]
    const uint32_t* signs;    // [d_out][d_in/32]
    const float* alpha;       // [d_out] or [1]
    int64_t T, d_out, d_in;
    int per_row;
    void* y;                  // [T][d_out]
    int out_f32;
    uint32_t* err;
};

cudaError_t launch_skinny(const SkinnyArgs& a, cudaStream_t stream);

// ---- multi-variant linear (bd_multi.cu) -------------------------------------------------------

struct MultiArgs {
    const uint16_t* x;        // [T][d_in] bf16 bits, T <= kSkinnyMaxTokens
    const int32_t* vid;       // [T]
    const uint16_t* w_base;   // [d_out][d_in]
    int64_t T, d_out, d_in;
    int V;
    int per_row;
    const uint32_t* signs[kMaxVariants];
    const float* alpha[kMaxVariants];
    void* y;                  // [T][d_out]
    int out_f32;
    uint32_t* err;
    uint8_t* xp;              // scratch [multi_max_ptiles(T, V)][8][d_in] bf16: padded per-variant tiles
    float* corr;              // scratch [T][multi_corr_splits(d_in)]: partial corrections of the recoded sign sums
};

// Upper bound of the zero-padded 8-token tiles of a group of T tokens over V
// variants: sum over variants of ceil(n_v / 8) <= (T + 7 min(T, V)) / 8.
int multi_max_ptiles(int T, int V);

// Tokens per multi-variant launch for V variants: 64, or fewer when a group
// could need more zero-padded tiles than tensor memory holds.
int multi_group_tokens(int V);

// Column splits of the prepare pass (partial corrections per token).
int multi_corr_splits(int64_t d_in);

cudaError_t launch_multi(const MultiArgs& a, cudaStream_t stream);

// ---- materialised variant (bd_materialize.cu) -------------------------------------------------

cudaError_t launch_materialize(const uint16_t* w_base, const uint32_t* signs, const float* alpha, int per_row,
                               int64_t d_out, int64_t d_in, uint16_t* w_eff, int sm_count, cudaStream_t stream);

// ---- router (bd_route.cu) ---------------------------------------------------------------------

cudaError_t launch_route(const int32_t* vid, int64_t T, int V, int32_t* perm, int32_t* seg_off, uint32_t* err,
                         cudaStream_t stream);

// ---- prefill GEMM (bd_prefill.cu) -------------------------------------------------------------

struct PrefillArgs {
    const uint16_t* x;        // [T][d_in]
    const uint16_t* w_base;   // [d_out][d_in]
    const uint32_t* signs;    // [d_out][d_in/32]
    const float* alpha;
    int per_row;
    int64_t T, d_out, d_in;
    void* y;
    int out_f32;
    uint32_t* err;
};

bool prefill_available();
cudaError_t launch_prefill(const PrefillArgs& a, int sm_count, cudaStream_t stream);

// Multi-variant prefill on the tensor cores: tokens routed by bd_route's
// perm / seg_off, x gathered into sorted order, one prefill tile per
// (256-token block inside one variant's segment, 128 rows).
struct GroupedPrefillArgs {
    const uint16_t* x;            // [T][d_in] caller order
    const int32_t* perm;          // [T] sorted position -> caller token (bd_route)
    const int32_t* seg_off;       // [V + 2] (bd_route)
    const uint16_t* w_base;       // [d_out][d_in]
    const uint32_t* signs[kMaxVariants];
    const float* alpha[kMaxVariants];
    int V, per_row;
    int64_t T, d_out, d_in;
    void* y;                      // [T][d_out] caller order
    int out_f32;
    uint32_t* err;
    uint16_t* xs;                 // scratch [T][d_in]: x in sorted order
    int4* plan;                   // scratch [grouped_prefill_blocks(T, V)]
};

// Upper bound of the 256-token blocks of a grouped prefill: ceil(T / 256) + V + 1.
int grouped_prefill_blocks(int64_t T, int V);

// ---- MonoSoup merge (bd_monosoup.cu) ---------------------------------------------------------

struct MonoSoupArgs {
    const uint16_t* w_base;        // [d_out][d_in] bf16 bits
    const uint16_t* const* w_ft;   // host array of k device pointers, each [d_out][d_in]
    int k;
    int64_t d_out, d_in;
    int rank, l, power_iters;
    const float* omega;            // [d_in][l] Gaussian test matrix (rank > 0)
    void* out;                     // [d_out][d_in] bf16 or fp32
    int out_f32;
    void* ws;                      // monosoup_workspace_size bytes
    uint32_t* err;                 // the asynchronous error word (start of ws)
    int sm_count;                  // SMs of the current device
};

// bounds-checked builds: the flag words of each translation unit, read and
// cleared (0 in normal builds)
uint32_t bounds_take_compress();
uint32_t bounds_take_skinny();
uint32_t bounds_take_multi();
uint32_t bounds_take_prefill();
uint32_t bounds_take_route();
uint32_t bounds_take_materialize();
uint32_t bounds_take_monosoup();

int monosoup_max_l();
size_t monosoup_workspace_size(int64_t d_out, int64_t d_in, int k, int r, int l);
cudaError_t launch_monosoup(const MonoSoupArgs& a, cudaStream_t stream);
cudaError_t launch_prefill_grouped(const GroupedPrefillArgs& a, cudaStream_t stream);

}  // namespace bd
