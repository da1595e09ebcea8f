// bd_compress_noalloc: the compression entry point for callers that cannot
// allocate device memory (see include/bitdelta.h).  Its only scratch, the
// per-CTA partial sums of the per-matrix alpha, lives in a fixed-size device
// array of this library instead of a caller-provided workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/bitdelta.h"
#include "bd_internal.h"

namespace {

constexpr int64_t kMaxRows = BD_NOALLOC_MAX_ROWS;
static_assert(kMaxRows % bd::kCompressRowsPerCta == 0, "whole compression CTAs");
constexpr size_t kPartials = static_cast<size_t>(kMaxRows / bd::kCompressRowsPerCta);

// One fp64 partial sum per compression CTA (kCompressRowsPerCta = 4 rows):
// 65536 doubles.  Every GPU that loads the library holds these 512 KiB until
// the process exits.
static __device__ __align__(256) double g_noalloc_partials[kPartials];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
double* g_partials_addr[kMaxDevices];  // device address of g_noalloc_partials, per device

// Resolves (once per device, with that device current) the device address of
// the scratch array; host code must not use the array's name as a pointer.
bd_status scratch_for_current_device(double** out)
{
    int dev = 0;
    if (const int cs_ = bd::cuda_status(cudaGetDevice(&dev))) return static_cast<bd_status>(cs_);
    if (dev < 0 || dev >= kMaxDevices) return BD_ERR_DEVICE;
    int major = 0, minor = 0;
    cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (e != cudaSuccess) return static_cast<bd_status>(bd::cuda_status(e));
    if (major * 10 + minor != 103) return BD_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_partials_addr[dev] == nullptr) {
        void* p = nullptr;
        if (const int cs_ = bd::cuda_status(cudaGetSymbolAddress(&p, g_noalloc_partials)))
            return static_cast<bd_status>(cs_);
        if (p == nullptr) return BD_ERR_CUDA;
        g_partials_addr[dev] = static_cast<double*>(p);
    }
    *out = g_partials_addr[dev];
    return BD_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb)
{
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

}  // namespace

extern "C" bd_status bd_compress_noalloc(const uint16_t* w_base, const uint16_t* w_ft, int64_t d_out, int64_t d_in,
                                         int alpha_mode, uint32_t* signs, float* alpha, void* stream)
{
    BD_NVTX_RANGE("bd_compress_noalloc");
    if (alpha_mode != BD_ALPHA_PER_MATRIX && alpha_mode != BD_ALPHA_PER_ROW) return BD_ERR_INVALID_ARG;
    if (d_out < 0 || d_out > kMaxRows) return BD_ERR_UNSUPPORTED_SHAPE;
    if (d_in <= 0 || d_in % 128 != 0) return BD_ERR_UNSUPPORTED_SHAPE;
    if (d_out == 0) return BD_OK;
    if (!w_base || !w_ft || !signs || !alpha) return BD_ERR_INVALID_ARG;
    if (!aligned(w_base, 16) || !aligned(w_ft, 16) || !aligned(signs, 16) || !aligned(alpha, 4))
        return BD_ERR_MISALIGNED;
    const size_t wbytes = static_cast<size_t>(d_out) * d_in * 2;
    const size_t sbytes = static_cast<size_t>(d_out) * (d_in / 8);
    const size_t abytes = (alpha_mode == BD_ALPHA_PER_ROW ? static_cast<size_t>(d_out) : 1u) * 4;
    if (overlaps(signs, sbytes, w_base, wbytes) || overlaps(signs, sbytes, w_ft, wbytes) ||
        overlaps(alpha, abytes, w_base, wbytes) || overlaps(alpha, abytes, w_ft, wbytes) ||
        overlaps(signs, sbytes, alpha, abytes))
        return BD_ERR_INVALID_ARG;
    double* partials = nullptr;
    if (bd_status s = scratch_for_current_device(&partials)) return s;
    // Every CTA overwrites its own partial and the final sum reads only those,
    // so nothing in the scratch has to be cleared between calls.  No error
    // word: a non-finite delta shows up as a non-finite alpha.
    const cudaError_t e = bd::launch_compress(w_base, w_ft, d_out, d_in, alpha_mode == BD_ALPHA_PER_ROW, signs,
                                              alpha, partials, nullptr, static_cast<cudaStream_t>(stream));
    return static_cast<bd_status>(bd::cuda_status(e));
}
