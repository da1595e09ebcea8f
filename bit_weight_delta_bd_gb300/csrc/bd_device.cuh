// Device-side helpers for the BitDelta kernels (sm_103a): shared-memory
// addresses, mbarriers with bounded waits, bulk async copies, the warp-level
// bf16 MMA, and the asynchronous error word.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bd_internal.h"

namespace bd {

// Bits of the asynchronous error word (bit n <=> bd_status n).
constexpr uint32_t kErrBadVariant = 1u << 4;
constexpr uint32_t kErrNonFinite = 1u << 5;
constexpr uint32_t kErrTimeout = 1u << 7;

// Bounded waits give up after this many nanoseconds of %globaltimer.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ void raise_error(uint32_t* err, uint32_t bits)
{
    if (err) atomicOr(err, bits);
}

// ---------------------------------------------------------------- bounds-checked builds
// With -DBD_DEBUG_BOUNDS the plain global loads and stores of the kernels are
// preceded by bd_in(kernel, i, n): true when 0 <= i < n; otherwise bit
// `kernel` of the translation unit's flag word is set and the caller skips
// the access (no trap).  bd_debug_bounds_check() reads and clears the flag
// words of every translation unit.  TMA copies need no check: the hardware
// fills the out-of-range elements of a load and drops them from a store.  In
// normal builds bd_in is the constant true.
enum BoundsKernel : uint32_t {
    kBkCompress = 0, kBkAlphaFinalize, kBkReconstruct, kBkSkinny, kBkMultiPrepare, kBkMulti, kBkPrefill,
    kBkPrefillPlan, kBkGather, kBkRoute, kBkMaterialize, kBkMsProd, kBkMsSplit, kBkMsSlices, kBkMsGram,
    kBkMsGramSum, kBkMsChol, kBkMsEig, kBkMsTri, kBkMsApply, kBkMsMerge
};
#ifdef BD_DEBUG_BOUNDS
namespace {
__device__ uint32_t g_bounds_flags = 0;  // one word per translation unit
}
__device__ __forceinline__ bool bd_in(uint32_t kernel, int64_t i, int64_t n)
{
    if (i >= 0 && i < n) return true;
    atomicOr(&g_bounds_flags, 1u << kernel);
    return false;
}
// the range [i, i + len) lies in [0, n)
__device__ __forceinline__ bool bd_in_range(uint32_t kernel, int64_t i, int64_t len, int64_t n)
{
    if (i >= 0 && len >= 0 && i + len <= n) return true;
    atomicOr(&g_bounds_flags, 1u << kernel);
    return false;
}
// host: the flags of this translation unit, cleared (synchronises the device)
#define BD_BOUNDS_TAKE(fn)                                                \
    uint32_t fn()                                                         \
    {                                                                     \
        uint32_t v = 0, z = 0;                                            \
        if (cudaMemcpyFromSymbol(&v, g_bounds_flags, sizeof v) != cudaSuccess) return ~0u; \
        if (cudaMemcpyToSymbol(g_bounds_flags, &z, sizeof z) != cudaSuccess) return ~0u;   \
        return v;                                                         \
    }
#else
__device__ __forceinline__ constexpr bool bd_in(uint32_t, int64_t, int64_t) { return true; }
__device__ __forceinline__ constexpr bool bd_in_range(uint32_t, int64_t, int64_t, int64_t) { return true; }
#define BD_BOUNDS_TAKE(fn) \
    uint32_t fn() { return 0; }
#endif

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for the phase with the given parity to complete; gives up after
// kWaitLimitNs and returns false (the caller reports kErrTimeout).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
    return true;
}

// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy (bulk copy / TMA) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------- bulk async copies

// Global -> shared bulk copy completing on an mbarrier.  dst, src and bytes
// must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 2-D tiled TMA load (tensor map in param/const/global space) completing on
// an mbarrier.  c0 is the inner (contiguous) coordinate; c0 * element size
// must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// ------------------------------------------------------------ clusters

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster arrives and waits (release /
// acquire at cluster scope).
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrives on the mbarrier at the same shared-memory offset as `bar` in the
// cluster's CTA of rank `cta`, with the default (CTA-scope) release.  For
// signals whose data is already complete when the arrive is issued (tensor-
// memory stores waited for with tcgen05.wait::st, TMA data whose
// complete_tx was observed): a cluster-scope release would also make the
// SM drain its memory traffic in flight, which in a TMA-fed pipeline
// serialises the stage ring (2.4x the time of a 4096 x 8192 x 8192
// prefill on GB300).
__device__ __forceinline__ void mbar_arrive_remote(uint64_t* bar, uint32_t cta)
{
    asm volatile(
        "{\n\t.reg .b32 ra;\n\t"
        "mapa.shared::cluster.u32 ra, %0, %1;\n\t"
        "mbarrier.arrive.shared::cluster.b64 _, [ra];\n\t}" ::"r"(smem_u32(bar)),
        "r"(cta)
        : "memory");
}

// try_wait with acquire at cluster scope: pairs with arrivals made by other
// CTAs of the cluster (mbar_arrive_remote).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// ------------------------------------------------------------ warp MMA

// D += A * B, m16n8k16, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------ programmatic dependent launch
// In a kernel launched with programmatic stream serialization: wait until the
// preceding kernel of the stream has completed and its memory is visible
// (returns at once when the launch had no such dependency).
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// In the preceding kernel: allow the dependent kernel to start launching now.
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------ loads

// Read-only (non-coherent) 16-byte load of data that no kernel writes
// during the launch.
__device__ __forceinline__ uint4 ld_nc_v4(const void* p) { return __ldg(static_cast<const uint4*>(p)); }

// Streaming load (no L1 allocation): for data read exactly once.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}


}  // namespace bd
