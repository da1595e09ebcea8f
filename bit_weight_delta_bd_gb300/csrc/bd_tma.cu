// TMA tensor-map encoding (see bd_tma.h).
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "bd_tma.h"

namespace bd {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

struct MapKey {
    uintptr_t base;
    uint64_t cols, rows, row_bytes;
    uint32_t box_cols, box_rows;
    int dtype, swizzle;
    bool operator==(const MapKey& o) const
    {
        return base == o.base && cols == o.cols && rows == o.rows && row_bytes == o.row_bytes &&
               box_cols == o.box_cols && box_rows == o.box_rows && dtype == o.dtype && swizzle == o.swizzle;
    }
};

struct MapKeyHash {
    size_t operator()(const MapKey& k) const
    {
        uint64_t h = 1469598103934665603ull;
        const uint64_t v[8] = {static_cast<uint64_t>(k.base), k.cols, k.rows, k.row_bytes, k.box_cols, k.box_rows,
                               static_cast<uint64_t>(k.dtype), static_cast<uint64_t>(k.swizzle)};
        for (uint64_t x : v) h = (h ^ x) * 1099511628211ull;
        return static_cast<size_t>(h);
    }
};

constexpr size_t kMapCacheMax = 4096;

}  // namespace

bool encode_tma_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t cols, uint64_t rows,
                   uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle)
{
    thread_local std::unordered_map<MapKey, CUtensorMap, MapKeyHash> cache;
    const MapKey key{reinterpret_cast<uintptr_t>(base), cols, rows, row_bytes, box_cols, box_rows,
                     static_cast<int>(dtype), static_cast<int>(swizzle)};
    auto it = cache.find(key);
    if (it != cache.end()) {
        std::memcpy(map, &it->second, sizeof(CUtensorMap));
        return true;
    }
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t elem[2] = {1, 1};
    if (fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    if (cache.size() >= kMapCacheMax) cache.clear();
    cache.emplace(key, *map);
    return true;
}

cudaError_t ensure_dynamic_smem(const void* kernel, size_t bytes, std::atomic<size_t>* per_device)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kHostMaxDevices) return cudaErrorInvalidDevice;
    if (per_device[dev].load(std::memory_order_acquire) >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e != cudaSuccess) return e;
    // all of the unified L1/shared storage as shared memory, so that as many
    // CTAs (and thread-block clusters) as the shared memory allows are resident
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess) per_device[dev].store(bytes, std::memory_order_release);
    return e;
}

}  // namespace bd
