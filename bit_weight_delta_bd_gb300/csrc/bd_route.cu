// Router for multi-variant batches (section "Sunum mimarisi" of the BitDelta
// post: the request router that sends each request to its variant's delta):
// a stable counting sort of token indices by key = vid + 1, where key 0 holds
// the base-model tokens (vid = -1) and any out-of-range id (flagged).
//
// One CTA of 1024 threads.  Pass 1 counts keys with shared-memory atomics
// (counts do not depend on order) and writes seg_off.  Pass 2 walks the
// tokens in 1024-token rounds: inside a warp, __match_any_sync finds the
// lanes holding the same key and the lane's rank among them; a per-key scan
// over the 32 warps of the round gives each warp's offset; a running base per
// key carries the count across rounds.  Positions are therefore exactly those
// of a stable sort.
#include "bd_device.cuh"

namespace bd {
namespace {

constexpr int kRouteThreads = 1024;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kKeys = kMaxVariants + 1;

__global__ void __launch_bounds__(kRouteThreads)
    route_kernel(const int32_t* __restrict__ vid, int64_t T, int V, int32_t* __restrict__ perm,
                 int32_t* __restrict__ seg_off, uint32_t* err)
{
    __shared__ int total[kKeys];
    __shared__ int running[kKeys];
    __shared__ int warp_cnt[kRouteWarps][kKeys];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n_keys = V + 1;
    grid_launch_dependents();  // a kernel launched after this one with programmatic dependent launch may start

    for (int k = tid; k < kKeys; k += kRouteThreads) total[k] = 0;
    __syncthreads();
    bool bad = false;
    for (int64_t t = tid; t < T; t += kRouteThreads) {
        const int v = vid[t];
        const bool ok = (v >= -1 && v < V);
        bad |= !ok;
        atomicAdd(&total[ok ? v + 1 : 0], 1);
    }
    if (__syncthreads_or(bad) && tid == 0) raise_error(err, kErrBadVariant);
    if (tid == 0) {
        int acc = 0;
        for (int k = 0; k < n_keys; ++k) {
            if (bd_in(kBkRoute, k, n_keys + 1)) seg_off[k] = acc;
            running[k] = acc;
            acc += total[k];
        }
        if (bd_in(kBkRoute, n_keys, n_keys + 1)) seg_off[n_keys] = acc;
    }
    __syncthreads();

    for (int64_t base = 0; base < T; base += kRouteThreads) {
        const int64_t t = base + tid;
        int key = -1;  // lanes past T take part in the warp vote with a key no token has
        if (t < T) {
            const int v = vid[t];
            key = (v >= -1 && v < V) ? v + 1 : 0;
        }
        for (int i = tid; i < kRouteWarps * kKeys; i += kRouteThreads) (&warp_cnt[0][0])[i] = 0;
        __syncthreads();
        const unsigned peers = __match_any_sync(0xffffffffu, key);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (key >= 0 && rank == 0) warp_cnt[warp][key] = __popc(peers);
        __syncthreads();
        if (tid < n_keys) {
            int run = running[tid];
            for (int w = 0; w < kRouteWarps; ++w) {
                const int c = warp_cnt[w][tid];
                warp_cnt[w][tid] = run;
                run += c;
            }
            running[tid] = run;
        }
        __syncthreads();
        if (key >= 0 && bd_in(kBkRoute, warp_cnt[warp][key] + rank, T))
            perm[warp_cnt[warp][key] + rank] = static_cast<int32_t>(t);
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_route(const int32_t* vid, int64_t T, int V, int32_t* perm, int32_t* seg_off, uint32_t* err,
                         cudaStream_t stream)
{
    route_kernel<<<1, kRouteThreads, 0, stream>>>(vid, T, V, perm, seg_off, err);
    return cudaGetLastError();
}

BD_BOUNDS_TAKE(bounds_take_route)

}  // namespace bd
