// Delta cache (section "Altyapı ayrıntıları" of the BitDelta post: cold
// start, request-rate-weighted LRU eviction with the most requested variants
// pinned, and per-variant queueing while a delta loads), host side only.
//
// The cache divides a caller-owned device arena into equal slots; each slot
// holds one variant's delta blob (whatever the caller packs: signs and alpha
// of one or more linears).  A serving step hands the cache the variant ids of
// its requests:
//   - every id's request rate is r = r * decay + (requests this step);
//   - the n_pinned registered variants with the highest rate (ties: lower id)
//     are pinned: their slots are never evicted;
//   - a requested variant that is resident is a hit; one that is not is
//     loaded once (one host -> device copy on the copy stream, however many
//     requests ask for it) into a free slot or, failing that, into the least
//     recently used slot whose variant is neither pinned nor used by this step;
//   - when no such slot exists the variant's requests are queued: the caller
//     keeps them for a later step;
//   - the compute stream waits for the copies of every slot the step uses (a
//     delta still loading from an earlier step is waited for, not reloaded),
//     and bd_cache_release records when the step's kernels are done with its
//     slots, which a later load of the same slot waits for on the copy stream.
// A cache created without an arena runs the same policy without any CUDA call
// and reports slot offsets instead of addresses (planning and tests).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>
#include <new>
#include <unordered_map>
#include <vector>

#include "../../include/bitdelta.h"
#include "bd_internal.h"

struct bd_cache {
    struct Slot {
        int32_t variant = -1;
        uint64_t last_use = 0;
        cudaEvent_t ready = nullptr;     // the slot's last copy finished
        cudaEvent_t released = nullptr;  // the last step using the slot finished
        bool released_recorded = false;
    };
    struct Source {
        const void* host = nullptr;
        size_t bytes = 0;
    };
    std::mutex mu;
    char* arena = nullptr;  // nullptr: dry run (no CUDA calls)
    size_t slot_bytes = 0;
    int32_t n_pinned = 0;
    double decay = 1.0;
    cudaStream_t copy = nullptr;
    std::vector<Slot> slots;
    std::unordered_map<int32_t, Source> src;
    std::unordered_map<int32_t, double> rate;
    std::unordered_map<int32_t, int> slot_of;  // resident variant -> slot
    std::vector<int32_t> pinned;               // current pinned set
    std::vector<int> acquired;                 // slots handed out by the pending step
    int64_t fail_countdown = 0;                // test aid: the n-th load from now fails (0: never)
    uint64_t tick = 0;
    bd_cache_stats st{};
};

namespace {

bool is_pinned(const bd_cache& c, int32_t v)
{
    return std::find(c.pinned.begin(), c.pinned.end(), v) != c.pinned.end();
}

// The n_pinned registered variants of highest rate (ties: lower id).
void update_pinned(bd_cache& c)
{
    std::vector<std::pair<double, int32_t>> r;
    r.reserve(c.src.size());
    for (const auto& kv : c.src) {
        const auto it = c.rate.find(kv.first);
        r.emplace_back(it == c.rate.end() ? 0.0 : it->second, kv.first);
    }
    std::sort(r.begin(), r.end(), [](const auto& a, const auto& b) {
        return a.first != b.first ? a.first > b.first : a.second < b.second;
    });
    c.pinned.clear();
    for (size_t i = 0; i < r.size() && static_cast<int32_t>(i) < c.n_pinned; ++i)
        if (r[i].first > 0.0) c.pinned.push_back(r[i].second);
}

// A slot for a variant that is not resident: a free one, else the least
// recently used slot whose variant is unpinned and not used by this step.
int find_slot(const bd_cache& c)
{
    int best = -1;
    for (int s = 0; s < static_cast<int>(c.slots.size()); ++s) {
        const auto& sl = c.slots[s];
        if (sl.variant < 0) return s;
        if (is_pinned(c, sl.variant)) continue;
        if (std::find(c.acquired.begin(), c.acquired.end(), s) != c.acquired.end()) continue;
        if (best < 0 || sl.last_use < c.slots[best].last_use) best = s;
    }
    return best;
}

}  // namespace

extern "C" {

bd_status bd_cache_create(void* device_arena, size_t arena_bytes, size_t slot_bytes, int32_t n_pinned,
                          double rate_decay, void* copy_stream, bd_cache** out)
{
    if (!out) return BD_ERR_INVALID_ARG;
    *out = nullptr;
    if (slot_bytes == 0 || arena_bytes < slot_bytes || n_pinned < 0 || !(rate_decay > 0.0 && rate_decay <= 1.0))
        return BD_ERR_INVALID_ARG;
    if (device_arena && (reinterpret_cast<uintptr_t>(device_arena) % 256 != 0 || slot_bytes % 256 != 0))
        return BD_ERR_MISALIGNED;
    const size_t n = arena_bytes / slot_bytes;
    if (n > (1u << 20)) return BD_ERR_INVALID_ARG;
    bd_cache* c = new (std::nothrow) bd_cache();
    if (!c) return BD_ERR_INVALID_ARG;
    c->arena = static_cast<char*>(device_arena);
    c->slot_bytes = slot_bytes;
    c->n_pinned = n_pinned;
    c->decay = rate_decay;
    c->copy = static_cast<cudaStream_t>(copy_stream);
    c->slots.resize(n);
    if (c->arena) {
        for (auto& sl : c->slots) {
            cudaError_t e = cudaEventCreateWithFlags(&sl.ready, cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&sl.released, cudaEventDisableTiming);
            if (e != cudaSuccess) {
                bd_cache_destroy(c);
                return static_cast<bd_status>(bd::cuda_status(e));
            }
        }
    }
    c->st.slots = static_cast<int32_t>(n);
    *out = c;
    return BD_OK;
}

void bd_cache_destroy(bd_cache* c)
{
    if (!c) return;
    for (auto& sl : c->slots) {
        if (sl.ready) cudaEventDestroy(sl.ready);
        if (sl.released) cudaEventDestroy(sl.released);
    }
    delete c;
}

bd_status bd_cache_set_source(bd_cache* c, int32_t variant, const void* host_src, size_t bytes)
{
    if (!c || variant < 0 || (bytes > 0 && !host_src)) return BD_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(c->mu);
    if (bytes > c->slot_bytes) return BD_ERR_INVALID_ARG;
    if (c->slot_of.count(variant)) return BD_ERR_INVALID_ARG;  // resident: its copy may be in use
    c->src[variant] = bd_cache::Source{host_src, bytes};
    return BD_OK;
}

bd_status bd_cache_step(bd_cache* c, const int32_t* vid, int64_t n, void* stream, const void** delta, int32_t* state)
{
    BD_NVTX_RANGE("bd_cache_step");
    if (!c || n < 0 || (n > 0 && (!vid || !delta || !state))) return BD_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(c->mu);
    if (!c->acquired.empty()) return BD_ERR_INVALID_ARG;  // the previous step was not released
    // requests per variant (validated before anything changes)
    std::unordered_map<int32_t, int64_t> count;
    std::vector<int32_t> order;  // first-appearance order
    for (int64_t i = 0; i < n; ++i) {
        const int32_t v = vid[i];
        if (v < -1) return BD_ERR_BAD_VARIANT;
        if (v == -1) continue;
        if (!c->src.count(v)) return BD_ERR_BAD_VARIANT;
        if (count[v]++ == 0) order.push_back(v);
    }
    ++c->tick;
    ++c->st.steps;
    for (auto& kv : c->rate) kv.second *= c->decay;
    for (const auto& kv : count) c->rate[kv.first] += static_cast<double>(kv.second);
    update_pinned(*c);
    // most requested variants get slots first when slots are short
    std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) { return count[a] > count[b]; });
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    std::unordered_map<int32_t, int> granted;
    for (const int32_t v : order) {
        const int64_t k = count[v];
        c->st.requests += k;
        auto it = c->slot_of.find(v);
        int s = -1;
        if (it != c->slot_of.end()) {
            s = it->second;
            c->st.hits += k;
        } else {
            s = find_slot(*c);
            if (s < 0) {
                c->st.queued += k;
                continue;
            }
            auto& sl = c->slots[s];
            if (sl.variant >= 0) {
                c->slot_of.erase(sl.variant);
                ++c->st.evictions;
            }
            const bd_cache::Source& so = c->src[v];
            cudaError_t e = cudaSuccess;
            if (c->fail_countdown > 0 && --c->fail_countdown == 0) e = cudaErrorUnknown;  // injected (test aid)
            if (e == cudaSuccess && c->arena && so.bytes > 0) {
                // the copy overwrites the slot only after the last step using it finished
                e = sl.released_recorded ? cudaStreamWaitEvent(c->copy, sl.released, 0) : cudaSuccess;
                if (e == cudaSuccess)
                    e = cudaMemcpyAsync(c->arena + static_cast<size_t>(s) * c->slot_bytes, so.host, so.bytes,
                                        cudaMemcpyHostToDevice, c->copy);
                if (e == cudaSuccess) e = cudaEventRecord(sl.ready, c->copy);
            }
            if (e != cudaSuccess) {
                // the slot's old contents are gone (evicted above, perhaps partly overwritten): leave it
                // empty; hand out nothing, so the failed step needs no release
                sl.variant = -1;
                sl.last_use = 0;
                c->acquired.clear();
                return static_cast<bd_status>(bd::cuda_status(e));
            }
            sl.variant = v;
            c->slot_of[v] = s;
            ++c->st.loads;
            c->st.bytes_loaded += static_cast<int64_t>(so.bytes);
            c->st.misses += k;
        }
        c->slots[s].last_use = c->tick;
        c->acquired.push_back(s);
        granted[v] = s;
        if (c->arena)
            if (const int cs_ = bd::cuda_status(cudaStreamWaitEvent(st, c->slots[s].ready, 0))) {
                c->acquired.clear();  // nothing handed out (the slot keeps its loaded variant)
                return static_cast<bd_status>(cs_);
            }
    }
    for (int64_t i = 0; i < n; ++i) {
        const int32_t v = vid[i];
        if (v == -1) {
            state[i] = BD_CACHE_BASE;
            delta[i] = nullptr;
            continue;
        }
        const auto g = granted.find(v);
        if (g == granted.end()) {
            state[i] = BD_CACHE_QUEUED;
            delta[i] = nullptr;
        } else {
            state[i] = BD_CACHE_SERVED;
            const size_t off = static_cast<size_t>(g->second) * c->slot_bytes;
            delta[i] = c->arena ? static_cast<const void*>(c->arena + off) : reinterpret_cast<const void*>(off);
        }
    }
    return BD_OK;
}

bd_status bd_cache_release(bd_cache* c, void* stream)
{
    if (!c) return BD_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(c->mu);
    for (const int s : c->acquired) {
        auto& sl = c->slots[s];
        if (c->arena) {
            if (const int cs_ = bd::cuda_status(cudaEventRecord(sl.released, static_cast<cudaStream_t>(stream))))
                return static_cast<bd_status>(cs_);
            sl.released_recorded = true;
        }
    }
    c->acquired.clear();
    return BD_OK;
}

bd_status bd_cache_debug_fail_load(bd_cache* c, int64_t n)
{
    if (!c || n < 0) return BD_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(c->mu);
    c->fail_countdown = n;
    return BD_OK;
}

bd_status bd_cache_get_stats(bd_cache* c, bd_cache_stats* out)
{
    if (!c || !out) return BD_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(c->mu);
    *out = c->st;
    out->resident = static_cast<int32_t>(c->slot_of.size());
    out->pinned = static_cast<int32_t>(c->pinned.size());
    return BD_OK;
}

bd_status bd_cache_query(bd_cache* c, int32_t variant, int32_t* resident, int32_t* pinned, double* rate)
{
    if (!c || !resident || !pinned || !rate) return BD_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(c->mu);
    *resident = c->slot_of.count(variant) ? 1 : 0;
    *pinned = is_pinned(*c, variant) ? 1 : 0;
    const auto it = c->rate.find(variant);
    *rate = it == c->rate.end() ? 0.0 : it->second;
    return BD_OK;
}

}  // extern "C"
