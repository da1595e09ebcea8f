// C ABI of libbitdelta.so: argument checks, workspace layout and dispatch to
// the sm_103a kernels.  Every entry point is declared and documented in
// include/bitdelta.h.
#include <atomic>
#include <cstring>

#include "../../include/bitdelta.h"
#include "bd_internal.h"

namespace {

constexpr int kVersion = 10000;  // 1.0.0
constexpr size_t kWsHeader = 256;  // error word + padding; scratch starts here

// The calling thread's last failed CUDA result (bd_last_cuda_error).
thread_local int g_last_cuda_error = 0;

// Per-device cache of (compute capability, SM count).
constexpr int kMaxDevices = 64;
std::atomic<int> g_dev_cc[kMaxDevices];
std::atomic<int> g_dev_sms[kMaxDevices];

bd_status device_info(int* sm_count)
{
    int dev = 0;
    if (const int cs_ = bd::cuda_status(cudaGetDevice(&dev))) return static_cast<bd_status>(cs_);
    if (dev < 0 || dev >= kMaxDevices) return BD_ERR_DEVICE;
    int cc = g_dev_cc[dev].load(std::memory_order_acquire);
    if (cc == 0) {
        int major = 0, minor = 0, sms = 0;
        cudaError_t e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return static_cast<bd_status>(bd::cuda_status(e));
        cc = major * 10 + minor;
        g_dev_sms[dev].store(sms, std::memory_order_relaxed);
        g_dev_cc[dev].store(cc, std::memory_order_release);
    }
    if (cc != 103) return BD_ERR_DEVICE;
    *sm_count = g_dev_sms[dev].load(std::memory_order_relaxed);
    return BD_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb)
{
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

bd_status check_d_in(int64_t d_in) { return (d_in > 0 && d_in % 128 == 0) ? BD_OK : BD_ERR_UNSUPPORTED_SHAPE; }

bd_status check_ws(const void* ws, size_t ws_bytes, size_t need)
{
    if (!ws || ws_bytes < need) return BD_ERR_WORKSPACE;
    if (!aligned(ws, 256)) return BD_ERR_MISALIGNED;
    return BD_OK;
}

bd_status launched(cudaError_t e) { return static_cast<bd_status>(bd::cuda_status(e)); }

uint32_t* err_word(void* ws) { return static_cast<uint32_t*>(ws); }

}  // namespace

int bd::cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return BD_OK;
    g_last_cuda_error = static_cast<int>(e);
    return BD_ERR_CUDA;
}

extern "C" {

int bd_version(void) { return kVersion; }

int bd_last_cuda_error(void) { return g_last_cuda_error; }

const char* bd_cuda_error_string(int code)
{
    const char* name = cudaGetErrorName(static_cast<cudaError_t>(code));
    return name ? name : "unknown CUDA error";
}

const char* bd_status_string(bd_status s)
{
    switch (s) {
        case BD_OK: return "BD_OK";
        case BD_ERR_INVALID_ARG: return "BD_ERR_INVALID_ARG: invalid argument";
        case BD_ERR_UNSUPPORTED_SHAPE: return "BD_ERR_UNSUPPORTED_SHAPE: d_in must be a positive multiple of 128";
        case BD_ERR_MISALIGNED: return "BD_ERR_MISALIGNED: pointer alignment rule broken";
        case BD_ERR_BAD_VARIANT: return "BD_ERR_BAD_VARIANT: variant id outside [-1, V)";
        case BD_ERR_NONFINITE: return "BD_ERR_NONFINITE: non-finite delta in compression";
        case BD_ERR_CUDA: return "BD_ERR_CUDA: CUDA runtime error";
        case BD_ERR_TIMEOUT: return "BD_ERR_TIMEOUT: an in-kernel wait timed out";
        case BD_ERR_WORKSPACE: return "BD_ERR_WORKSPACE: workspace missing or too small";
        case BD_ERR_DEVICE: return "BD_ERR_DEVICE: current device is not compute capability 10.3";
        case BD_ERR_BOUNDS: return "BD_ERR_BOUNDS: a kernel met an index outside its buffer (bounds-checked build)";
    }
    return "BD_ERR_UNKNOWN";
}

// ------------------------------------------------------------------ compress

size_t bd_compress_workspace_size(int64_t d_out, int64_t /*d_in*/, int alpha_mode)
{
    if (d_out < 0) return 0;
    size_t n = kWsHeader;
    if (alpha_mode == BD_ALPHA_PER_MATRIX) {
        const size_t ctas = static_cast<size_t>((d_out + bd::kCompressRowsPerCta - 1) / bd::kCompressRowsPerCta);
        n += ctas * sizeof(double);
    }
    return (n + 255) & ~static_cast<size_t>(255);
}

bd_status bd_compress(const uint16_t* w_base, const uint16_t* w_ft, int64_t d_out, int64_t d_in, int alpha_mode,
                      uint32_t* signs, float* alpha, void* ws, size_t ws_bytes, void* stream)
{
    BD_NVTX_RANGE("bd_compress");
    if (alpha_mode != BD_ALPHA_PER_MATRIX && alpha_mode != BD_ALPHA_PER_ROW) return BD_ERR_INVALID_ARG;
    if (d_out < 0) return BD_ERR_UNSUPPORTED_SHAPE;
    if (bd_status s = check_d_in(d_in)) return s;
    if (bd_status s = check_ws(ws, ws_bytes, bd_compress_workspace_size(d_out, d_in, alpha_mode))) return s;
    if (d_out == 0) return BD_OK;
    if (!w_base || !w_ft || !signs || !alpha) return BD_ERR_INVALID_ARG;
    if (!aligned(w_base, 16) || !aligned(w_ft, 16) || !aligned(signs, 16) || !aligned(alpha, 4))
        return BD_ERR_MISALIGNED;
    const size_t wbytes = static_cast<size_t>(d_out) * d_in * 2;
    const size_t sbytes = static_cast<size_t>(d_out) * (d_in / 8);
    const size_t abytes = (alpha_mode == BD_ALPHA_PER_ROW ? static_cast<size_t>(d_out) : 1u) * 4;
    if (overlaps(signs, sbytes, w_base, wbytes) || overlaps(signs, sbytes, w_ft, wbytes) ||
        overlaps(alpha, abytes, w_base, wbytes) || overlaps(alpha, abytes, w_ft, wbytes) ||
        overlaps(signs, sbytes, alpha, abytes) || overlaps(ws, ws_bytes, signs, sbytes) ||
        overlaps(ws, ws_bytes, alpha, abytes))
        return BD_ERR_INVALID_ARG;
    int sms = 0;
    if (bd_status s = device_info(&sms)) return s;
    auto* partials = reinterpret_cast<double*>(static_cast<char*>(ws) + kWsHeader);
    return launched(bd::launch_compress(w_base, w_ft, d_out, d_in, alpha_mode == BD_ALPHA_PER_ROW, signs, alpha,
                                        partials, err_word(ws), static_cast<cudaStream_t>(stream)));
}

bd_status bd_debug_reconstruct(const uint16_t* w_base, const uint32_t* signs, const float* alpha, int alpha_mode,
                               int64_t d_out, int64_t d_in, float* w_eff, void* stream)
{
    BD_NVTX_RANGE("bd_debug_reconstruct");
    if (alpha_mode != BD_ALPHA_PER_MATRIX && alpha_mode != BD_ALPHA_PER_ROW) return BD_ERR_INVALID_ARG;
    if (d_out < 0) return BD_ERR_UNSUPPORTED_SHAPE;
    if (bd_status s = check_d_in(d_in)) return s;
    if (d_out == 0) return BD_OK;
    if (!w_base || !signs || !alpha || !w_eff) return BD_ERR_INVALID_ARG;
    int sms = 0;
    if (bd_status s = device_info(&sms)) return s;
    return launched(bd::launch_debug_reconstruct(w_base, signs, alpha, alpha_mode == BD_ALPHA_PER_ROW, d_out, d_in,
                                                 w_eff, static_cast<cudaStream_t>(stream)));
}

bd_status bd_materialize(const uint16_t* w_base, const uint32_t* signs, const float* alpha, int alpha_mode,
                         int64_t d_out, int64_t d_in, uint16_t* w_eff, void* stream)
{
    BD_NVTX_RANGE("bd_materialize");
    if (alpha_mode != BD_ALPHA_PER_MATRIX && alpha_mode != BD_ALPHA_PER_ROW) return BD_ERR_INVALID_ARG;
    if (d_out < 0) return BD_ERR_UNSUPPORTED_SHAPE;
    if (bd_status s = check_d_in(d_in)) return s;
    if (d_out == 0) return BD_OK;
    if (!w_base || !signs || !alpha || !w_eff) return BD_ERR_INVALID_ARG;
    if (!aligned(w_base, 16) || !aligned(w_eff, 16) || !aligned(signs, 4) || !aligned(alpha, 4))
        return BD_ERR_MISALIGNED;
    const size_t wbytes = static_cast<size_t>(d_out) * static_cast<size_t>(d_in) * 2;
    const size_t abytes = (alpha_mode == BD_ALPHA_PER_ROW ? static_cast<size_t>(d_out) : 1u) * 4;
    if (overlaps(w_eff, wbytes, w_base, wbytes) || overlaps(w_eff, wbytes, signs, wbytes / 16) ||
        overlaps(w_eff, wbytes, alpha, abytes))
        return BD_ERR_INVALID_ARG;
    int sms = 0;
    if (bd_status s = device_info(&sms)) return s;
    return launched(bd::launch_materialize(w_base, signs, alpha, alpha_mode == BD_ALPHA_PER_ROW, d_out, d_in, w_eff,
                                           sms, static_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------------------ MonoSoup merge

size_t bd_monosoup_workspace_size(int64_t d_out, int64_t d_in, int32_t k, int32_t rank, int32_t l)
{
    if (d_out < 0 || d_in < 0 || k < 1 || rank < 0 || l < 1) return 0;
    return bd::monosoup_workspace_size(d_out, d_in, k, rank, l);
}

bd_status bd_monosoup_merge(const uint16_t* w_base, const uint16_t* const* w_ft, int32_t k, int64_t d_out,
                            int64_t d_in, int32_t rank, int32_t l, int32_t power_iters, const float* omega,
                            void* w_merged, int out_dtype, void* ws, size_t ws_bytes, void* stream)
{
    BD_NVTX_RANGE("bd_monosoup_merge");
    if (out_dtype != BD_OUT_BF16 && out_dtype != BD_OUT_F32) return BD_ERR_INVALID_ARG;
    if (k < 1 || k > BD_MAX_VARIANTS || rank < 0 || l < 4 || l > bd::monosoup_max_l() || l % 4 != 0 || rank > l ||
        power_iters < 0 || power_iters > 16)
        return BD_ERR_INVALID_ARG;
    if (d_out < 0) return BD_ERR_UNSUPPORTED_SHAPE;
    if (bd_status s = check_d_in(d_in)) return s;
    if (d_out == 0) return BD_OK;
    if (!w_base || !w_ft || !w_merged || (rank > 0 && !omega)) return BD_ERR_INVALID_ARG;
    const size_t wbytes = static_cast<size_t>(d_out) * static_cast<size_t>(d_in) * 2;
    const size_t obytes = wbytes * (out_dtype == BD_OUT_F32 ? 2 : 1);
    if (!aligned(w_base, 16) || !aligned(w_merged, 16) || (omega && !aligned(omega, 16))) return BD_ERR_MISALIGNED;
    if (overlaps(w_merged, obytes, w_base, wbytes)) return BD_ERR_INVALID_ARG;
    for (int32_t i = 0; i < k; ++i) {
        if (!w_ft[i]) return BD_ERR_INVALID_ARG;
        if (!aligned(w_ft[i], 16)) return BD_ERR_MISALIGNED;
        if (overlaps(w_merged, obytes, w_ft[i], wbytes)) return BD_ERR_INVALID_ARG;
    }
    if (omega && overlaps(w_merged, obytes, omega, static_cast<size_t>(d_in) * l * 4)) return BD_ERR_INVALID_ARG;
    if (bd_status s = check_ws(ws, ws_bytes, bd::monosoup_workspace_size(d_out, d_in, k, rank, l))) return s;
    if (overlaps(ws, ws_bytes, w_merged, obytes)) return BD_ERR_INVALID_ARG;
    int sms = 0;
    if (bd_status s = device_info(&sms)) return s;
    bd::MonoSoupArgs a{};
    a.w_base = w_base;
    a.w_ft = w_ft;
    a.k = k;
    a.d_out = d_out;
    a.d_in = d_in;
    a.rank = rank;
    a.l = l;
    a.power_iters = power_iters;
    a.omega = omega;
    a.out = w_merged;
    a.out_f32 = out_dtype == BD_OUT_F32;
    a.ws = ws;
    a.err = err_word(ws);
    a.sm_count = sms;
    return launched(bd::launch_monosoup(a, static_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------------------ linear

size_t bd_linear_workspace_size(int64_t /*T*/, int64_t /*d_out*/, int64_t /*d_in*/) { return kWsHeader; }

static bd_status check_linear_common(const uint16_t* x, int64_t T, const uint16_t* w_base, int64_t d_out,
                                     int64_t d_in, void* y, int out_dtype, void* ws, size_t ws_bytes, size_t ws_need)
{
    if (out_dtype != BD_OUT_BF16 && out_dtype != BD_OUT_F32) return BD_ERR_INVALID_ARG;
    if (T < 0 || d_out < 0) return BD_ERR_UNSUPPORTED_SHAPE;
    if (bd_status s = check_d_in(d_in)) return s;
    if (bd_status s = check_ws(ws, ws_bytes, ws_need)) return s;
    if (T == 0 || d_out == 0) return BD_OK;
    if (!x || !w_base || !y) return BD_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(w_base, 16) || !aligned(y, 16)) return BD_ERR_MISALIGNED;
    const size_t ybytes = static_cast<size_t>(T) * d_out * (out_dtype == BD_OUT_F32 ? 4 : 2);
    if (overlaps(y, ybytes, x, static_cast<size_t>(T) * d_in * 2) ||
        overlaps(y, ybytes, w_base, static_cast<size_t>(d_out) * d_in * 2) || overlaps(y, ybytes, ws, ws_bytes))
        return BD_ERR_INVALID_ARG;
    return BD_OK;
}

bd_status bd_linear(const uint16_t* x, int64_t T, const uint16_t* w_base, const uint32_t* signs, const float* alpha,
                    int alpha_mode, int64_t d_out, int64_t d_in, void* y, int out_dtype, void* ws, size_t ws_bytes,
                    void* stream)
{
    BD_NVTX_RANGE("bd_linear");
    if (alpha_mode != BD_ALPHA_PER_MATRIX && alpha_mode != BD_ALPHA_PER_ROW) return BD_ERR_INVALID_ARG;
    if (bd_status s = check_linear_common(x, T, w_base, d_out, d_in, y, out_dtype, ws, ws_bytes,
                                          bd_linear_workspace_size(T, d_out, d_in)))
        return s;
    if (T == 0 || d_out == 0) return BD_OK;
    if (!signs || !alpha) return BD_ERR_INVALID_ARG;
    if (!aligned(signs, 16) || !aligned(alpha, 4)) return BD_ERR_MISALIGNED;
    const size_t ybytes = static_cast<size_t>(T) * d_out * (out_dtype == BD_OUT_F32 ? 4 : 2);
    const size_t abytes = (alpha_mode == BD_ALPHA_PER_ROW ? static_cast<size_t>(d_out) : 1u) * 4;
    if (overlaps(y, ybytes, signs, static_cast<size_t>(d_out) * (d_in / 8)) || overlaps(y, ybytes, alpha, abytes))
        return BD_ERR_INVALID_ARG;
    int sms = 0;
    if (bd_status s = device_info(&sms)) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t ysz = out_dtype == BD_OUT_F32 ? 4 : 2;

    if (T > bd::kSkinnyMaxTokens && bd::prefill_available()) {
        bd::PrefillArgs p{};
        p.x = x; p.w_base = w_base; p.signs = signs; p.alpha = alpha;
        p.per_row = alpha_mode == BD_ALPHA_PER_ROW;
        p.T = T; p.d_out = d_out; p.d_in = d_in; p.y = y; p.out_f32 = out_dtype == BD_OUT_F32;
        p.err = err_word(ws);
        return launched(bd::launch_prefill(p, sms, st));
    }
    // decode kernel over groups of up to 64 tokens
    for (int64_t t0 = 0; t0 < T; t0 += bd::kSkinnyMaxTokens) {
        bd::SkinnyArgs a{};
        a.x = x + t0 * d_in;
        a.w_base = w_base;
        a.signs = signs;
        a.alpha = alpha;
        a.T = (T - t0) < bd::kSkinnyMaxTokens ? (T - t0) : bd::kSkinnyMaxTokens;
        a.d_out = d_out; a.d_in = d_in;
        a.per_row = alpha_mode == BD_ALPHA_PER_ROW;
        a.y = static_cast<char*>(y) + static_cast<size_t>(t0) * d_out * ysz;
        a.out_f32 = out_dtype == BD_OUT_F32;
        a.err = err_word(ws);
        if (bd_status s = launched(bd::launch_skinny(a, st))) return s;
    }
    return BD_OK;
}

// Multi-variant workspace for one group of up to 64 tokens: the error word,
// then (at 1 KiB) the zero-padded per-variant x tiles of the sign phases and
// the per-token partial corrections.
namespace {

struct MultiWs {
    size_t xp, corr, total;
};

MultiWs multi_ws_layout(int64_t T, int32_t V, int64_t d_in)
{
    const int64_t group = bd::multi_group_tokens(V);
    const int64_t tg = T < group ? T : group;
    const auto up = [](size_t n) { return (n + 255) & ~static_cast<size_t>(255); };
    MultiWs w{};
    w.xp = 1024;
    const size_t ptiles = static_cast<size_t>(bd::multi_max_ptiles(static_cast<int>(tg), V));
    w.corr = w.xp + up(ptiles * 8 * static_cast<size_t>(d_in) * 2);
    w.total = w.corr + up(static_cast<size_t>(tg) * static_cast<size_t>(bd::multi_corr_splits(d_in)) * 4);
    return w;
}

// From this many tokens on, bd_linear_multi runs the grouped tensor-core
// prefill (one 256-token block per variant segment piece) instead of the
// decode kernel on 64-token groups: at 512 tokens over 14 variants the plan
// has at most 17 blocks per row block against 8 decode groups that each
// re-read W_base.
constexpr int64_t kMultiPrefillMinT = 512;

bool use_grouped_prefill(int64_t T) { return T >= kMultiPrefillMinT && bd::prefill_available(); }

// Grouped prefill workspace: the error word, then the router's perm [T] and
// seg_off [V + 2], the block plan and x in sorted order [T][d_in].
struct GroupedWs {
    size_t perm, seg, plan, xs, total;
};

GroupedWs grouped_ws_layout(int64_t T, int32_t V, int64_t d_in)
{
    const auto up = [](size_t n) { return (n + 255) & ~static_cast<size_t>(255); };
    GroupedWs w{};
    w.perm = 1024;
    w.seg = w.perm + up(static_cast<size_t>(T) * 4);
    w.plan = w.seg + up(static_cast<size_t>(V + 2) * 4);
    w.xs = w.plan + up(static_cast<size_t>(bd::grouped_prefill_blocks(T, V)) * 16);
    w.total = w.xs + up(static_cast<size_t>(T) * static_cast<size_t>(d_in) * 2);
    return w;
}

}  // namespace

size_t bd_linear_multi_workspace_size(int64_t T, int32_t V, int64_t /*d_out*/, int64_t d_in)
{
    if (T < 0 || d_in < 0 || V < 1 || V > BD_MAX_VARIANTS) return kWsHeader;
    if (use_grouped_prefill(T)) return grouped_ws_layout(T, V, d_in).total;
    return multi_ws_layout(T, V, d_in).total;
}

bd_status bd_linear_multi(const uint16_t* x, int64_t T, const int32_t* vid, int32_t V,
                          const uint32_t* const* signs_tab, const float* const* alpha_tab, int alpha_mode,
                          const uint16_t* w_base, int64_t d_out, int64_t d_in, void* y, int out_dtype, void* ws,
                          size_t ws_bytes, void* stream)
{
    BD_NVTX_RANGE("bd_linear_multi");
    if (alpha_mode != BD_ALPHA_PER_MATRIX && alpha_mode != BD_ALPHA_PER_ROW) return BD_ERR_INVALID_ARG;
    if (V < 1 || V > BD_MAX_VARIANTS) return BD_ERR_INVALID_ARG;
    if (bd_status s = check_linear_common(x, T, w_base, d_out, d_in, y, out_dtype, ws, ws_bytes,
                                          bd_linear_multi_workspace_size(T, V, d_out, d_in)))
        return s;
    if (T == 0 || d_out == 0) return BD_OK;
    if (!vid || !signs_tab || !alpha_tab) return BD_ERR_INVALID_ARG;
    if (!aligned(vid, 4)) return BD_ERR_MISALIGNED;
    const size_t ybytes = static_cast<size_t>(T) * d_out * (out_dtype == BD_OUT_F32 ? 4 : 2);
    const size_t abytes = (alpha_mode == BD_ALPHA_PER_ROW ? static_cast<size_t>(d_out) : 1u) * 4;
    for (int v = 0; v < V; ++v) {
        if (!signs_tab[v] || !alpha_tab[v]) return BD_ERR_INVALID_ARG;
        if (!aligned(signs_tab[v], 16) || !aligned(alpha_tab[v], 4)) return BD_ERR_MISALIGNED;
        if (overlaps(y, ybytes, signs_tab[v], static_cast<size_t>(d_out) * (d_in / 8)) ||
            overlaps(y, ybytes, alpha_tab[v], abytes))
            return BD_ERR_INVALID_ARG;
    }
    if (overlaps(y, ybytes, vid, static_cast<size_t>(T) * 4)) return BD_ERR_INVALID_ARG;
    int sms = 0;
    if (bd_status s = device_info(&sms)) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (use_grouped_prefill(T)) {
        if (T > INT32_MAX) return BD_ERR_UNSUPPORTED_SHAPE;
        const GroupedWs lay = grouped_ws_layout(T, V, d_in);
        char* w = static_cast<char*>(ws);
        bd::GroupedPrefillArgs g{};
        g.x = x;
        g.perm = reinterpret_cast<int32_t*>(w + lay.perm);
        g.seg_off = reinterpret_cast<int32_t*>(w + lay.seg);
        g.w_base = w_base;
        for (int v = 0; v < V; ++v) {
            g.signs[v] = signs_tab[v];
            g.alpha[v] = alpha_tab[v];
        }
        g.V = V;
        g.per_row = alpha_mode == BD_ALPHA_PER_ROW;
        g.T = T;
        g.d_out = d_out;
        g.d_in = d_in;
        g.y = y;
        g.out_f32 = out_dtype == BD_OUT_F32;
        g.err = err_word(ws);
        g.xs = reinterpret_cast<uint16_t*>(w + lay.xs);
        g.plan = reinterpret_cast<int4*>(w + lay.plan);
        if (bd_status s = launched(bd::launch_route(vid, T, V, reinterpret_cast<int32_t*>(w + lay.perm),
                                                    reinterpret_cast<int32_t*>(w + lay.seg), g.err, st)))
            return s;
        return launched(bd::launch_prefill_grouped(g, st));
    }
    const size_t ysz = out_dtype == BD_OUT_F32 ? 4 : 2;
    const int64_t group = bd::multi_group_tokens(V);
    const MultiWs lay = multi_ws_layout(T, V, d_in);
    for (int64_t t0 = 0; t0 < T; t0 += group) {
        bd::MultiArgs a{};
        a.x = x + t0 * d_in;
        a.vid = vid + t0;
        a.w_base = w_base;
        a.T = (T - t0) < group ? (T - t0) : group;
        a.d_out = d_out; a.d_in = d_in; a.V = V;
        a.per_row = alpha_mode == BD_ALPHA_PER_ROW;
        for (int v = 0; v < V; ++v) {
            a.signs[v] = signs_tab[v];
            a.alpha[v] = alpha_tab[v];
        }
        a.y = static_cast<char*>(y) + static_cast<size_t>(t0) * d_out * ysz;
        a.out_f32 = out_dtype == BD_OUT_F32;
        a.err = err_word(ws);
        a.xp = reinterpret_cast<uint8_t*>(static_cast<char*>(ws) + lay.xp);
        a.corr = reinterpret_cast<float*>(static_cast<char*>(ws) + lay.corr);
        if (bd_status s = launched(bd::launch_multi(a, st))) return s;
    }
    return BD_OK;
}

// ------------------------------------------------------------------ router

size_t bd_route_workspace_size(int64_t /*T*/, int32_t /*V*/) { return kWsHeader; }

bd_status bd_route(const int32_t* vid, int64_t T, int32_t V, int32_t* perm, int32_t* seg_off, void* ws,
                   size_t ws_bytes, void* stream)
{
    BD_NVTX_RANGE("bd_route");
    if (V < 0 || V > BD_MAX_VARIANTS) return BD_ERR_INVALID_ARG;
    if (T < 0 || T > INT32_MAX) return BD_ERR_UNSUPPORTED_SHAPE;
    if (bd_status s = check_ws(ws, ws_bytes, bd_route_workspace_size(T, V))) return s;
    if (!seg_off || (T > 0 && (!vid || !perm))) return BD_ERR_INVALID_ARG;
    if (!aligned(seg_off, 4) || (T > 0 && (!aligned(vid, 4) || !aligned(perm, 4)))) return BD_ERR_MISALIGNED;
    if (overlaps(perm, static_cast<size_t>(T) * 4, vid, static_cast<size_t>(T) * 4) ||
        overlaps(seg_off, static_cast<size_t>(V + 2) * 4, vid, static_cast<size_t>(T) * 4) ||
        overlaps(seg_off, static_cast<size_t>(V + 2) * 4, perm, static_cast<size_t>(T) * 4))
        return BD_ERR_INVALID_ARG;
    int sms = 0;
    if (bd_status s = device_info(&sms)) return s;
    return launched(bd::launch_route(vid, T, V, perm, seg_off, err_word(ws), static_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------------------ async errors

int bd_debug_bounds_check(uint32_t* kernels)
{
    const uint32_t f = bd::bounds_take_compress() | bd::bounds_take_skinny() | bd::bounds_take_multi() |
                       bd::bounds_take_prefill() | bd::bounds_take_route() | bd::bounds_take_materialize() |
                       bd::bounds_take_monosoup();
    if (kernels) *kernels = f;
    if (f == ~0u) return BD_ERR_CUDA;
    return f ? BD_ERR_BOUNDS : BD_OK;
}

int bd_debug_bounds_enabled(void)
{
#ifdef BD_DEBUG_BOUNDS
    return 1;
#else
    return 0;
#endif
}

bd_status bd_check_async(void* ws, void* stream)
{
    if (!ws) return BD_ERR_WORKSPACE;
    if (!aligned(ws, 256)) return BD_ERR_MISALIGNED;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    if (const int cs_ = bd::cuda_status(cudaMemcpyAsync(&word, ws, sizeof word, cudaMemcpyDeviceToHost, st))) return static_cast<bd_status>(cs_);
    if (const int cs_ = bd::cuda_status(cudaStreamSynchronize(st))) return static_cast<bd_status>(cs_);
    if (word == 0) return BD_OK;
    const uint32_t zero = 0;
    if (const int cs_ = bd::cuda_status(cudaMemcpyAsync(ws, &zero, sizeof zero, cudaMemcpyHostToDevice, st))) return static_cast<bd_status>(cs_);
    if (const int cs_ = bd::cuda_status(cudaStreamSynchronize(st))) return static_cast<bd_status>(cs_);
    if (word & (1u << BD_ERR_TIMEOUT)) return BD_ERR_TIMEOUT;
    if (word & (1u << BD_ERR_BAD_VARIANT)) return BD_ERR_BAD_VARIANT;
    if (word & (1u << BD_ERR_NONFINITE)) return BD_ERR_NONFINITE;
    return BD_ERR_CUDA;
}

}  // extern "C"
