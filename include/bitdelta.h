/*
 * bitdelta.h -- C ABI of libbitdelta.so, the GB300 (sm_103a) BitDelta path.
 *
 * BitDelta ("BitDelta: Tek bir GPU kumesinden 14 Zen modeli sunmak", Hanzo
 * blog, 2026-02-28) stores a fine-tuned variant of a base model as the sign
 * of its weight delta, one bit per weight, plus a float32 scale alpha, and
 * serves it with a fused kernel that reads the base weight and the bits
 * together without ever writing the effective weight to device memory.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers named as device buffers must point to device memory of the
 *    current CUDA device; host arrays are marked "host".  The caller owns
 *    every buffer; the library never allocates or frees memory.
 *  - bf16 tensors are passed as uint16_t bit patterns, row-major, contiguous.
 *  - Packed signs: uint32 [d_out][d_in/32]; bit b of word w of row r holds
 *    column 32*w + b; bit = 1 <=> sign +1; sign(0) := +1 (also for -0.0).
 *    On a little-endian GPU the same bytes are the int8 [d_out][d_in/8]
 *    layout of the post's storage format (section "Altyapi ayrintilari").
 *  - alpha: float32, one per output row (BD_ALPHA_PER_ROW) or one per matrix
 *    (BD_ALPHA_PER_MATRIX).
 *  - Shapes: d_in must be a positive multiple of 128 (every packed sign row
 *    then starts on a 16-byte boundary, which the bulk copies need; the bit
 *    packing alone would only need a multiple of 32, so this is the stricter
 *    rule of this library); d_out >= 0 and T >= 0 are otherwise free (zero
 *    sizes are a no-op).
 *  - Alignment: bf16 and sign buffers and y must be 16-byte aligned; alpha,
 *    vid, perm, seg_off 4-byte aligned; workspaces 256-byte aligned.
 *  - Asynchrony: all work is enqueued on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream).  The return value reports only the
 *    synchronous argument checks and launch errors.
 *  - Workspace: a caller-owned device buffer of at least the size that the
 *    matching *_workspace_size function returns.  Its first 4 bytes are the
 *    asynchronous error word; fill the buffer with zeros once before its
 *    first use.  Errors found by a kernel (an out-of-range variant id, a
 *    non-finite delta, a wait that timed out) set bits there; read and clear
 *    them with bd_check_async.  Calls that share a workspace must be ordered
 *    on one stream.
 *  - No exceptions cross this boundary.  Mutable global state: a per-device
 *    cache of device attributes and kernel settings (filled once, under a
 *    lock or with atomics), the thread_local launch
 *    parameter blocks of the multi-variant and prefill launches (one per
 *    host thread), and the fixed scratch array of bd_compress_noalloc.  The
 *    library may be called from several host threads.
 */
#ifndef BITDELTA_H
#define BITDELTA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum bd_status {
    BD_OK = 0,
    BD_ERR_INVALID_ARG = 1,       /* null pointer, bad enum, aliasing output, V out of range */
    BD_ERR_UNSUPPORTED_SHAPE = 2, /* d_in not a positive multiple of 128, negative size */
    BD_ERR_MISALIGNED = 3,        /* a pointer breaks the alignment rules above */
    BD_ERR_BAD_VARIANT = 4,       /* (async) a variant id outside [-1, V) */
    BD_ERR_NONFINITE = 5,         /* (async) a non-finite delta met by bd_compress */
    BD_ERR_CUDA = 6,              /* a CUDA runtime call or launch failed */
    BD_ERR_TIMEOUT = 7,           /* (async) a bounded in-kernel wait gave up */
    BD_ERR_WORKSPACE = 8,         /* workspace null or smaller than required */
    BD_ERR_DEVICE = 9,            /* current device is not a compute capability 10.3 GPU */
    BD_ERR_BOUNDS = 10            /* (bounds-checked builds) a kernel met an index outside its buffer */
} bd_status;

typedef enum bd_alpha_mode { BD_ALPHA_PER_MATRIX = 0, BD_ALPHA_PER_ROW = 1 } bd_alpha_mode;

typedef enum bd_out_dtype { BD_OUT_BF16 = 0, BD_OUT_F32 = 1 } bd_out_dtype;

/* Largest number of variants one bd_linear_multi call can address. */
#define BD_MAX_VARIANTS 64

/* Library version, major*10000 + minor*100 + patch. */
int bd_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char* bd_status_string(bd_status status);

/* The cudaError_t code of the last CUDA runtime call or kernel launch made
 * by this library on the calling thread that failed -- the cause behind the
 * last BD_ERR_CUDA the thread saw -- or 0 if none has failed.  Kept per
 * thread; a later success does not clear it. */
int bd_last_cuda_error(void);

/* CUDA's name of a cudaError_t code, e.g. "cudaErrorInvalidValue" (static
 * string, never NULL). */
const char* bd_cuda_error_string(int code);

/* ------------------------------------------------------------------------
 * Compression -- section "Matematiksel temel", eqs. (1)-(3):
 *   Delta = W_ft - W_base,  alpha = mean |Delta| (per row or per matrix),
 *   signs = sign(Delta) packed one bit per weight.
 * w_base, w_ft : device bf16 [d_out][d_in]
 * signs        : device uint32 [d_out][d_in/32] (written)
 * alpha        : device float32 [d_out] (per row) or [1] (per matrix) (written)
 * Delta is formed in fp32 registers (the sign is always exact); alpha is
 * accumulated in fp64 and rounded to float32 once.  The result does not
 * depend on launch timing (no floating-point atomics).  A non-finite delta
 * sets BD_ERR_NONFINITE in the error word; the signs of that row are still
 * written and its alpha is then undefined.
 * ------------------------------------------------------------------------ */
size_t bd_compress_workspace_size(int64_t d_out, int64_t d_in, int alpha_mode);

bd_status bd_compress(const uint16_t* w_base, const uint16_t* w_ft, int64_t d_out, int64_t d_in, int alpha_mode,
                      uint32_t* signs, float* alpha, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Fused linear -- section "Sunum mimarisi": the conceptual
 * fused_bitdelta_linear listing and the fused-kernel paragraph after it:
 *   y[t][r] = sum_j x[t][j] * (W_base[r][j] + alpha_r * s_rj)
 * computed in one pass that reads W_base and the packed bits together; the
 * effective weight exists only in registers / shared memory.
 * x     : device bf16 [T][d_in] (the listing's [batch, seq, d_in] flattened)
 * w_base: device bf16 [d_out][d_in];  signs, alpha as produced by bd_compress
 * y     : device [T][d_out], bf16 (BD_OUT_BF16) or float32 (BD_OUT_F32);
 *         must not overlap any input.
 * Accumulation is fp32.  T <= 64 runs the decode kernel (the base and the
 * sign contraction are kept apart, so W_eff is never rounded); larger T runs
 * the prefill GEMM, which rounds W_eff to bf16 in tensor memory (the A
 * operand of the tensor-core contraction) before multiplying.  For a given (T, d_in) the result of a row does
 * not depend on d_out, so a row-sharded call reproduces the unsharded one
 * bit for bit.
 * ------------------------------------------------------------------------ */
size_t bd_linear_workspace_size(int64_t T, int64_t d_out, int64_t d_in);

bd_status bd_linear(const uint16_t* x, int64_t T, const uint16_t* w_base, const uint32_t* signs, const float* alpha,
                    int alpha_mode, int64_t d_out, int64_t d_in, void* y, int out_dtype, void* ws, size_t ws_bytes,
                    void* stream);

/* ------------------------------------------------------------------------
 * Multi-variant fused linear -- section "Sunum mimarisi": one W_base in
 * device memory, shared read by every variant's delta in the delta cache,
 * and a router that picks each request's variant (serving steps 1-3).
 * Token t uses variant vid[t]; vid[t] == -1 means the base model alone.
 * x        : device bf16 [T][d_in];  vid: device int32 [T]
 * signs_tab: host array of V device pointers, each uint32 [d_out][d_in/32]
 * alpha_tab: host array of V device pointers, each float32 [d_out] or [1]
 *            (host arrays, read during the call: the library builds each
 *            variant's tensor map from them; the pointed-to data is read by
 *            the kernels in stream order)
 * y        : device [T][d_out] in the caller's token order.
 * 1 <= V <= BD_MAX_VARIANTS.  An id outside [-1, V) sets BD_ERR_BAD_VARIANT
 * in the error word and that token is computed as a base-model token.
 * Accumulation is fp32.  Two paths, chosen by T:
 *  - T < 512 (decode batches): groups of up to 64 tokens; each W_base tile
 *    is read from device memory once per group, the tokens are grouped by
 *    variant inside the kernel and every active variant's sign tile is
 *    applied to its own tokens only.  The sign contraction runs on an exact
 *    recoding of the +-1 operand: each sign bit becomes a mantissa or sign
 *    bit of a constant of its column (mod 4), and the token's share of those
 *    constants is subtracted once at the end; its fp32 rounding error is at
 *    most about 20 times that of the plain form (relative to
 *    alpha * sum_j |x_j|), and non-finite x give non-finite outputs.
 *  - T >= 512 (multi-tenant prefill): the tokens are routed as by bd_route,
 *    x is gathered by variant into the workspace, and the tensor-core
 *    prefill GEMM runs per 256-token block of each variant's segment with
 *    that variant's W_eff (rounded to bf16, as in bd_linear's prefill path;
 *    W_eff = W_base for base-model tokens).  The workspace then holds the
 *    gathered x: bd_linear_multi_workspace_size grows by 2 T d_in bytes.
 * ------------------------------------------------------------------------ */
size_t bd_linear_multi_workspace_size(int64_t T, int32_t V, int64_t d_out, int64_t d_in);

bd_status bd_linear_multi(const uint16_t* x, int64_t T, const int32_t* vid, int32_t V,
                          const uint32_t* const* signs_tab, const float* const* alpha_tab, int alpha_mode,
                          const uint16_t* w_base, int64_t d_out, int64_t d_in, void* y, int out_dtype, void* ws,
                          size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Router on its own -- section "Sunum mimarisi", serving steps 1-3: a request
 * names its variant, the router looks that variant's delta up and sends the
 * request to the fused kernel with it.  This is the grouping that
 * bd_linear_multi does internally, exposed so that it can be checked.
 * perm   : device int32 [T]   -- token indices, stably sorted by vid+1
 * seg_off: device int32 [V+2] -- seg_off[k] = number of tokens with
 *          vid+1 < k; segment 0 holds the base-model tokens.
 * Out-of-range ids are grouped with the base tokens and flagged
 * (BD_ERR_BAD_VARIANT).  0 <= V <= BD_MAX_VARIANTS.
 * ------------------------------------------------------------------------ */
size_t bd_route_workspace_size(int64_t T, int32_t V);

bd_status bd_route(const int32_t* vid, int64_t T, int32_t V, int32_t* perm, int32_t* seg_off, void* ws,
                   size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Test aid, not on the serving path: writes W_eff = W_base + alpha * s as
 * float32 [d_out][d_in] so the elementwise identities |W_eff - W_base| =
 * alpha and sign(W_eff - W_base) = s of section "Matematiksel temel",
 * eq. (2), can be checked on the device's own unpacking.
 * ------------------------------------------------------------------------ */
bd_status bd_debug_reconstruct(const uint16_t* w_base, const uint32_t* signs, const float* alpha, int alpha_mode,
                               int64_t d_out, int64_t d_in, float* w_eff, void* stream);

/* ------------------------------------------------------------------------
 * Materialised variant -- the reading of section "Sunum mimarisi" in which a
 * variant's effective weights are built once and a standard matmul follows
 * (the fused entry points above never build them in device memory):
 *   w_eff[r][j] = RN_bf16(W_base[r][j] + alpha_r * s_rj)
 * rounded once (to nearest, ties to even) from the exact sum.
 * w_base: device bf16 [d_out][d_in] (16-byte aligned); signs, alpha as
 * produced by bd_compress; w_eff: device bf16 [d_out][d_in] (written,
 * 16-byte aligned, overlapping no input).  Reads 2.125 and writes 2 bytes per
 * weight.
 * ------------------------------------------------------------------------ */
bd_status bd_materialize(const uint16_t* w_base, const uint32_t* signs, const float* alpha, int alpha_mode,
                         int64_t d_out, int64_t d_in, uint16_t* w_eff, void* stream);

/* ------------------------------------------------------------------------
 * MonoSoup merge -- section "MonoSoup" of the BitDelta post: for k
 * fine-tuned checkpoints W_1..W_k of one base matrix,
 *   Delta_i = W_i - W_base,  tau_i = the rank-`rank` truncated SVD of Delta_i,
 *   W_merged = W_base + (1/k) * sum_i tau_i.
 * The truncated SVD is computed by randomized subspace iteration (Halko,
 * Martinsson & Tropp 2011): a sketch Delta_i * omega with the caller's
 * Gaussian test matrix `omega` (device fp32 [d_in][l], rank <= l <= 64; the
 * same matrix for every checkpoint), `power_iters` power iterations with
 * re-orthonormalisation, then the exact SVD of the l x d_in projection.  It
 * equals the exact truncated SVD when Delta_i has rank <= l; otherwise its
 * error is governed by the singular values past l (more power iterations and
 * a larger l reduce it).  The products with Delta_i and the final merge run
 * on the tensor cores on exact three-piece bf16 splits of their fp32
 * operands (fp32 accumulation; l <= 32 -- wider sketches use fp32 CUDA-core
 * products); the Gram matrices and their Cholesky factors are float-float,
 * the l x l symmetric eigenproblem fp32 (Householder tridiagonalisation,
 * bisection on Sturm counts, inverse iteration).  The result is rounded once to
 * `out_dtype`.
 *   w_base    device bf16 [d_out][d_in], 16-byte aligned
 *   w_ft      HOST array of k device pointers, each bf16 [d_out][d_in],
 *             16-byte aligned; 1 <= k <= BD_MAX_VARIANTS
 *   rank      0 (W_merged = W_base) .. l
 *   omega     device fp32 [d_in][l], 16-byte aligned (may be NULL if rank = 0)
 *   w_merged  device [d_out][d_in], bf16 or fp32 by out_dtype, 16-byte
 *             aligned, overlapping no input and not the workspace
 *   ws        bd_monosoup_workspace_size(d_out, d_in, k, rank, l) bytes,
 *             256-byte aligned: the asynchronous error word at its start (a
 *             bounded wait of a product or merge kernel that timed out sets
 *             BD_ERR_TIMEOUT; read it with bd_check_async), then scratch (the
 *             sketches, Gram partials, split operands and the rank-`rank`
 *             factors of every checkpoint)
 * d_in must be a positive multiple of 128 (BD_ERR_UNSUPPORTED_SHAPE); l
 * must be a multiple of 4 (rows of the l-column operands move as 16-byte
 * units); out-of-range k, rank, l or power_iters (0..16) give
 * BD_ERR_INVALID_ARG.
 * Stream-ordered; the inputs must stay valid until the work completes.
 * ------------------------------------------------------------------------ */
size_t bd_monosoup_workspace_size(int64_t d_out, int64_t d_in, int32_t k, int32_t rank, int32_t l);
bd_status bd_monosoup_merge(const uint16_t* w_base, const uint16_t* const* w_ft, int32_t k, int64_t d_out,
                            int64_t d_in, int32_t rank, int32_t l, int32_t power_iters, const float* omega,
                            void* w_merged, int out_dtype, void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Compression that allocates nothing (the BitDelta post has no counterpart
 * for this entry point; it exists for callers of this library).
 * Some callers cannot call cudaMalloc or hand the library a workspace: code
 * running under an allocator that is locked or reserved by a framework,
 * code that must not allocate while a stream is being captured, or plain C
 * hosts with no device allocator of their own.  This variant computes
 * exactly what bd_compress computes, but keeps the per-matrix partial sums
 * in a fixed device array of the library (one fp64 sum per 4-row block of
 * BD_NOALLOC_MAX_ROWS rows: 512 KiB on every GPU that loads the library,
 * held until the process exits) instead of in `ws`.
 *  - d_out may be at most BD_NOALLOC_MAX_ROWS, else BD_ERR_UNSUPPORTED_SHAPE.
 *  - The first call on a device looks up that array's device address (once
 *    per device, with the device current); make that first call before any
 *    stream capture.
 *  - All calls share the one array: calls that may run at the same time on
 *    the GPU (other streams, other host threads) race and must be ordered
 *    by the caller.  Each call overwrites every partial sum it reads, so the
 *    array needs no clearing between calls.
 *  - There is no error word: a non-finite delta shows up as a non-finite
 *    alpha (the row's, or the matrix's).
 * Other arguments, conventions and results are those of bd_compress.
 * ------------------------------------------------------------------------ */
#define BD_NOALLOC_MAX_ROWS 262144

bd_status bd_compress_noalloc(const uint16_t* w_base, const uint16_t* w_ft, int64_t d_out, int64_t d_in,
                              int alpha_mode, uint32_t* signs, float* alpha, void* stream);

/* ------------------------------------------------------------------------
 * Delta cache -- section "Altyapı ayrıntıları": a variant's packed delta is
 * loaded into device memory on its first request (the cold start) and stays
 * there until evicted; eviction is request-rate-weighted LRU (the most
 * requested variants are pinned, the others share the remaining space in
 * least-recently-used order); requests for a variant whose delta is being
 * loaded wait for that one load instead of starting their own.
 *
 * bd_cache_create: the cache divides `device_arena` (caller-owned device
 *   memory, 256-byte aligned, or NULL) into arena_bytes / slot_bytes slots
 *   (slot_bytes a multiple of 256) of one variant's delta each.  n_pinned
 *   variants are pinned; request rates decay by `rate_decay` (0 < d <= 1) per
 *   step.  Copies run on `copy_stream` (a cudaStream_t; NULL = legacy default
 *   stream).  With device_arena == NULL no CUDA call is ever made and steps
 *   report slot offsets instead of addresses (a dry run of the policy).  The
 *   cache object itself is host memory owned by the library until
 *   bd_cache_destroy.  One cache may be used from several host threads.
 * bd_cache_set_source: the host copy (page-locked memory for asynchronous
 *   copies) of `variant`'s delta, bytes <= slot_bytes; not allowed while the
 *   variant is resident.
 * bd_cache_step: one serving step; vid[n] are host variant ids of its
 *   requests (-1 = base model).  Updates the rates and the pinned set (the
 *   n_pinned registered variants of highest rate), loads each missing
 *   requested variant once (most requested first) into a free slot or the
 *   least recently used slot of an unpinned variant not used by this step,
 *   makes `stream` wait for the loads of every slot handed out, and writes
 *   per request state[i] (BD_CACHE_SERVED, _BASE, _QUEUED) and delta[i] (the
 *   slot's device address, or NULL).  Queued requests found no slot: keep
 *   them for a later step.  An id < -1 or without a source returns
 *   BD_ERR_BAD_VARIANT and changes nothing.  Each step must be followed by
 *   bd_cache_release before the next.
 * bd_cache_release: records on `stream` (after the step's kernels were
 *   enqueued) that the step's slots are free to be overwritten; later loads
 *   into them wait for that point on the copy stream.
 * bd_cache_destroy: frees the cache object and its events; copies already
 *   issued may still be writing the arena, so the caller keeps the arena and
 *   the host sources alive until the copy stream has drained.
 * A step that fails with BD_ERR_CUDA hands out no slot (the next step needs
 *   no bd_cache_release first).  Loads it issued before the failure stay
 *   valid and resident; the slot whose load failed is left empty (its former
 *   variant was evicted); its rate and statistics updates stand.
 * ------------------------------------------------------------------------ */
typedef struct bd_cache bd_cache;

typedef struct bd_cache_stats {
    int64_t steps;        /* bd_cache_step calls */
    int64_t requests;     /* requests with a variant (base-model requests excluded) */
    int64_t hits;         /* requests whose variant was resident or already loading */
    int64_t misses;       /* requests whose variant their step loaded */
    int64_t queued;       /* requests left without a slot */
    int64_t loads;        /* host -> device copies issued */
    int64_t evictions;    /* resident deltas replaced by another variant's */
    int64_t bytes_loaded;
    int32_t slots, resident, pinned;
} bd_cache_stats;

#define BD_CACHE_SERVED 0
#define BD_CACHE_BASE 1
#define BD_CACHE_QUEUED 2

bd_status bd_cache_create(void* device_arena, size_t arena_bytes, size_t slot_bytes, int32_t n_pinned,
                          double rate_decay, void* copy_stream, bd_cache** out);
void bd_cache_destroy(bd_cache* cache);
bd_status bd_cache_set_source(bd_cache* cache, int32_t variant, const void* host_src, size_t bytes);
bd_status bd_cache_step(bd_cache* cache, const int32_t* vid, int64_t n, void* stream, const void** delta,
                        int32_t* state);
bd_status bd_cache_release(bd_cache* cache, void* stream);
bd_status bd_cache_get_stats(bd_cache* cache, bd_cache_stats* out);
/* resident / pinned (0 or 1) and current request rate of one variant */
bd_status bd_cache_query(bd_cache* cache, int32_t variant, int32_t* resident, int32_t* pinned, double* rate);
/* Test aid, not for serving: the n-th load issued from now on (n >= 1; 0
 * cancels) fails as if its copy had returned a CUDA error, before any copy
 * is enqueued, so that the failure path above can be exercised on the host
 * (also by a dry-run cache, which makes no CUDA call). */
bd_status bd_cache_debug_fail_load(bd_cache* cache, int64_t n);

/* Bounds-checked builds (compiled with -DBD_DEBUG_BOUNDS; the library
 * built as libbitdelta_bounds.so): every plain global load and store of the
 * kernels checks its index against its buffer and skips the access when it
 * lies outside (TMA copies are bounded by the hardware).  This is a test
 * aid, not part of the BitDelta post.  bd_debug_bounds_check synchronises the
 * device, reads and clears the flags of every kernel and returns
 * BD_ERR_BOUNDS if one met an out-of-range index since the last call (the
 * kernels' bits in *kernels, if not NULL; bit numbers in the library
 * source), BD_ERR_CUDA if the flags could not be read, else BD_OK (always
 * BD_OK in normal builds).  bd_debug_bounds_enabled returns 1 in a
 * bounds-checked build, 0 otherwise.
 *
 * Profiling: each compute entry point (compress, linear, multi, route,
 * materialise, reconstruct, MonoSoup merge, cache step) pushes an NVTX range
 * named after itself for the length of the call, so that a profiler can
 * select one call's launches (unless built with -DBD_NO_NVTX). */
int bd_debug_bounds_check(uint32_t* kernels);
int bd_debug_bounds_enabled(void);

/* Waits for `stream`, then reads and clears the error word in `ws`.
 * Returns BD_OK, or the first asynchronous error found (in the order
 * BD_ERR_TIMEOUT, BD_ERR_BAD_VARIANT, BD_ERR_NONFINITE). */
bd_status bd_check_async(void* ws, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BITDELTA_H */
