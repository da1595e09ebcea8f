/*
 * BitDelta CPU oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 statement of what the fused BitDelta path computes.
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this library; the product path never does.  It shares no code, table
 * or helper with the CUDA kernels.
 *
 * Source: "BitDelta: Tek bir GPU kumesinden 14 Zen modeli sunmak" (Hanzo
 * blog, 2026-02-28; the Spanish edition is the same text):
 *   - section "Matematiksel temel" (mathematical foundation):
 *       eq. (1)  Delta = W_ft - W_base
 *       eq. (2)  W_ft ~= W_base + alpha * sign(Delta)
 *       eq. (3)  alpha = (1/n) * ||Delta||_1 = mean |Delta_ij|
 *     and the sentence that sign keeps one bit per element, plus or minus;
 *   - section "Sunum mimarisi" (serving architecture): the conceptual
 *     fused_bitdelta_linear listing (unpacked signs in {-1,+1}, alpha per
 *     output row or scalar, W_eff = W_base + alpha*sign, y = linear(x, W_eff))
 *     and the five-step serving pipeline (router picks the variant's delta);
 *   - section "Altyapi ayrintilari" (infrastructure details): signs stored
 *     packed, 8 per byte, a 4096x4096 matrix becoming 4096x512 int8; alpha
 *     stored as float32, one per output dimension.
 *
 * Readings where the page is silent (each one is listed in the design notes):
 *   - sign(0) := +1 (the page names only plus and minus; the listing says
 *     {-1,+1}), and -0.0 counts as 0;
 *   - bit = 1 <=> +1, bit b of 32-bit word w of a row holds column 32*w + b
 *     (little-endian, so the byte view is int8 [d_out][d_in/8] with bit 0 of
 *     byte c covering column 8*c);
 *   - alpha is summed exactly enough (Neumaier-compensated fp64) and stored
 *     as the nearest float32;
 *   - W_eff and y are evaluated in fp64 (the listing's dtype promotion is
 *     garbled; mathematically W_eff = W_base + alpha*s);
 *   - multi-variant routing: a stable sort of token indices by key vid+1,
 *     vid = -1 meaning "base model only"; ids outside [-1, V) are routed as
 *     base and counted as errors.
 *
 * Every function here is single-pass and order-obvious; OpenMP only splits
 * independent rows (or tokens) across threads and never changes a result.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#include "bitdelta_oracle.h"

/* bf16 bit pattern -> exact double (bf16 is the top half of an fp32). */
static double bf16_bits_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Neumaier-compensated running sum (keeps the sum of |Delta| exact to far
 * below the float32 rounding of alpha). */
typedef struct {
    double s, c;
} neumaier;

static void neumaier_add(neumaier* a, double v)
{
    double t = a->s + v;
    if (fabs(a->s) >= fabs(v))
        a->c += (a->s - t) + v;
    else
        a->c += (v - t) + a->s;
    a->s = t;
}

static double neumaier_value(const neumaier* a) { return a->s + a->c; }

int oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* eq. (1) then the sign rule: one code per element, +1 unless Delta < 0. */
static int sign_code(double delta) { return (delta < 0.0) ? -1 : +1; }

int oracle_compress_rows(const uint16_t* w_base, const uint16_t* w_ft, int64_t d_out, int64_t d_in,
                         const int64_t* rows, int64_t n_rows, uint32_t* signs, float* alpha_rows)
{
    if (d_in <= 0 || d_in % 32 != 0 || d_out < 0 || n_rows < 0) return -1;
    const int64_t words = d_in / 32;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t k = 0; k < n_rows; ++k) {
        const int64_t i = rows ? rows[k] : k;
        if (i < 0 || i >= d_out) {
            bad |= 1;
            continue;
        }
        neumaier acc = {0.0, 0.0};
        uint32_t* out = signs + k * words;
        for (int64_t w = 0; w < words; ++w) out[w] = 0u;
        for (int64_t j = 0; j < d_in; ++j) {
            const double delta = bf16_bits_to_double(w_ft[i * d_in + j]) -
                                 bf16_bits_to_double(w_base[i * d_in + j]);
            if (sign_code(delta) > 0) out[j / 32] |= (uint32_t)1u << (j % 32);
            neumaier_add(&acc, fabs(delta));
        }
        /* eq. (3) per output row: alpha_i = (1/d_in) * sum_j |Delta_ij| */
        alpha_rows[k] = (float)(neumaier_value(&acc) / (double)d_in);
    }
    return bad ? -1 : 0;
}

int oracle_compress(const uint16_t* w_base, const uint16_t* w_ft, int64_t d_out, int64_t d_in, int per_row,
                    uint32_t* signs, float* alpha)
{
    if (d_in <= 0 || d_in % 32 != 0 || d_out < 0) return -1;
    if (per_row) return oracle_compress_rows(w_base, w_ft, d_out, d_in, NULL, d_out, signs, alpha);

    /* Per-matrix alpha: eq. (3) over all n = d_out * d_in elements, summed in
     * row-major order; the signs are the same as in the per-row case. */
    const int64_t words = d_in / 32;
    neumaier acc = {0.0, 0.0};
    for (int64_t i = 0; i < d_out; ++i) {
        uint32_t* out = signs + i * words;
        for (int64_t w = 0; w < words; ++w) out[w] = 0u;
        for (int64_t j = 0; j < d_in; ++j) {
            const double delta = bf16_bits_to_double(w_ft[i * d_in + j]) -
                                 bf16_bits_to_double(w_base[i * d_in + j]);
            if (sign_code(delta) > 0) out[j / 32] |= (uint32_t)1u << (j % 32);
            neumaier_add(&acc, fabs(delta));
        }
    }
    const double n = (double)d_out * (double)d_in;
    alpha[0] = (d_out > 0) ? (float)(neumaier_value(&acc) / n) : 0.0f;
    return 0;
}

/* bit(i, j) -> s_ij in {-1, +1} */
static int sign_of_bit(const uint32_t* signs_row, int64_t j)
{
    return ((signs_row[j / 32] >> (j % 32)) & 1u) ? +1 : -1;
}

int oracle_unpack_signs(const uint32_t* signs, int64_t d_out, int64_t d_in, int8_t* s)
{
    if (d_in <= 0 || d_in % 32 != 0 || d_out < 0) return -1;
    const int64_t words = d_in / 32;
    for (int64_t i = 0; i < d_out; ++i)
        for (int64_t j = 0; j < d_in; ++j) s[i * d_in + j] = (int8_t)sign_of_bit(signs + i * words, j);
    return 0;
}

int oracle_pack_signs(const int8_t* s, int64_t d_out, int64_t d_in, uint32_t* signs)
{
    if (d_in <= 0 || d_in % 32 != 0 || d_out < 0) return -1;
    const int64_t words = d_in / 32;
    for (int64_t i = 0; i < d_out; ++i) {
        uint32_t* out = signs + i * words;
        for (int64_t w = 0; w < words; ++w) out[w] = 0u;
        for (int64_t j = 0; j < d_in; ++j)
            if (s[i * d_in + j] > 0) out[j / 32] |= (uint32_t)1u << (j % 32);
    }
    return 0;
}

/* eq. (2) and the listing: W_eff_ij = W_base_ij + alpha_i * s_ij (fp64). */
static double weff(const uint16_t* w_base, const uint32_t* signs, const float* alpha, int per_row, int64_t d_in,
                   int64_t i, int64_t j)
{
    const double a = (double)(per_row ? alpha[i] : alpha[0]);
    return bf16_bits_to_double(w_base[i * d_in + j]) + a * (double)sign_of_bit(signs + i * (d_in / 32), j);
}

int oracle_reconstruct(const uint16_t* w_base, const uint32_t* signs, const float* alpha, int per_row,
                       int64_t d_out, int64_t d_in, double* w_eff)
{
    if (d_in <= 0 || d_in % 32 != 0 || d_out < 0) return -1;
    for (int64_t i = 0; i < d_out; ++i)
        for (int64_t j = 0; j < d_in; ++j) w_eff[i * d_in + j] = weff(w_base, signs, alpha, per_row, d_in, i, j);
    return 0;
}

/* y[t][k] = sum_j x[t][j] * W_eff[rows[k]][j]   (the listing's linear, fp64).
 * rows == NULL means all d_out rows; y is [T][n_rows]. */
int oracle_linear_rows(const uint16_t* x, int64_t T, const uint16_t* w_base, const uint32_t* signs,
                       const float* alpha, int per_row, int64_t d_out, int64_t d_in, const int64_t* rows,
                       int64_t n_rows, double* y)
{
    if (d_in <= 0 || d_in % 32 != 0 || d_out < 0 || T < 0 || n_rows < 0) return -1;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t k = 0; k < n_rows; ++k) {
        const int64_t i = rows ? rows[k] : k;
        if (i < 0 || i >= d_out) {
            bad |= 1;
            continue;
        }
        for (int64_t t = 0; t < T; ++t) {
            double acc = 0.0;
            for (int64_t j = 0; j < d_in; ++j)
                acc += bf16_bits_to_double(x[t * d_in + j]) * weff(w_base, signs, alpha, per_row, d_in, i, j);
            y[t * n_rows + k] = acc;
        }
    }
    return bad ? -1 : 0;
}

/* Router: key(t) = vid[t] + 1 (0 = base model), ids outside [-1, V) count as
 * errors and take key 0.  perm is the stable sort of token indices by key;
 * seg_off[k] = number of tokens whose key is < k, for k = 0 .. V+1.
 * Returns the number of out-of-range ids, or -1 on bad arguments. */
int64_t oracle_route(const int32_t* vid, int64_t T, int32_t V, int32_t* perm, int32_t* seg_off)
{
    if (T < 0 || V < 0) return -1;
    int64_t invalid = 0;
    int32_t* key = (int32_t*)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
    if (!key) return -1;
    for (int64_t t = 0; t < T; ++t) {
        if (vid[t] < -1 || vid[t] >= V) {
            key[t] = 0;
            ++invalid;
        } else {
            key[t] = vid[t] + 1;
        }
    }
    /* seg_off by counting: tokens with key < k */
    for (int32_t k = 0; k <= V + 1; ++k) {
        int32_t n = 0;
        for (int64_t t = 0; t < T; ++t) n += (key[t] < k);
        seg_off[k] = n;
    }
    /* stable placement: scan keys in ascending order, tokens in index order */
    int64_t p = 0;
    for (int32_t k = 0; k <= V; ++k)
        for (int64_t t = 0; t < T; ++t)
            if (key[t] == k) perm[p++] = (int32_t)t;
    free(key);
    return invalid;
}

/* Multi-variant linear: token t uses variant vid[t]'s (signs, alpha); vid -1
 * (or an out-of-range id) uses W_base alone.  y is [T][n_rows] for the given
 * rows (NULL = all d_out rows).  signs_tab / alpha_tab are host arrays of V
 * host pointers. */
int oracle_linear_multi_rows(const uint16_t* x, int64_t T, const int32_t* vid, int32_t V,
                             const uint32_t* const* signs_tab, const float* const* alpha_tab, int per_row,
                             const uint16_t* w_base, int64_t d_out, int64_t d_in, const int64_t* rows,
                             int64_t n_rows, double* y)
{
    if (d_in <= 0 || d_in % 32 != 0 || d_out < 0 || T < 0 || n_rows < 0 || V < 0) return -1;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t k = 0; k < n_rows; ++k) {
        const int64_t i = rows ? rows[k] : k;
        if (i < 0 || i >= d_out) {
            bad |= 1;
            continue;
        }
        for (int64_t t = 0; t < T; ++t) {
            const int32_t v = vid[t];
            const int use_delta = (v >= 0 && v < V);
            double acc = 0.0;
            for (int64_t j = 0; j < d_in; ++j) {
                const double w = use_delta ? weff(w_base, signs_tab[v], alpha_tab[v], per_row, d_in, i, j)
                                           : bf16_bits_to_double(w_base[i * d_in + j]);
                acc += bf16_bits_to_double(x[t * d_in + j]) * w;
            }
            y[t * n_rows + k] = acc;
        }
    }
    return bad ? -1 : 0;
}

/* Storage of one compressed matrix ("Altyapi ayrintilari"): one bit per
 * element packed 8 per byte, plus n_alpha float32 scales. */
int64_t oracle_compressed_bytes(int64_t d_out, int64_t d_in, int64_t n_alpha)
{
    return d_out * d_in / 8 + 4 * n_alpha;
}
