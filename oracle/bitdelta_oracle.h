/*
 * BitDelta CPU oracle -- TEST INFRASTRUCTURE ONLY (fp64 reference of the
 * fused BitDelta path; see bitdelta_oracle.c for the page citations and the
 * readings taken where the page is silent).  Not part of the product
 * library; it shares no code with it.
 *
 * Conventions: bf16 values are passed as their uint16 bit patterns; packed
 * signs are uint32 [rows][d_in/32], bit b of word w = column 32*w + b,
 * bit = 1 <=> sign +1.  All buffers are host memory owned by the caller.
 * Functions return 0 (or a count) on success and -1 on bad arguments.
 */
#ifndef BITDELTA_ORACLE_H
#define BITDELTA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

int oracle_set_threads(int n);

int oracle_compress(const uint16_t* w_base, const uint16_t* w_ft, int64_t d_out, int64_t d_in, int per_row,
                    uint32_t* signs, float* alpha);

int oracle_compress_rows(const uint16_t* w_base, const uint16_t* w_ft, int64_t d_out, int64_t d_in,
                         const int64_t* rows, int64_t n_rows, uint32_t* signs, float* alpha_rows);

int oracle_unpack_signs(const uint32_t* signs, int64_t d_out, int64_t d_in, int8_t* s);

int oracle_pack_signs(const int8_t* s, int64_t d_out, int64_t d_in, uint32_t* signs);

int oracle_reconstruct(const uint16_t* w_base, const uint32_t* signs, const float* alpha, int per_row,
                       int64_t d_out, int64_t d_in, double* w_eff);

int oracle_linear_rows(const uint16_t* x, int64_t T, const uint16_t* w_base, const uint32_t* signs,
                       const float* alpha, int per_row, int64_t d_out, int64_t d_in, const int64_t* rows,
                       int64_t n_rows, double* y);

int64_t oracle_route(const int32_t* vid, int64_t T, int32_t V, int32_t* perm, int32_t* seg_off);

int oracle_linear_multi_rows(const uint16_t* x, int64_t T, const int32_t* vid, int32_t V,
                             const uint32_t* const* signs_tab, const float* const* alpha_tab, int per_row,
                             const uint16_t* w_base, int64_t d_out, int64_t d_in, const int64_t* rows,
                             int64_t n_rows, double* y);

int64_t oracle_compressed_bytes(int64_t d_out, int64_t d_in, int64_t n_alpha);

#ifdef __cplusplus
}
#endif

#endif
