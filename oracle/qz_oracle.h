/*
 * qz_oracle.h -- plain CPU reference for the quantize / dequantize / error-statistics
 * path of the blog post "浅谈低精度浮点数" ("A brief talk on low-precision floats",
 * july-h5kf3.github.io column blog).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, imports or calls this
 * library; only the tests, __graft_entry__.smoke() and the CPU-baseline leg of bench.py
 * do.  It shares no code, header, table or constant with the CUDA library: the numeric
 * identifiers below have the same values as the public enums of the CUDA library because
 * they are an interface both sides have to agree on, but they are written out here
 * independently.
 *
 * Conventions of this oracle (each one a reading of the post; see the .c file):
 *  - every element code is found by a nearest-value search over a table of the
 *    format's finite values, obtained by decoding every code bit by bit;
 *  - all distance comparisons are done in double, where they are exact;
 *  - every scale and every element quotient is an IEEE-754 binary32 operation (the
 *    build uses -ffp-contract=off and no fast-math, so C float arithmetic is exactly
 *    binary32 with round-to-nearest-even and gradual underflow).
 */
#ifndef QZ_ORACLE_H
#define QZ_ORACLE_H
#include <stdint.h>
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element / tensor formats */
#define ORC_INT8 1
#define ORC_E4M3 2
#define ORC_E5M2 3
#define ORC_MXFP4 4
#define ORC_NVFP4 5
#define ORC_INT4 6 /* symmetric, q in [-7, 7], fp32 scale per group of block_size */
/* element formats only used by the table helpers */
#define ORC_E2M1 16
#define ORC_E8M0 17

/* high-precision tensor dtypes */
#define ORC_BF16 1
#define ORC_F32 2

/* scale granularity */
#define ORC_GRAN_TENSOR 1
#define ORC_GRAN_ROW 2
#define ORC_GRAN_BLOCK 3
#define ORC_GRAN_UNIT 4

/* block-scale rounding for MXFP4 / NVFP4 */
#define ORC_SCALE_UP 0
#define ORC_SCALE_NEAREST 1

/* return codes */
#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_NONFINITE 2

typedef struct {
  double sum_sq_err; /* sum of e_i^2, accumulated in double           */
  double mse;        /* sum_sq_err / n  (0 when n == 0)               */
  float max_rel_err; /* max over x_i != 0 of fl32(|e_i| / |x_i|)      */
  float max_abs_err; /* max |e_i|                                     */
  uint64_t n;        /* number of elements                            */
} orc_stats;

/* ---- number-format helpers (bit-by-bit decoders, nearest-value encoders) ---- */
double orc_decode_fp32(uint32_t bits);
double orc_decode_bf16(uint16_t bits);
uint32_t orc_encode_fp32(double v);          /* v must be exactly representable in binary32 */
uint16_t orc_bf16_rne(uint32_t fp32_bits);   /* binary32 -> bf16, round to nearest even     */
double orc_decode_code(int fmt, uint32_t code);   /* ORC_INT8 / INT4 / E4M3 / E5M2 / E2M1 / E8M0 */
uint32_t orc_encode_elem(int fmt, uint32_t v_fp32_bits); /* RNE, saturating, signed zero   */
int orc_mx_scale_exponent(uint32_t t_fp32_bits, int scale_round); /* k of s = 2^k          */
uint32_t orc_nv_block_scale_code(uint32_t t_fp32_bits, int scale_round); /* E4M3 code      */

/* ---- the path ---- */
int orc_amax(int in_dtype, int64_t rows, int64_t cols, int64_t ld, const void* x,
             float* amax_out, int nthreads);

int orc_quantize(int format, int in_dtype, int granularity, int block_size, int scale_round,
                 int64_t rows, int64_t cols, int64_t ld, const void* x,
                 void* codes, void* scales, float* tensor_scale_out,
                 const float* tensor_amax_in, orc_stats* stats_out, int nthreads);

int orc_dequantize(int format, int granularity, int block_size,
                   int64_t rows, int64_t cols, int64_t ld, const void* codes,
                   const void* scales, const float* tensor_scale, void* y, int out_dtype,
                   int nthreads);

int orc_error_stats(int format, int in_dtype, int granularity, int block_size,
                    int64_t rows, int64_t cols, int64_t ld, const void* x, const void* codes,
                    const void* scales, const float* tensor_scale, orc_stats* stats_out,
                    int nthreads);

/* Asymmetric 4-bit group dequantization (section "Puzzles 12 Quantized Matrix Mult" of the
 * blog's Triton post): y[r][c] = sc[r][c/group] * (w[r][c] - sh[r][c/group]).
 *   w       [rows, cols/8] 32-bit words, 8 unsigned 4-bit codes each, element c in bits
 *           [4*(c%8), 4*(c%8)+4) of word c/8 (the puzzle's extract: low nibble first)
 *   scales  [rows, cols/group] fp32
 *   shifts  [rows, ceil((cols/group)/8)] 32-bit words, 8 unsigned 4-bit shifts each, the
 *           same nibble order
 * cols % 8 == 0, group > 0, cols % group == 0.  w - sh is an exact small integer; the
 * product is one binary32 rounding, then y is written as bf16 (RNE) or fp32. */
int orc_dequant_asym4(int64_t rows, int64_t cols, int64_t group, const uint32_t* w,
                      const float* scales, const uint32_t* shifts, void* y, int out_dtype,
                      int nthreads);

/* The puzzle's quantized matrix product z[j][k] = sum_l sc (w[j][l] - sh) * y[l][k]:
 *   w, scales, shifts as orc_dequant_asym4 ([n0, mid] weights in groups of `group`);
 *   y [mid, n1] bf16 bit patterns (row-major, leading dimension n1);
 *   z [n0, n1] double: the dequantized weight taken as the binary32 value of
 *     orc_dequant_asym4's fp32 output, each product and the sum in double -- every product
 *     of a binary32 and a bf16 value is exact in double and the sum of mid of them is
 *     accurate to mid * 2^-53 of the sum of magnitudes;
 *   zabs [n0, n1] double (may be NULL): sum_l |deq * y|, the scale of the rounding error
 *     of any evaluation order. */
int orc_quant_dot(int64_t n0, int64_t mid, int64_t group, int64_t n1, const uint32_t* w,
                  const float* scales, const uint32_t* shifts, const uint16_t* y, double* z,
                  double* zabs, int nthreads);

#ifdef __cplusplus
}
#endif
#endif
