/*
 * qz_oracle.c -- plain, slow, obviously-correct CPU reference for quantizing a tensor to
 * INT8, FP8 E4M3 / E5M2, MXFP4 and NVFP4, dequantizing it, and measuring the error.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, by __graft_entry__.smoke() and by the
 * CPU-baseline leg of bench.py.  The CUDA library never links or calls it.
 *
 * Source of every step: the blog post "浅谈低精度浮点数" ("A brief talk on low-precision
 * floats") on the july-h5kf3.github.io column blog, sections
 *   "IEEE 754 标准浮点数"   binary32 layout, bias 127, hidden bit, worked example 25.125,
 *                            BF16 = 8 exponent + 7 fraction bits;
 *   "FP8"                    E4M3 / E5M2 (2^M samples per binade), symmetric INT8
 *                            x^ = s*round(x/s), q in [-127, 127], s = alpha/127;
 *   "FP4 / MXFP4 / NVFP4"    the E2M1 value set, MXFP4 (32-element blocks, power-of-two
 *                            E8M0 scale s = 2^round(log2(A/6)), rounded up in practice),
 *                            NVFP4 (16-element blocks, E4M3 block scale,
 *                            s_global = global_amax/(6*448),
 *                            s_block = (block_amax/6)/s_global, x^ = s_g*s_b*Q(x/(s_g*s_b)));
 * and the "Puzzles 12 Quantized Matrix Mult" section of the "Triton" post on the same
 * blog, whose extract() helper puts element j of a packed word in bits [4j, 4j+4): the low
 * nibble holds the first element.
 *
 * Readings taken where the post is silent (each also listed in the design notes):
 *  R1 element rounding is round-to-nearest, ties to the code with an even last bit;
 *  R2 values at or beyond the format maximum saturate to +-max;
 *  R3 FP formats keep the sign of zero (a negative value that rounds to zero gives the
 *     sign-only code); INT8 has a single zero;
 *  R4 E5M2 is IEEE-like (bias 15, exponent field 31 = Inf/NaN, max 57344); E4M3 has no
 *     Inf (S.1111.111 is NaN, max 448, which the post states); E8M0 has bias 127 and
 *     code 255 = NaN; E2M1 has bias 1 and no Inf/NaN;
 *  R5 the FP8 scale maps the amax onto the format maximum: s = alpha/448 or alpha/57344;
 *  R6 a per-tensor / per-row scale whose quotient alpha/qmax is zero is replaced by 1;
 *  R7 MXFP4 default scale rounding is UP (smallest 2^k >= A/6); NEAREST rounds log2 to
 *     the nearest integer; k is clamped to [-127, 127];
 *  R8 NVFP4 default block-scale rounding is UP (smallest E4M3 value >= the ideal scale,
 *     saturated at 448); NEAREST is RNE-saturating to E4M3; a zero block scale gives
 *     signed-zero codes; s_global = 0 is replaced by 1;
 *  R9 the fp32 operation order of every scale is the order in which the post writes it;
 *  R10 x/s is rounded to binary32 first and then to the grid (two roundings);
 *  R11 codes and block scales are dense row-major, blocks run along the columns.
 */
#include "qz_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------------------ */
/* binary32 and bf16, field by field ("IEEE 754 标准浮点数")                            */
/* ------------------------------------------------------------------------------------ */

double orc_decode_fp32(uint32_t bits) {
  const int sign = (int)(bits >> 31);
  const int E = (int)((bits >> 23) & 0xFFu); /* biased exponent, bias 127 */
  const uint32_t F = bits & 0x7FFFFFu;       /* 23 fraction bits          */
  double mag;
  if (E == 0)
    mag = ldexp((double)F, -149); /* zero or subnormal: 0.F x 2^-126 */
  else if (E == 255)
    mag = F ? NAN : INFINITY;
  else
    mag = ldexp((double)(F + 0x800000u), E - 150); /* hidden bit: 1.F x 2^(E-127) */
  return sign ? -mag : mag;
}

double orc_decode_bf16(uint16_t bits) {
  /* 1 sign, 8 exponent (bias 127), 7 fraction bits */
  const int sign = (bits >> 15) & 1;
  const int E = (bits >> 7) & 0xFF;
  const unsigned F = bits & 0x7Fu;
  double mag;
  if (E == 0)
    mag = ldexp((double)F, -133); /* 0.F x 2^-126 with 7 fraction bits */
  else if (E == 255)
    mag = F ? NAN : INFINITY;
  else
    mag = ldexp((double)(F + 128u), E - 134); /* 1.F x 2^(E-127) */
  return sign ? -mag : mag;
}

uint32_t orc_encode_fp32(double v) {
  const uint32_t sign = signbit(v) ? 0x80000000u : 0u;
  if (isnan(v)) return 0x7FC00000u;
  const double a = fabs(v);
  if (isinf(a)) return sign | 0x7F800000u;
  if (a == 0.0) return sign;
  int e;
  const double m = frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) -> a = 2m * 2^(e-1) */
  const int E = e - 1 + 127;
  if (E >= 1) {
    const double frac = ldexp(m, 24) - 8388608.0; /* (2m - 1) * 2^23 */
    return sign | ((uint32_t)E << 23) | (uint32_t)frac;
  }
  return sign | (uint32_t)ldexp(a, 149); /* subnormal: a = F * 2^-149 */
}

uint16_t orc_bf16_rne(uint32_t fp32_bits) {
  const double v = orc_decode_fp32(fp32_bits);
  if (isnan(v)) return 0x7FC0u;
  const int neg = signbit(v) ? 1 : 0;
  const double a = fabs(v);
  const uint16_t sgn = (uint16_t)(neg ? 0x8000u : 0u);
  if (isinf(a)) return (uint16_t)(sgn | 0x7F80u);
  double q = 0.0;
  if (a != 0.0) {
    int e;
    frexp(a, &e);
    int E = e - 1; /* a in [2^E, 2^(E+1)) */
    if (E < -126) E = -126;
    const double sp = ldexp(1.0, E - 7); /* bf16 spacing in this binade */
    const double lo = floor(a / sp) * sp, hi = lo + sp;
    const double dl = a - lo, dh = hi - a;
    if (dl < dh)
      q = lo;
    else if (dh < dl)
      q = hi;
    else
      q = (fmod(lo / sp, 2.0) == 0.0) ? lo : hi; /* tie: even last fraction bit */
  }
  if (q >= 0x1p128) return (uint16_t)(sgn | 0x7F80u); /* rounds past the largest: Inf */
  return (uint16_t)(sgn | (uint16_t)(orc_encode_fp32(q) >> 16));
}

/* ------------------------------------------------------------------------------------ */
/* element formats, decoded bit by bit ("FP8", "FP4 / MXFP4 / NVFP4")                   */
/* ------------------------------------------------------------------------------------ */

static double dec_int8(uint32_t c) {
  int v = (int)(c & 0xFFu);
  if (v >= 128) v -= 256;
  return (double)v;
}

/* INT4: a 4-bit two's complement nibble ("FP4 / MXFP4 / NVFP4", last paragraph: symmetric
 * INT4 with q in [-7, 7]); the pattern 1000 (-8) is decodable but never produced */
static double dec_int4(uint32_t c) {
  int v = (int)(c & 0xFu);
  if (v >= 8) v -= 16;
  return (double)v;
}

static double dec_e4m3(uint32_t c) { /* bias 7, no Inf, S.1111.111 = NaN */
  const int s = (int)((c >> 7) & 1u), e = (int)((c >> 3) & 0xFu), m = (int)(c & 7u);
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m, -9); /* m/8 x 2^-6 */
  else
    mag = ldexp((double)(8 + m), e - 10); /* (1 + m/8) x 2^(e-7) */
  return s ? -mag : mag;
}

static double dec_e5m2(uint32_t c) { /* bias 15, IEEE-like specials */
  const int s = (int)((c >> 7) & 1u), e = (int)((c >> 2) & 0x1Fu), m = (int)(c & 3u);
  double mag;
  if (e == 31) {
    if (m) return NAN;
    return s ? -INFINITY : INFINITY;
  }
  if (e == 0)
    mag = ldexp((double)m, -16); /* m/4 x 2^-14 */
  else
    mag = ldexp((double)(4 + m), e - 17); /* (1 + m/4) x 2^(e-15) */
  return s ? -mag : mag;
}

static double dec_e2m1(uint32_t c) { /* bias 1, no specials */
  const int s = (int)((c >> 3) & 1u), e = (int)((c >> 1) & 3u), m = (int)(c & 1u);
  double mag;
  if (e == 0)
    mag = 0.5 * m; /* m/2 x 2^0 */
  else
    mag = ldexp((double)(2 + m), e - 2); /* (1 + m/2) x 2^(e-1) */
  return s ? -mag : mag;
}

static double dec_e8m0(uint32_t c) { /* power of two, bias 127, 255 = NaN */
  c &= 0xFFu;
  if (c == 255u) return NAN;
  return ldexp(1.0, (int)c - 127);
}

double orc_decode_code(int fmt, uint32_t code) {
  switch (fmt) {
    case ORC_INT8: return dec_int8(code);
    case ORC_INT4: return dec_int4(code);
    case ORC_E4M3: return dec_e4m3(code);
    case ORC_E5M2: return dec_e5m2(code);
    case ORC_E2M1: return dec_e2m1(code);
    case ORC_E8M0: return dec_e8m0(code);
    default: return NAN;
  }
}

/* Table of a format's finite non-negative values, in code order (which is value order). */
typedef struct {
  int n;
  double val[128];
  uint32_t code[128];
} grid_t;

static grid_t G_INT8, G_INT4, G_E4M3, G_E5M2, G_E2M1;
static int grids_ready = 0;

static void fill_grid(grid_t* g, int fmt, uint32_t ncodes) {
  g->n = 0;
  for (uint32_t c = 0; c < ncodes; ++c) {
    const double v = orc_decode_code(fmt, c);
    if (!isfinite(v)) continue;
    g->val[g->n] = v;
    g->code[g->n] = c;
    g->n++;
  }
}

static void init_grids(void) {
  if (grids_ready) return;
#ifdef _OPENMP
#pragma omp critical(orc_grids)
#endif
  {
    if (!grids_ready) {
      fill_grid(&G_INT8, ORC_INT8, 128); /* 0..127: q in [-127, 127] */
      fill_grid(&G_INT4, ORC_INT4, 8);   /* 0..7: q in [-7, 7] */
      fill_grid(&G_E4M3, ORC_E4M3, 128);
      fill_grid(&G_E5M2, ORC_E5M2, 128);
      fill_grid(&G_E2M1, ORC_E2M1, 8);
      grids_ready = 1;
    }
  }
}

static const grid_t* grid_of(int fmt) {
  switch (fmt) {
    case ORC_INT8: return &G_INT8;
    case ORC_INT4: return &G_INT4;
    case ORC_E4M3: return &G_E4M3;
    case ORC_E5M2: return &G_E5M2;
    case ORC_E2M1:
    case ORC_MXFP4:
    case ORC_NVFP4: return &G_E2M1;
    default: return NULL;
  }
}

/* Index of the nearest table value to a >= 0 (R1 ties to an even code, R2 saturate). */
static int nearest_index(const grid_t* g, double a) {
  if (a >= g->val[g->n - 1]) return g->n - 1;
  int lo = 0, hi = g->n - 1; /* val[lo] <= a < val[hi] */
  while (hi - lo > 1) {
    const int mid = (lo + hi) / 2;
    if (g->val[mid] <= a)
      lo = mid;
    else
      hi = mid;
  }
  const double dl = a - g->val[lo], dh = g->val[hi] - a; /* exact in double */
  if (dl < dh) return lo;
  if (dh < dl) return hi;
  return (g->code[lo] & 1u) ? hi : lo;
}

/* Element code of the binary32 value v (R1, R2, R3). */
static uint32_t encode_value(int fmt, double v) {
  const grid_t* g = grid_of(fmt);
  const int neg = signbit(v) ? 1 : 0;
  const uint32_t mag = g->code[nearest_index(g, fabs(v))];
  if (fmt == ORC_INT8) return neg ? ((256u - mag) & 0xFFu) : mag;
  if (fmt == ORC_INT4) return neg ? ((16u - mag) & 0xFu) : mag; /* one zero, like INT8 */
  if (fmt == ORC_E4M3 || fmt == ORC_E5M2) return mag | (neg ? 0x80u : 0u);
  return mag | (neg ? 0x8u : 0u); /* E2M1 nibble */
}

uint32_t orc_encode_elem(int fmt, uint32_t v_fp32_bits) {
  init_grids();
  if (!grid_of(fmt)) return 0;
  return encode_value(fmt, orc_decode_fp32(v_fp32_bits));
}

/* MXFP4 scale exponent k, s = 2^k, from t = fl(A/6) (R7). */
static int mx_exponent(double t, int scale_round) {
  if (t == 0.0) return -127;
  int e;
  const double sig = 2.0 * frexp(t, &e); /* t = sig * 2^E, sig in [1, 2) */
  const int E = e - 1;
  int k;
  if (scale_round == ORC_SCALE_NEAREST)
    k = (sig * sig > 2.0) ? E + 1 : E; /* log2(sig) > 1/2  <=>  sig^2 > 2 (exact) */
  else
    k = (sig == 1.0) ? E : E + 1; /* smallest k with 2^k >= t */
  if (k < -127) k = -127;
  if (k > 127) k = 127;
  return k;
}

int orc_mx_scale_exponent(uint32_t t_fp32_bits, int scale_round) {
  return mx_exponent(orc_decode_fp32(t_fp32_bits), scale_round);
}

/* NVFP4 E4M3 block-scale code from the ideal scale t (R8). */
static uint32_t nv_block_code(double t, int scale_round) {
  const grid_t* g = &G_E4M3;
  if (scale_round == ORC_SCALE_NEAREST) return g->code[nearest_index(g, t)];
  if (t >= g->val[g->n - 1]) return g->code[g->n - 1]; /* saturate at 448 */
  for (int i = 0; i < g->n; ++i) /* smallest value >= t */
    if (g->val[i] >= t) return g->code[i];
  return g->code[g->n - 1];
}

uint32_t orc_nv_block_scale_code(uint32_t t_fp32_bits, int scale_round) {
  init_grids();
  return nv_block_code(orc_decode_fp32(t_fp32_bits), scale_round);
}

/* ------------------------------------------------------------------------------------ */
/* tensor access                                                                        */
/* ------------------------------------------------------------------------------------ */

static float load_x(const void* x, int dt, int64_t idx) {
  if (dt == ORC_BF16) {
    uint16_t h;
    memcpy(&h, (const char*)x + 2 * idx, 2);
    return (float)orc_decode_bf16(h);
  }
  uint32_t b;
  memcpy(&b, (const char*)x + 4 * idx, 4);
  return (float)orc_decode_fp32(b);
}

static void store_y(void* y, int dt, int64_t idx, float v) {
  const uint32_t b = orc_encode_fp32((double)v);
  if (dt == ORC_BF16) {
    const uint16_t h = orc_bf16_rne(b);
    memcpy((char*)y + 2 * idx, &h, 2);
  } else {
    memcpy((char*)y + 4 * idx, &b, 4);
  }
}

static uint32_t get_byte(const void* p, int64_t i) { return ((const uint8_t*)p)[i]; }
static void put_byte(void* p, int64_t i, uint32_t v) { ((uint8_t*)p)[i] = (uint8_t)v; }

/* FP4 nibble j of a row: element 2i in the low nibble of byte i, 2i+1 in the high nibble */
static uint32_t get_nibble(const void* codes, int64_t row_off, int64_t c) {
  const uint32_t b = get_byte(codes, row_off + c / 2);
  return (c & 1) ? (b >> 4) : (b & 0xFu);
}

static void put_nibble(void* codes, int64_t row_off, int64_t c, uint32_t v) {
  uint8_t* p = (uint8_t*)codes + row_off + c / 2;
  if (c & 1)
    *p = (uint8_t)((*p & 0x0Fu) | (v << 4));
  else
    *p = (uint8_t)((*p & 0xF0u) | (v & 0xFu));
}

static float get_f32(const void* p, int64_t i) {
  uint32_t b;
  memcpy(&b, (const char*)p + 4 * i, 4);
  return (float)orc_decode_fp32(b);
}

static void put_f32(void* p, int64_t i, float v) {
  const uint32_t b = orc_encode_fp32((double)v);
  memcpy((char*)p + 4 * i, &b, 4);
}

static int is8bit(int f) { return f == ORC_INT8 || f == ORC_E4M3 || f == ORC_E5M2; }

static float qmax_of(int f) { /* largest finite value of the element format */
  init_grids();
  const grid_t* g = grid_of(f);
  return (float)g->val[g->n - 1];
}

static int check_shape(int format, int granularity, int block_size, int64_t rows,
                       int64_t cols, int64_t ld) {
  if (rows < 0 || cols < 0 || ld < cols) return ORC_ERR_ARG;
  if (is8bit(format)) {
    if (granularity != ORC_GRAN_TENSOR && granularity != ORC_GRAN_ROW &&
        granularity != ORC_GRAN_UNIT)
      return ORC_ERR_ARG;
  } else if (format == ORC_INT4) {
    if (granularity != ORC_GRAN_BLOCK) return ORC_ERR_ARG;
    if (block_size != 16 && block_size != 32 && block_size != 64 && block_size != 128)
      return ORC_ERR_ARG;
    if (cols % block_size) return ORC_ERR_ARG;
  } else if (format == ORC_MXFP4 || format == ORC_NVFP4) {
    const int bs = (format == ORC_MXFP4) ? 32 : 16;
    if (block_size != bs) return ORC_ERR_ARG;
    if (granularity != ORC_GRAN_BLOCK && granularity != ORC_GRAN_UNIT) return ORC_ERR_ARG;
    if (cols % bs) return ORC_ERR_ARG;
  } else {
    return ORC_ERR_ARG;
  }
  return ORC_OK;
}

static int nthreads_of(int nt) {
#ifdef _OPENMP
  return nt > 0 ? nt : omp_get_max_threads();
#else
  (void)nt;
  return 1;
#endif
}

/* max |x| over the tensor; ORC_ERR_NONFINITE if any element is NaN or Inf */
static int amax_all(int dt, int64_t rows, int64_t cols, int64_t ld, const void* x, float* out,
                    int nt) {
  float m = 0.0f;
  int bad = 0;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nt) reduction(max : m) reduction(| : bad)
#endif
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t c = 0; c < cols; ++c) {
      const float v = load_x(x, dt, r * ld + c);
      if (!isfinite(v)) bad = 1;
      const float a = fabsf(v);
      if (a > m) m = a;
    }
  }
  (void)nt;
  *out = m;
  return bad ? ORC_ERR_NONFINITE : ORC_OK;
}

int orc_amax(int in_dtype, int64_t rows, int64_t cols, int64_t ld, const void* x,
             float* amax_out, int nthreads) {
  if (!amax_out || rows < 0 || cols < 0 || ld < cols) return ORC_ERR_ARG;
  if (in_dtype != ORC_BF16 && in_dtype != ORC_F32) return ORC_ERR_ARG;
  if (rows * cols > 0 && !x) return ORC_ERR_ARG;
  return amax_all(in_dtype, rows, cols, ld, x, amax_out, nthreads_of(nthreads));
}

/* R6: per-tensor / per-row scale s = alpha / qmax, replaced by 1 when the quotient is 0 */
static float scale_from_amax(float alpha, float qmax) {
  float s = alpha / qmax;
  if (s == 0.0f) s = 1.0f;
  return s;
}

/* per-row error accumulators, combined in row order so the sum does not depend on the
 * thread count */
typedef struct {
  double sum_sq;
  float max_abs, max_rel;
} row_acc;

static void acc_elem(row_acc* a, float x, float xh) {
  const float e = x - xh;
  const float ae = fabsf(e);
  a->sum_sq += (double)e * (double)e;
  if (ae > a->max_abs) a->max_abs = ae;
  if (x != 0.0f) {
    const float rel = ae / fabsf(x);
    if (rel > a->max_rel) a->max_rel = rel;
  }
}

static void finish_stats(orc_stats* st, const row_acc* acc, int64_t rows, int64_t n) {
  double s = 0.0;
  float ma = 0.0f, mr = 0.0f;
  for (int64_t r = 0; r < rows; ++r) {
    s += acc[r].sum_sq;
    if (acc[r].max_abs > ma) ma = acc[r].max_abs;
    if (acc[r].max_rel > mr) mr = acc[r].max_rel;
  }
  st->sum_sq_err = s;
  st->mse = n > 0 ? s / (double)n : 0.0;
  st->max_abs_err = ma;
  st->max_rel_err = mr;
  st->n = (uint64_t)n;
}

/* Per-tensor scale of the tensor (8-bit TENSOR: s; NVFP4 BLOCK: s_global; else 1). */
static float tensor_scale_of(int format, int granularity, float alpha) {
  if (is8bit(format) && granularity == ORC_GRAN_TENSOR)
    return scale_from_amax(alpha, qmax_of(format));
  if (format == ORC_NVFP4 && granularity == ORC_GRAN_BLOCK) {
    float sg = alpha / 2688.0f; /* global_amax / (6 * 448) */
    if (sg == 0.0f) sg = 1.0f;
    return sg;
  }
  return 1.0f;
}

/* ------------------------------------------------------------------------------------ */
/* quantize                                                                             */
/* ------------------------------------------------------------------------------------ */

/* One row; acc may be NULL. */
static void quantize_row(int format, int dt, int granularity, int scale_round, int block_size,
                         int64_t r, int64_t cols, int64_t ld, const void* x, void* codes,
                         void* scales, float tscale, row_acc* acc) {
  const int64_t xo = r * ld;
  if (is8bit(format)) {
    float s;
    if (granularity == ORC_GRAN_ROW) {
      float a = 0.0f;
      for (int64_t c = 0; c < cols; ++c) {
        const float v = fabsf(load_x(x, dt, xo + c));
        if (v > a) a = v;
      }
      s = scale_from_amax(a, qmax_of(format));
      put_f32(scales, r, s);
    } else {
      s = (granularity == ORC_GRAN_TENSOR) ? tscale : 1.0f;
    }
    for (int64_t c = 0; c < cols; ++c) {
      const float xv = load_x(x, dt, xo + c);
      const float v = xv / s; /* fl32(x / s) */
      const uint32_t q = encode_value(format, (double)v);
      put_byte(codes, r * cols + c, q);
      if (acc) acc_elem(acc, xv, (float)orc_decode_code(format, q) * s);
    }
    return;
  }
  if (format == ORC_INT4) { /* symmetric INT4: s = A / 7 per group (R6 for A = 0) */
    const int64_t nb = cols / block_size, co = r * (cols / 2);
    for (int64_t b = 0; b < nb; ++b) {
      float A = 0.0f;
      for (int i = 0; i < block_size; ++i) {
        const float v = fabsf(load_x(x, dt, xo + b * block_size + i));
        if (v > A) A = v;
      }
      const float s = scale_from_amax(A, 7.0f);
      put_f32(scales, r * nb + b, s);
      for (int i = 0; i < block_size; ++i) {
        const int64_t c = b * block_size + i;
        const float xv = load_x(x, dt, xo + c);
        const uint32_t q = encode_value(ORC_INT4, (double)(xv / s));
        put_nibble(codes, co, c, q);
        if (acc) acc_elem(acc, xv, (float)dec_int4(q) * s);
      }
    }
    return;
  }
  const int bs = (format == ORC_MXFP4) ? 32 : 16;
  const int64_t nb = cols / bs, co = r * (cols / 2);
  for (int64_t b = 0; b < nb; ++b) {
    float A = 0.0f;
    for (int i = 0; i < bs; ++i) {
      const float v = fabsf(load_x(x, dt, xo + b * bs + i));
      if (v > A) A = v;
    }
    float s;
    uint32_t scode;
    if (format == ORC_MXFP4) {
      int k = 0;
      if (granularity == ORC_GRAN_BLOCK) k = mx_exponent((double)(A / 6.0f), scale_round);
      scode = (uint32_t)(k + 127);
      s = (float)ldexp(1.0, k); /* exact, 2^-127 is a binary32 subnormal */
    } else {
      if (granularity == ORC_GRAN_BLOCK) {
        const float t = (A / 6.0f) / tscale; /* (block_amax / 6) / s_global */
        scode = nv_block_code((double)t, scale_round);
      } else {
        scode = 0x38u; /* E4M3 1.0 */
      }
      s = tscale * (float)dec_e4m3(scode); /* s_global * s_block */
    }
    put_byte(scales, r * nb + b, scode);
    for (int i = 0; i < bs; ++i) {
      const int64_t c = b * bs + i;
      const float xv = load_x(x, dt, xo + c);
      uint32_t q;
      if (s == 0.0f)
        q = signbit(xv) ? 0x8u : 0x0u; /* zero block scale: signed-zero code */
      else
        q = encode_value(ORC_E2M1, (double)(xv / s));
      put_nibble(codes, co, c, q);
      if (acc) acc_elem(acc, xv, (float)dec_e2m1(q) * s);
    }
  }
}

int orc_quantize(int format, int in_dtype, int granularity, int block_size, int scale_round,
                 int64_t rows, int64_t cols, int64_t ld, const void* x, void* codes,
                 void* scales, float* tensor_scale_out, const float* tensor_amax_in,
                 orc_stats* stats_out, int nthreads) {
  init_grids();
  if (check_shape(format, granularity, block_size, rows, cols, ld)) return ORC_ERR_ARG;
  if (in_dtype != ORC_BF16 && in_dtype != ORC_F32) return ORC_ERR_ARG;
  if (scale_round != ORC_SCALE_UP && scale_round != ORC_SCALE_NEAREST) return ORC_ERR_ARG;
  const int64_t n = rows * cols;
  const int nt = nthreads_of(nthreads);
  const int need_scales = (granularity == ORC_GRAN_ROW) || format == ORC_MXFP4 ||
                          format == ORC_NVFP4 || format == ORC_INT4;
  if (n > 0 && (!x || !codes || (need_scales && !scales))) return ORC_ERR_ARG;

  float alpha = 0.0f;
  {
    const int rc = amax_all(in_dtype, rows, cols, ld, x, &alpha, nt); /* also finiteness */
    if (rc) return rc;
  }
  if (tensor_amax_in) {
    if (!(*tensor_amax_in >= 0.0f) || isinf(*tensor_amax_in)) return ORC_ERR_ARG;
    alpha = *tensor_amax_in;
  }
  const float tscale = tensor_scale_of(format, granularity, alpha);
  if (tensor_scale_out) *tensor_scale_out = tscale;

  row_acc* acc = NULL;
  if (stats_out) {
    acc = (row_acc*)calloc((size_t)(rows > 0 ? rows : 1), sizeof(row_acc));
    if (!acc) return ORC_ERR_ARG;
  }
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nt)
#endif
  for (int64_t r = 0; r < rows; ++r)
    quantize_row(format, in_dtype, granularity, scale_round, block_size, r, cols, ld, x, codes,
                 scales, tscale, acc ? &acc[r] : NULL);
  if (stats_out) {
    finish_stats(stats_out, acc, rows, n);
    free(acc);
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------------------ */
/* dequantize and standalone error statistics                                           */
/* ------------------------------------------------------------------------------------ */

/* x^ of element (r, c): decode(q) * s, s as in quantize */
static float dequant_elem(int format, int granularity, int block_size, int64_t r, int64_t c,
                          int64_t cols, const void* codes, const void* scales, float tscale) {
  if (format == ORC_INT4) {
    const float s = get_f32(scales, r * (cols / block_size) + c / block_size);
    return (float)dec_int4(get_nibble(codes, r * (cols / 2), c)) * s;
  }
  if (is8bit(format)) {
    float s = 1.0f;
    if (granularity == ORC_GRAN_ROW) s = get_f32(scales, r);
    if (granularity == ORC_GRAN_TENSOR) s = tscale;
    return (float)orc_decode_code(format, get_byte(codes, r * cols + c)) * s;
  }
  const int bs = (format == ORC_MXFP4) ? 32 : 16;
  const int64_t nb = cols / bs;
  const uint32_t sc = get_byte(scales, r * nb + c / bs);
  float s;
  if (format == ORC_MXFP4)
    s = (float)dec_e8m0(sc);
  else
    s = tscale * (float)dec_e4m3(sc);
  return (float)dec_e2m1(get_nibble(codes, r * (cols / 2), c)) * s;
}

int orc_dequantize(int format, int granularity, int block_size, int64_t rows, int64_t cols,
                   int64_t ld, const void* codes, const void* scales,
                   const float* tensor_scale, void* y, int out_dtype, int nthreads) {
  init_grids();
  if (check_shape(format, granularity, block_size, rows, cols, ld)) return ORC_ERR_ARG;
  if (out_dtype != ORC_BF16 && out_dtype != ORC_F32) return ORC_ERR_ARG;
  const int64_t n = rows * cols;
  if (n == 0) return ORC_OK;
  const int need_scales = (granularity == ORC_GRAN_ROW) || format == ORC_MXFP4 ||
                          format == ORC_NVFP4 || format == ORC_INT4;
  const int need_ts = (is8bit(format) && granularity == ORC_GRAN_TENSOR) ||
                      (format == ORC_NVFP4 && granularity == ORC_GRAN_BLOCK);
  if (!codes || !y || (need_scales && !scales) || (need_ts && !tensor_scale))
    return ORC_ERR_ARG;
  const float ts = need_ts ? *tensor_scale : 1.0f;
  const int nt = nthreads_of(nthreads);
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nt)
#endif
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c)
      store_y(y, out_dtype, r * ld + c,
              dequant_elem(format, granularity, block_size, r, c, cols, codes, scales, ts));
  (void)nt;
  return ORC_OK;
}

int orc_error_stats(int format, int in_dtype, int granularity, int block_size, int64_t rows,
                    int64_t cols, int64_t ld, const void* x, const void* codes,
                    const void* scales, const float* tensor_scale, orc_stats* stats_out,
                    int nthreads) {
  init_grids();
  if (!stats_out) return ORC_ERR_ARG;
  if (check_shape(format, granularity, block_size, rows, cols, ld)) return ORC_ERR_ARG;
  if (in_dtype != ORC_BF16 && in_dtype != ORC_F32) return ORC_ERR_ARG;
  const int64_t n = rows * cols;
  const int need_scales = (granularity == ORC_GRAN_ROW) || format == ORC_MXFP4 ||
                          format == ORC_NVFP4 || format == ORC_INT4;
  const int need_ts = (is8bit(format) && granularity == ORC_GRAN_TENSOR) ||
                      (format == ORC_NVFP4 && granularity == ORC_GRAN_BLOCK);
  if (n > 0 && (!x || !codes || (need_scales && !scales) || (need_ts && !tensor_scale)))
    return ORC_ERR_ARG;
  const int nt = nthreads_of(nthreads);
  float dummy;
  const int rc = amax_all(in_dtype, rows, cols, ld, x, &dummy, nt);
  if (rc) return rc;
  const float ts = (need_ts && n > 0) ? *tensor_scale : 1.0f;
  row_acc* acc = (row_acc*)calloc((size_t)(rows > 0 ? rows : 1), sizeof(row_acc));
  if (!acc) return ORC_ERR_ARG;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nt)
#endif
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c)
      acc_elem(&acc[r], load_x(x, in_dtype, r * ld + c),
               dequant_elem(format, granularity, block_size, r, c, cols, codes, scales, ts));
  finish_stats(stats_out, acc, rows, n);
  free(acc);
  return ORC_OK;
}

/* ------------------------------------------------------------------------------------ */
/* asymmetric 4-bit group dequantization ("Puzzles 12 Quantized Matrix Mult")             */
/* ------------------------------------------------------------------------------------ */

/* nibble i of a 32-bit word, low nibble first */
static uint32_t word_nibble(const uint32_t* words, int64_t i) {
  return (words[i / 8] >> (4 * (i % 8))) & 0xFu;
}

int orc_dequant_asym4(int64_t rows, int64_t cols, int64_t group, const uint32_t* w,
                      const float* scales, const uint32_t* shifts, void* y, int out_dtype,
                      int nthreads) {
  if (rows < 0 || cols < 0 || group <= 0 || cols % 8 || cols % group) return ORC_ERR_ARG;
  if (out_dtype != ORC_BF16 && out_dtype != ORC_F32) return ORC_ERR_ARG;
  if (rows * cols == 0) return ORC_OK;
  if (!w || !scales || !shifts || !y) return ORC_ERR_ARG;
  const int64_t ng = cols / group, sw = (ng + 7) / 8;
  const int nt = nthreads_of(nthreads);
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nt)
#endif
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t c = 0; c < cols; ++c) {
      const int64_t j = c / group;
      const int q = (int)word_nibble(w + r * (cols / 8), c);
      const int sh = (int)word_nibble(shifts + r * sw, j);
      const float d = (float)(q - sh); /* exact: |q - sh| <= 15 */
      store_y(y, out_dtype, r * cols + c, get_f32(scales, r * ng + j) * d);
    }
  }
  (void)nt;
  return ORC_OK;
}

int orc_quant_dot(int64_t n0, int64_t mid, int64_t group, int64_t n1, const uint32_t* w,
                  const float* scales, const uint32_t* shifts, const uint16_t* y, double* z,
                  double* zabs, int nthreads) {
  if (n0 < 0 || mid < 0 || n1 < 0 || group <= 0 || mid % 8 || mid % group) return ORC_ERR_ARG;
  if (n0 * n1 == 0) return ORC_OK;
  if (!w || !scales || !shifts || !y || !z) return ORC_ERR_ARG;
  const int64_t ng = mid / group, sw = (ng + 7) / 8;
  const int nt = nthreads_of(nthreads);
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nt)
#endif
  for (int64_t j = 0; j < n0; ++j) {
    for (int64_t k = 0; k < n1; ++k) {
      double s = 0.0, sa = 0.0;
      for (int64_t l = 0; l < mid; ++l) {
        const int64_t g = l / group;
        const int q = (int)word_nibble(w + j * (mid / 8), l);
        const int sh = (int)word_nibble(shifts + j * sw, g);
        const float deq = get_f32(scales, j * ng + g) * (float)(q - sh); /* one binary32 rounding */
        const double p = (double)deq * orc_decode_bf16(y[l * n1 + k]);
        s += p;
        sa += fabs(p);
      }
      z[j * n1 + k] = s;
      if (zabs) zabs[j * n1 + k] = sa;
    }
  }
  (void)nt;
  return ORC_OK;
}
