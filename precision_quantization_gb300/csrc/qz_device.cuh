// qz_device.cuh -- device-side building blocks of libqz (sm_103a).
//
// Number formats and rules follow the blog post "浅谈低精度浮点数" (sections "FP8" and
// "FP4 / MXFP4 / NVFP4"); the exact semantics are spelled out in include/qz.h.
//
// Build requirement: compiled with --fmad=false and without fast-math, so every fp32
// operation written as a separate multiply / add stays a separately rounded IEEE
// operation and subnormals are kept (no flush to zero).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "qz.h"

namespace qz {

constexpr uint32_t kFull = 0xffffffffu;
constexpr int kThreads = 256;  // threads per CTA of the streaming kernels
constexpr int kWarps = kThreads / 32;

// ---------------------------------------------------------------------------------------
// workspace layout (caller-allocated, zeroed once; every call leaves it reusable)
// ---------------------------------------------------------------------------------------
constexpr int kMaxCtas = 4096;  // upper bound of any grid that writes partials
struct WsHeader {
  uint32_t status;        // QZ_FLAG_* bits, sticky
  uint32_t amax_counter;  // CTAs of the amax pass that are done (wraps to 0)
  uint32_t stats_counter; // CTAs of a stats reduction that are done (wraps to 0)
  float amax;             // result of the last in-library amax pass
  uint32_t pad[60];
};
struct StatPartial {
  double sum_sq;
  float max_abs;
  float max_rel;
};
constexpr size_t kWsAmaxOff = sizeof(WsHeader);
constexpr size_t kWsStatsOff = kWsAmaxOff + sizeof(float) * kMaxCtas;
constexpr size_t kWsBytes = kWsStatsOff + sizeof(StatPartial) * kMaxCtas;
static_assert(sizeof(WsHeader) == 256, "header size");

__device__ __forceinline__ WsHeader* ws_header(void* ws) { return reinterpret_cast<WsHeader*>(ws); }
__device__ __forceinline__ float* ws_amax_partials(void* ws) {
  return reinterpret_cast<float*>(static_cast<char*>(ws) + kWsAmaxOff);
}
__device__ __forceinline__ StatPartial* ws_stat_partials(void* ws) {
  return reinterpret_cast<StatPartial*>(static_cast<char*>(ws) + kWsStatsOff);
}

// ---------------------------------------------------------------------------------------
// global memory access
// ---------------------------------------------------------------------------------------
// 32 contiguous bytes, read-only, not kept in L1 (each byte of x is read once per pass).
__device__ __forceinline__ void ld32B(uint32_t (&w)[8], const void* p) {
  asm volatile(
      "ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]),
        "=r"(w[7])
      : "l"(p));
}
__device__ __forceinline__ void st32B(void* p, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]),
               "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}
__device__ __forceinline__ uint4 ld16B(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ld8B(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld4B(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld1B(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.u8 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// ---------------------------------------------------------------------------------------
// high-precision element access: DT = QZ_BF16 (2 bytes) or QZ_F32 (4 bytes)
// ---------------------------------------------------------------------------------------
template <int DT>
struct Elem {
  static constexpr int kBytes = DT == QZ_BF16 ? 2 : 4;
  static constexpr int kPer32B = 32 / kBytes;  // elements per 32-byte chunk
};

// Widen element i of a 32-byte chunk (bf16 -> fp32 is exact: the top half of binary32).
template <int DT>
__device__ __forceinline__ float chunk_elem(const uint32_t (&w)[8], int i) {
  if constexpr (DT == QZ_BF16) {
    const uint32_t v = w[i >> 1];
    return (i & 1) ? __uint_as_float(v & 0xffff0000u) : __uint_as_float(v << 16);
  } else {
    return __uint_as_float(w[i]);
  }
}

template <int DT>
__device__ __forceinline__ float load_elem(const void* x, int64_t idx) {
  if constexpr (DT == QZ_BF16) {
    const uint16_t h = static_cast<const uint16_t*>(x)[idx];
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  } else {
    return static_cast<const float*>(x)[idx];
  }
}

template <int DT>
__device__ __forceinline__ void store_elem(void* y, int64_t idx, float v) {
  if constexpr (DT == QZ_BF16) {
    uint16_t h;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(v));
    static_cast<uint16_t*>(y)[idx] = h;
  } else {
    static_cast<float*>(y)[idx] = v;
  }
}

// Largest magnitude with NaN propagation (a NaN input makes the result NaN).
__device__ __forceinline__ float absmax_nan(float m, float x) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(m), "f"(fabsf(x)));
  return d;
}

__device__ __forceinline__ bool is_finite_f(float a) { return fabsf(a) <= 3.402823466e38f; }

// ---------------------------------------------------------------------------------------
// exact division
// ---------------------------------------------------------------------------------------
// fl32(x / s) from r = RN(1/s) with one FMA correction (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. R&D 34(1), 1990:
// with y the correctly rounded reciprocal, q = RN(x*y), r = x - s*q exact by FMA,
// RN(q + r*y) is the correctly rounded quotient).  Exact when s, 1/s and the quotient are
// normal binary32 numbers and x is not tiny; callers guard the ranges where that fails
// (fast_div_ok) and use __fdiv_rn there.
// The quotient of x by s > 0 has the sign of x; the correction step alone would turn
// x = -0 into +0 (fma(+0, r, -0) = +0), so the sign is copied from x.
__device__ __forceinline__ float div_by(float x, float s, float r) {
  const float q = __fmul_rn(x, r);
  const float rem = __fmaf_rn(-q, s, x);
  return copysignf(__fmaf_rn(rem, r, q), x);
}

// Range in which div_by is exact for every quotient that can change a code: s in
// [2^-80, 2^126] keeps 1/s a normal number, and every x whose quotient reaches the first
// rounding threshold of any element format (>= 2^-18) has |x| >= 2^-98, far from
// underflow.  Every scale computed from a finite amax lies below 2^126 (INT8 <= 2^121,
// NVFP4 <= 2^125.4).  The quotients themselves must stay below 2^126 (callers check the
// block / chunk amax times 1/s where a supplied amax could make them larger).
__device__ __forceinline__ bool fast_div_ok(float s) {
  return s >= 0x1p-80f && s <= 0x1p126f;
}

// ---------------------------------------------------------------------------------------
// element casts (round to nearest even, saturating; cvt .satfinite)
// ---------------------------------------------------------------------------------------
// two fp32 -> E2M1 pair in one byte; `lo` ends up in bits [0,4), `hi` in bits [4,8)
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}
// two fp32 -> FP8 pair in 16 bits; `lo` in bits [0,8)
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t cvt_e5m2x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// fp32 -> INT8 in [-127, 127] (two's complement byte); round to nearest even
__device__ __forceinline__ uint32_t cvt_int8(float v) {
  int q = __float2int_rn(v);
  q = max(-127, min(127, q));
  return static_cast<uint32_t>(q) & 0xffu;
}

template <int FMT>
__device__ __forceinline__ uint32_t cvt8x2(float lo, float hi) {
  if constexpr (FMT == QZ_FP8_E4M3) return cvt_e4m3x2(lo, hi);
  else if constexpr (FMT == QZ_FP8_E5M2) return cvt_e5m2x2(lo, hi);
  else return cvt_int8(lo) | (cvt_int8(hi) << 8);
}

// decoders: packed codes -> two f16 values (exact for every code of these formats)
__device__ __forceinline__ void f16x2_to_f32(uint32_t h2, float& lo, float& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h2));
}
__device__ __forceinline__ void dec_e2m1x2(uint32_t byte, float& lo, float& hi) {
  uint32_t h2;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(h2)
      : "r"(byte));
  f16x2_to_f32(h2, lo, hi);
}
__device__ __forceinline__ void dec_e4m3x2(uint32_t pair, float& lo, float& hi) {
  uint32_t h2;
  const uint16_t p = static_cast<uint16_t>(pair);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(p));
  f16x2_to_f32(h2, lo, hi);
}
__device__ __forceinline__ void dec_e5m2x2(uint32_t pair, float& lo, float& hi) {
  uint32_t h2;
  const uint16_t p = static_cast<uint16_t>(pair);
  asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(h2) : "h"(p));
  f16x2_to_f32(h2, lo, hi);
}
__device__ __forceinline__ float dec_int8(uint32_t byte) {
  return static_cast<float>(static_cast<int>(static_cast<int8_t>(static_cast<uint8_t>(byte))));
}
template <int FMT>
__device__ __forceinline__ void dec8x2(uint32_t pair, float& lo, float& hi) {
  if constexpr (FMT == QZ_FP8_E4M3) dec_e4m3x2(pair, lo, hi);
  else if constexpr (FMT == QZ_FP8_E5M2) dec_e5m2x2(pair, lo, hi);
  else {
    lo = dec_int8(pair & 0xffu);
    hi = dec_int8((pair >> 8) & 0xffu);
  }
}
__device__ __forceinline__ float dec_e4m3(uint32_t code) {
  float lo, hi;
  dec_e4m3x2(code & 0xffu, lo, hi);
  return lo;
}

template <int FMT>
struct Fmt8 {
  static constexpr float kMax = FMT == QZ_INT8 ? 127.0f : (FMT == QZ_FP8_E4M3 ? 448.0f : 57344.0f);
};

// ---------------------------------------------------------------------------------------
// block scales
// ---------------------------------------------------------------------------------------
constexpr float kRcp6 = 0x1.555556p-3f;  // RN(1/6)

// fl32(a / s) for a >= 0 (no sign of zero to keep), from r = RN(1/s)
__device__ __forceinline__ float div_pos(float a, float s, float r) {
  const float q = __fmul_rn(a, r);
  return __fmaf_rn(__fmaf_rn(-q, s, a), r, q);
}

// fl32(A / 6), A >= 0
__device__ __forceinline__ float div6(float A) {
  return A >= 0x1p-100f ? div_pos(A, 6.0f, kRcp6) : __fdiv_rn(A, 6.0f);
}

// MXFP4: exponent k of the E8M0 scale 2^k from t = fl32(A/6); UP: smallest k with
// 2^k >= t, NEAREST: k = round(log2 t); clamped to [-127, 127]; t == 0 -> -127.
__device__ __forceinline__ int mx_exponent(float t, int scale_round) {
  const uint32_t b = __float_as_uint(t);
  if (b == 0u) return -127;
  int E = static_cast<int>(b >> 23);          // t >= 0: no sign bit
  uint32_t F = b & 0x7fffffu;
  if (E == 0) {                                // subnormal t = F * 2^-149: normalise
    const int p = 31 - __clz(F);               // F in [2^p, 2^(p+1))
    E = p - 149 + 127;
    F = (F << (23 - p)) & 0x7fffffu;
  }
  int k = E - 127;
  if (scale_round == QZ_SCALE_NEAREST) {
    const float sig = __uint_as_float(0x3f800000u | F);  // in [1, 2)
    if (__fmaf_rn(sig, sig, -2.0f) > 0.0f) k += 1;       // log2(sig) > 1/2
  } else {
    if (F != 0u) k += 1;
  }
  return max(-127, min(127, k));
}

// 2^-k as fp32 (k in [-127, 127]; 2^-127 is subnormal)
__device__ __forceinline__ float exp2_neg(int k) {
  return k == 127 ? __uint_as_float(0x00400000u) : __uint_as_float(static_cast<uint32_t>(127 - k) << 23);
}
__device__ __forceinline__ float exp2_pos(int k) {
  return k == -127 ? __uint_as_float(0x00400000u) : __uint_as_float(static_cast<uint32_t>(127 + k) << 23);
}

// NVFP4: E4M3 code of the block scale from the ideal scale t >= 0.
__device__ __forceinline__ uint32_t nv_block_code(float t, int scale_round) {
  uint32_t c = cvt_e4m3x2(t, 0.0f) & 0xffu;  // RNE, saturating at 448
  if (scale_round == QZ_SCALE_UP && c < 0x7eu && dec_e4m3(c) < t) c += 1u;
  return c;
}

// ---------------------------------------------------------------------------------------
// error statistics
// ---------------------------------------------------------------------------------------
// Per-thread accumulators.  sum of e^2: fp32 partial per chunk, added into a compensated
// (Fast2Sum) fp32 pair.  max |e|: plain max.  max fl32(|e|/|x|): exact, with a warp-uniform
// threshold T = the warp's best ratio so far.  An element can raise the maximum only if
// |e| > T*|x| exactly; fl32(T*|x| - |e|) computed by one FMA is <= 0 in every such case
// (RN keeps signs and rounds tiny negatives to -0), so the cheap test never misses; the
// rare candidates get an exact __fdiv_rn.  No ratio exceeds 1 (0 is a grid value, so the
// nearest code is never farther from x than 0 is), so once T == 1 the test is skipped.
struct StatAcc {
  // sum of e^2 in three fixed-scale compensated fp32 buckets, chosen by the largest |e| of
  // a chunk: [2^-40, 2^40] unscaled; above 2^40 scaled by 2^-90; below 2^-40 by 2^+87.
  // Each bucket's squares stay inside the normal fp32 range (no overflow, no flush), so
  // no fp64 arithmetic is needed per chunk.
  float s = 0.0f, c = 0.0f;
  float sL = 0.0f, cL = 0.0f;
  float sS = 0.0f, cS = 0.0f;
  float max_abs = 0.0f;
  float max_abs_sq = 0.0f;  // fl32(max_abs^2)
  float rel = 0.0f;   // this lane's exact best ratio
  float T = 0.0f;     // warp-uniform: max of `rel` over the warp
};

// Fast2Sum of p into the compensated pair (s, c), larger operand first
__device__ __forceinline__ void comp_add(float& s, float& c, float p) {
  const float hi = fmaxf(s, p), lo = fminf(s, p);
  const float t = __fadd_rn(hi, lo);
  c = __fadd_rn(c, __fsub_rn(lo, __fsub_rn(t, hi)));
  s = t;
}
__device__ __forceinline__ void acc_add_sum(StatAcc& a, float p) { comp_add(a.s, a.c, p); }
constexpr float kLargeScale = 0x1p-90f;  // squares weigh 2^180
constexpr float kSmallScale = 0x1p87f;   // squares weigh 2^-174

// Is element (x, e) a candidate for a new maximum ratio?
__device__ __forceinline__ bool rel_candidate(float T, float x, float ae) {
  return (__fmaf_rn(T, fabsf(x), -ae) <= 0.0f) && (ae != 0.0f);
}

__device__ __forceinline__ float rel_exact(float x, float ae) {
  return (ae != 0.0f && x != 0.0f) ? __fdiv_rn(ae, fabsf(x)) : 0.0f;
}

__device__ __forceinline__ float warp_max(float v);

// Accumulate the error of N elements (x, x^) of one chunk.  Every lane of the warp must
// call this the same number of times (the candidate vote is warp-wide); lanes without
// data pass x = x^ = 0.
template <int N>
__device__ __forceinline__ void acc_chunk(StatAcc& acc, const float (&xs)[N], const float (&xh)[N]) {
  bool cand = false;
  const bool want_rel = acc.T < 1.0f;  // warp-uniform
  float e[N];
  bool ci[N];       // element i can raise the maximum of |e| / |x|
  float cm = 0.0f;  // largest |e| of the chunk
#pragma unroll
  for (int i = 0; i < N; ++i) {
    e[i] = __fsub_rn(xs[i], xh[i]);
    cm = fmaxf(cm, fabsf(e[i]));
    ci[i] = want_rel && rel_candidate(acc.T, xs[i], fabsf(e[i]));
    cand |= ci[i];
  }
  acc.max_abs = fmaxf(acc.max_abs, cm);
  // the bucket of the chunk (see StatAcc): scale 1 for a largest |e| in [2^-40, 2^40] (or
  // 0), where every e^2 <= 2^80 and the squares that underflow (|e| < 2^-75) are below
  // 2^-70 of the chunk's largest; otherwise the errors scaled by a power of two (exact)
  const bool normal = cm <= 0x1p40f && (cm >= 0x1p-40f || cm == 0.0f);
  const float sc = normal ? 1.0f : (cm > 0x1p40f ? kLargeScale : kSmallScale);
  float part = 0.0f;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const float es = __fmul_rn(e[i], sc);
    part = __fmaf_rn(es, es, part);
  }
  if (normal) comp_add(acc.s, acc.c, part);
  else if (cm > 0x1p40f) comp_add(acc.sL, acc.cL, part);
  else comp_add(acc.sS, acc.cS, part);
  if (want_rel && __any_sync(kFull, cand)) {
    if (cand) {  // the exact quotient for the candidates only
#pragma unroll
      for (int i = 0; i < N; ++i)
        if (ci[i]) acc.rel = fmaxf(acc.rel, rel_exact(xs[i], fabsf(e[i])));
    }
    acc.T = warp_max(acc.rel);
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}
__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Knuth's TwoSum folded into a compensated pair: (s, c) += (s2, c2), exact error of s + s2
// kept in c.  Any operand order; an infinite s makes c NaN, which `bucket_value` discards.
__device__ __forceinline__ void two_sum_into(float& s, float& c, float s2, float c2) {
  const float t = __fadd_rn(s, s2);
  const float bb = __fsub_rn(t, s);
  const float err = __fadd_rn(__fsub_rn(s, __fsub_rn(t, bb)), __fsub_rn(s2, bb));
  c = __fadd_rn(__fadd_rn(c, c2), err);
  s = t;
}
__device__ __forceinline__ void warp_two_sum(float& s, float& c) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float s2 = __shfl_xor_sync(kFull, s, o), c2 = __shfl_xor_sync(kFull, c, o);
    two_sum_into(s, c, s2, c2);
  }
}
// a bucket whose sum reached +Inf (x^ beyond the fp32 range) has a NaN compensation term
// (Inf - Inf); the sum alone is then the answer
__device__ __forceinline__ double bucket_value(float s, float c) {
  return static_cast<double>(s) + (isinf(s) ? 0.0 : static_cast<double>(c));
}

// CTA reduction of the accumulators into this CTA's partial, then the last CTA to finish
// (atomicInc wraps the counter back to 0) folds all partials in a fixed order into *out.
// Within the CTA the three buckets stay compensated fp32 pairs (fp64 arithmetic is slow on
// this part); one thread per CTA weighs them into the fp64 partial.
__device__ __forceinline__ void stats_finish(const StatAcc& a, void* ws, qz_stats* out, uint64_t n) {
  __shared__ double s_sum[kWarps];
  __shared__ float s_b[kWarps][6];
  __shared__ float s_abs[kWarps], s_rel[kWarps];
  __shared__ bool s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float b[6] = {a.s, a.c, a.sL, a.cL, a.sS, a.cS};
#pragma unroll
  for (int k = 0; k < 3; ++k) warp_two_sum(b[2 * k], b[2 * k + 1]);
  float mabs = warp_max(a.max_abs), mrel = warp_max(a.rel);
  if (lane == 0) {
#pragma unroll
    for (int k = 0; k < 6; ++k) s_b[warp][k] = b[k];
    s_abs[warp] = mabs;
    s_rel[warp] = mrel;
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < 6; ++k) b[k] = lane < kWarps ? s_b[lane][k] : 0.0f;
#pragma unroll
    for (int k = 0; k < 3; ++k) warp_two_sum(b[2 * k], b[2 * k + 1]);
    if (lane == 0)
      s_sum[0] = bucket_value(b[0], b[1]) + ldexp(bucket_value(b[2], b[3]), 180) +
                 ldexp(bucket_value(b[4], b[5]), -174);
  }
  __syncthreads();
  StatPartial* parts = ws_stat_partials(ws);
  if (threadIdx.x == 0) {
    float ma = 0.0f, mr = 0.0f;
    for (int w = 0; w < kWarps; ++w) {
      ma = fmaxf(ma, s_abs[w]);
      mr = fmaxf(mr, s_rel[w]);
    }
    parts[blockIdx.x].sum_sq = s_sum[0];
    parts[blockIdx.x].max_abs = ma;
    parts[blockIdx.x].max_rel = mr;
    __threadfence();
    const uint32_t done = atomicInc(&ws_header(ws)->stats_counter, gridDim.x - 1);
    s_last = (done == gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  double t = 0.0;
  float ma = 0.0f, mr = 0.0f;
  for (int i = threadIdx.x; i < static_cast<int>(gridDim.x); i += blockDim.x) {
    const volatile StatPartial* p = parts + i;
    t += p->sum_sq;
    ma = fmaxf(ma, p->max_abs);
    mr = fmaxf(mr, p->max_rel);
  }
  t = warp_sum(t);
  ma = warp_max(ma);
  mr = warp_max(mr);
  __syncthreads();
  if (lane == 0) {
    s_sum[warp] = t;
    s_abs[warp] = ma;
    s_rel[warp] = mr;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double tot = 0.0;
    for (int w = 0; w < kWarps; ++w) {
      tot += s_sum[w];
      ma = fmaxf(ma, s_abs[w]);
      mr = fmaxf(mr, s_rel[w]);
    }
    out->sum_sq_err = tot;
    out->mse = n ? tot / static_cast<double>(n) : 0.0;
    out->max_abs_err = ma;
    out->max_rel_err = mr;
    out->n = n;
  }
}

__device__ __forceinline__ void flag_status(void* ws, uint32_t bits) {
  if (ws) atomicOr(&ws_header(ws)->status, bits);
}

}  // namespace qz
