// qz_pipe.cuh -- shared-memory staging with 1-D bulk copies (cp.async.bulk + mbarrier) and
// packed fp32 arithmetic (f32x2) for the streaming kernels of libqz (sm_103a).
#pragma once

#include <cstdint>

#include "qz_device.cuh"

namespace qz {

// ---------------------------------------------------------------------------------------
// packed fp32 pairs: one 64-bit register holds {lo, hi}; one instruction does both lanes
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint64_t pk(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fma2_rm(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rm.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// fl32(a * b) for both lanes as an fma whose addend z2 is a zero the assembler cannot see
// (a kernel argument).  A mul.rn.f32x2 feeding a sub.rn.f32x2 -- or an fma with a literal
// zero addend, which is folded into a multiply -- can be contracted into one fma, skipping
// the rounding of the product; an fma with an opaque addend cannot.  RN(a*b + 0) = RN(a*b),
// up to the sign of an exact zero product, which no error statistic observes.
__device__ __forceinline__ uint64_t mul2_rounded(uint64_t a, uint64_t b, uint64_t z2) {
  return fma2(a, b, z2);
}

// fl32(x / s) for both lanes from r = RN(1/s) and ns = -s (the FMA-corrected quotient of
// div_by).  The remainder fma rounds toward -inf: it is exact whenever the quotient
// matters, and for x = +-0 it makes the remainder -0, so the final fma keeps the sign of
// zero of x (-0 / s = -0) without a separate copysign.
__device__ __forceinline__ uint64_t div2(uint64_t x, uint64_t r2, uint64_t ns2) {
  const uint64_t q = mul2(x, r2);
  const uint64_t rem = fma2_rm(q, ns2, x);
  return fma2(rem, r2, q);
}

// largest magnitude of three with NaN propagation
__device__ __forceinline__ float absmax3(float m, float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(m), "f"(fabsf(a)), "f"(fabsf(b)));
  return d;
}
__device__ __forceinline__ float max3(float m, float a, float b) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(m), "f"(a), "f"(b));
  return d;
}

// two bf16 in one word -> fp32 pair {lo, hi}: x + (-0) with a bf16 operand widens it
// exactly (signed zeros and subnormals kept) on the FMA pipe instead of the integer ALU
__device__ __forceinline__ uint64_t widen_bf16x2(uint32_t w) {
  float lo, hi;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "add.rn.f32.bf16 %0, l, %3;\n\tadd.rn.f32.bf16 %1, h, %3;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(w), "f"(-0.0f));
  return pk(lo, hi);
}

// Largest |x| of the 16 bf16 values in w[0..7], NaN propagating: a tree of packed
// bf16x2 maxima of magnitudes (the sign of each partial result is immaterial), then the
// two halves of the last word widened (exactly) and compared.
__device__ __forceinline__ float bf16x16_absmax(const uint32_t (&w)[8]) {
  uint32_t m0, m1, m2, m3;
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m0) : "r"(w[0]), "r"(w[1]));
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m1) : "r"(w[2]), "r"(w[3]));
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m2) : "r"(w[4]), "r"(w[5]));
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m3) : "r"(w[6]), "r"(w[7]));
  asm("max.NaN.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m0) : "r"(m1));
  asm("max.NaN.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m2) : "r"(m3));
  asm("max.NaN.xorsign.abs.bf16x2 %0, %0, %1;" : "+r"(m0) : "r"(m2));
  float lo, hi;
  upk(widen_bf16x2(m0), lo, hi);
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(fabsf(lo)), "f"(fabsf(hi)));
  return d;
}

// Eight quotients -> one 32-bit word of E2M1 codes (element 0 in bits [0,4)) and the
// decoded code values as four f16x2 words.
__device__ __forceinline__ uint32_t e2m1x8(const float (&v)[8], uint32_t (&h)[4]) {
  uint32_t w;
  asm("{\n\t.reg .b8 c0, c1, c2, c3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c0, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c1, %8, %7;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c2, %10, %9;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c3, %12, %11;\n\t"
      "mov.b32 %0, {c0, c1, c2, c3};\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, c0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, c1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, c2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %4, c3;\n\t}"
      : "=r"(w), "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return w;
}
// the same without the decoded values
__device__ __forceinline__ uint32_t e2m1x8_codes(const float (&v)[8]) {
  uint32_t w;
  asm("{\n\t.reg .b8 c0, c1, c2, c3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c3, %8, %7;\n\t"
      "mov.b32 %0, {c0, c1, c2, c3};\n\t}"
      : "=r"(w)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return w;
}
// f16x2 -> fp32 pair (exact)
__device__ __forceinline__ uint64_t f16x2_to_f32x2(uint32_t h) {
  uint64_t r;
  asm("{\n\t.reg .b16 l, h;\n\t.reg .f32 fl, fh;\n\tmov.b32 {l, h}, %1;\n\t"
      "cvt.f32.f16 fl, l;\n\tcvt.f32.f16 fh, h;\n\tmov.b64 %0, {fl, fh};\n\t}"
      : "=l"(r)
      : "r"(h));
  return r;
}

// e = fl32(x - q * 2^k) for the two code values q of the f16x2 word h, given -2^k as the
// f16 bits ns16 (k in [-24, 15]): one fused multiply-add per element whose f16 operands
// widen exactly, so each result is rounded once
__device__ __forceinline__ uint64_t fma_f16_pair(uint32_t h, uint16_t ns16, uint64_t x) {
  float x0, x1, e0, e1;
  upk(x, x0, x1);
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "fma.rn.f32.f16 %0, l, %3, %4;\n\tfma.rn.f32.f16 %1, h, %3, %5;\n\t}"
      : "=f"(e0), "=f"(e1)
      : "r"(h), "h"(ns16), "f"(x0), "f"(x1));
  return pk(e0, e1);
}
// f16 bits of -2^k, k in [-24, 15] (k < -14: an f16 subnormal)
__device__ __forceinline__ uint16_t f16_neg_pow2(int k) {
  return static_cast<uint16_t>(0x8000u | (k >= -14 ? static_cast<uint32_t>(k + 15) << 10 : 1u << (k + 24)));
}

__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

template <int NP>
struct Pairs {
  uint64_t v[NP];
};

// Sum of the squares of 2*NP values held as fp32 pairs (two accumulator chains)
template <int NP>
__device__ __forceinline__ float pairs_sumsq(const uint64_t (&e)[NP]) {
  uint64_t pa = mul2(e[0], e[0]);
  uint64_t pb = pk(0.0f, 0.0f);
  if constexpr (NP > 1) pb = mul2(e[1], e[1]);
#pragma unroll
  for (int p = 2; p < NP; p += 2) {
    pa = fma2(e[p], e[p], pa);
    if (p + 1 < NP) pb = fma2(e[p + 1], e[p + 1], pb);
  }
  float p0, p1, p2, p3;
  upk(pa, p0, p1);
  upk(pb, p2, p3);
  return __fadd_rn(__fadd_rn(p0, p1), __fadd_rn(p2, p3));
}

// Largest |value| of 2*NP values held as fp32 pairs: a tree of 3-input maxima.
template <int NP>
__device__ __forceinline__ float pairs_max_abs(const uint64_t (&p2)[NP]) {
  float v[2 * NP];
#pragma unroll
  for (int p = 0; p < NP; ++p) upk(p2[p], v[2 * p], v[2 * p + 1]);
  constexpr int T = (2 * NP + 2) / 3;
  float t[T];
#pragma unroll
  for (int i = 0; i < T; ++i) {
    const float a1 = 3 * i + 1 < 2 * NP ? fabsf(v[3 * i + 1]) : 0.0f;
    const float a2 = 3 * i + 2 < 2 * NP ? fabsf(v[3 * i + 2]) : 0.0f;
    t[i] = max3(fabsf(v[3 * i]), a1, a2);
  }
  float m = t[0];
#pragma unroll
  for (int i = 1; i + 1 < T; i += 2) m = max3(m, t[i], t[i + 1]);
  if constexpr (T % 2 == 0) m = fmaxf(m, t[T - 1]);
  return m;
}

// Accumulate the errors e (fp32 pairs) of one chunk whose inputs are x: largest |e|, sum
// of e^2, and -- REL, while the warp's exact max |e|/|x| search is open -- the candidates
// of rel_candidate.  Every lane of the warp must make the same calls (the REL part votes).
//
// Largest |e|: the chunk's fp32 sum of squares `part` is at least fl(e^2) of each of its
// elements (RN is monotone and never rounds a sum of non-negative terms below a term), so
// part < fl(max_abs^2) proves every |e| < max_abs and the chunk is skipped.
// Sum of squares: `part` itself when it lies in [2^-80, 2^80] (no square overflowed, and
// the squares below the normal range are under 2^-42 of the chunk's largest); otherwise
// the chunk's errors go, scaled by a power of two (exact), to the bucket of their largest
// magnitude (see StatAcc).
template <int NP, bool REL>
__device__ __forceinline__ void acc_pairs(StatAcc& acc, const uint64_t (&xp)[NP], const Pairs<NP>& e,
                                          float& tpart) {
  const float part = pairs_sumsq<NP>(e.v);
  float cm = -1.0f;  // largest |e| of the chunk, -1 while not needed
  if (!(part < acc.max_abs_sq)) {
    cm = pairs_max_abs<NP>(e.v);
    acc.max_abs = fmaxf(acc.max_abs, cm);
    acc.max_abs_sq = __fmul_rn(acc.max_abs, acc.max_abs);
  }
  if (part >= 0x1p-80f && part <= 0x1p80f) {
    tpart = __fadd_rn(tpart, part);
  } else {
    if (cm < 0.0f) cm = pairs_max_abs<NP>(e.v);
    if (cm <= 0x1p40f && (cm >= 0x1p-40f || cm == 0.0f)) {
      tpart = __fadd_rn(tpart, part);
    } else {
      const float sc = cm > 0x1p40f ? kLargeScale : kSmallScale;
      const uint64_t sc2 = pk(sc, sc);
      uint64_t es[NP];
#pragma unroll
      for (int p = 0; p < NP; ++p) es[p] = mul2(e.v[p], sc2);
      const float ps = pairs_sumsq<NP>(es);
      if (cm > 0x1p40f) comp_add(acc.sL, acc.cL, ps);
      else comp_add(acc.sS, acc.cS, ps);
    }
  }
  if constexpr (REL) {
    // An element can raise the maximum only if |e| > T |x|, and then (only then)
    // fl32(T |x| - |e|) is negative or -0; such elements get the exact quotient
    float d[2 * NP];
    uint32_t sg = 0u;
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      float x0, x1, e0, e1;
      upk(xp[p], x0, x1);
      upk(e.v[p], e0, e1);
      d[2 * p] = __fmaf_rn(acc.T, fabsf(x0), -fabsf(e0));
      d[2 * p + 1] = __fmaf_rn(acc.T, fabsf(x1), -fabsf(e1));
      sg |= __float_as_uint(d[2 * p]) | __float_as_uint(d[2 * p + 1]);
    }
    const bool cand = (sg & 0x80000000u) != 0u;
    if (__any_sync(kFull, cand)) {
      if (cand) {
#pragma unroll
        for (int p = 0; p < NP; ++p) {
          float x0, x1, e0, e1;
          upk(xp[p], x0, x1);
          upk(e.v[p], e0, e1);
          if (__float_as_uint(d[2 * p]) & 0x80000000u) acc.rel = fmaxf(acc.rel, rel_exact(x0, fabsf(e0)));
          if (__float_as_uint(d[2 * p + 1]) & 0x80000000u) acc.rel = fmaxf(acc.rel, rel_exact(x1, fabsf(e1)));
        }
      }
      acc.T = warp_max(acc.rel);
    }
  }
}

// CTA maximum of per-thread maxima (m: bf16 -> two 16-bit magnitudes, fp32 -> one), written
// as this CTA's partial; the last CTA to finish folds the partials into *out and flags a
// non-finite maximum.
template <int DT>
__device__ __forceinline__ void amax_finish(uint32_t m, float* out, void* ws) {
  uint32_t bits;  // fp32 bit pattern of this thread's maximum
  if constexpr (DT == QZ_BF16) bits = max(m & 0xffffu, m >> 16) << 16;
  else bits = m;
#pragma unroll
  for (int o = 16; o; o >>= 1) bits = max(bits, __shfl_xor_sync(kFull, bits, o));
  __shared__ uint32_t s_w[kWarps];
  __shared__ bool s_last;
  if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = bits;
  __syncthreads();
  float* parts = ws_amax_partials(ws);
  if (threadIdx.x == 0) {
    uint32_t b = 0;
    for (int w = 0; w < kWarps; ++w) b = max(b, s_w[w]);
    reinterpret_cast<uint32_t*>(parts)[blockIdx.x] = b;
    __threadfence();
    const uint32_t done = atomicInc(&ws_header(ws)->amax_counter, gridDim.x - 1);
    s_last = (done == gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  uint32_t b = 0;
  for (int i = threadIdx.x; i < static_cast<int>(gridDim.x); i += kThreads)
    b = max(b, reinterpret_cast<volatile uint32_t*>(parts)[i]);
#pragma unroll
  for (int o = 16; o; o >>= 1) b = max(b, __shfl_xor_sync(kFull, b, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) s_w[threadIdx.x >> 5] = b;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t t = 0;
    for (int w = 0; w < kWarps; ++w) t = max(t, s_w[w]);
    if (t >= 0x7f800000u) atomicOr(&ws_header(ws)->status, QZ_FLAG_NONFINITE_INPUT);
    *out = __uint_as_float(t);
  }
}

// ---------------------------------------------------------------------------------------
// mbarrier + bulk copy global -> shared
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Wait for phase `parity` of the barrier, giving up after `limit_ns` (returns false).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() - t0 > limit_ns) return false;
  return true;
}
// bytes (multiple of 16, both addresses 16-byte aligned) from global to shared; completion
// is signalled on the barrier as transaction bytes
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void lds32B(uint32_t (&w)[8], uint32_t addr) {
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
               : "r"(addr));
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(w[4]), "=r"(w[5]), "=r"(w[6]), "=r"(w[7])
               : "r"(addr + 16));
}

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far beyond any copy's latency

// Geometry of the staged streaming kernels: a tile is kPipeCPT 32-byte chunks per thread
// (32 KiB for 256 threads), kPipeStages tiles in flight per CTA (64 KiB, 3 CTAs per SM).
// Measured against 16 KiB tiles in 4 stages on a 32768 x 8192 bf16 tensor: fewer waits,
// block synchronisations and refills per chunk made every staged kernel as fast or faster
// (amax 84.6 -> 82.6 us, NVFP4 quantize with statistics 162 -> 156 us, INT4 166 -> 160 us).
constexpr int kPipeCPT = 4;
constexpr int kPipeTileChunks = kThreads * kPipeCPT;
constexpr int kPipeTileBytes = kPipeTileChunks * 32;
constexpr int kPipeStages = 2;
constexpr size_t kPipeSmem = static_cast<size_t>(kPipeStages) * kPipeTileBytes;

// Streams the tiles of one CTA through S shared-memory stages.  Tile k of this CTA is
// tile (blockIdx.x + k * gridDim.x) of the tensor (counted from the end when `reverse`),
// TILE bytes (the last tile of the tensor shorter).
// Thread 0 issues the copies; every thread waits on the tile's barrier; the CTA
// synchronises once per tile before thread 0 refills the stage it has left.
template <int S, int TILE>
struct BulkPipe {
  uint32_t base;      // shared address of stage 0
  uint32_t bars;      // shared address of barrier 0
  const char* src;
  int64_t nbytes;
  int64_t ntiles;
  bool reverse;  // hand out the tiles from the end of the tensor

  __device__ __forceinline__ int64_t slot_of(int64_t k) const {
    return static_cast<int64_t>(blockIdx.x) + k * gridDim.x;
  }
  __device__ __forceinline__ bool has(int64_t k) const { return slot_of(k) < ntiles; }
  __device__ __forceinline__ int64_t tile_of(int64_t k) const {
    const int64_t t = slot_of(k);
    return reverse ? ntiles - 1 - t : t;
  }
  __device__ __forceinline__ uint32_t bytes_of(int64_t tile) const {
    const int64_t rest = nbytes - tile * TILE;
    return static_cast<uint32_t>(rest < TILE ? rest : TILE);
  }
  __device__ __forceinline__ void issue(int64_t k) const {  // thread 0 only
    if (!has(k)) return;
    const int64_t tile = tile_of(k);
    const uint32_t s = static_cast<uint32_t>(k % S);
    const uint32_t bar = bars + 8u * s, bytes = bytes_of(tile);
    mbar_expect_tx(bar, bytes);
    bulk_g2s(base + s * TILE, src + tile * TILE, bytes, bar);
  }
  // thread 0, before the first tile (after the barriers are initialised and fenced)
  __device__ __forceinline__ void prologue() const {
    for (int k = 0; k < S; ++k) issue(k);
  }
  __device__ __forceinline__ bool wait(int64_t k) const {
    const uint32_t s = static_cast<uint32_t>(k % S);
    return mbar_wait(bars + 8u * s, static_cast<uint32_t>((k / S) & 1), kWaitLimitNs);
  }
  __device__ __forceinline__ uint32_t stage(int64_t k) const {
    return base + static_cast<uint32_t>(k % S) * TILE;
  }
  // After an aborted wait: let the copies already issued for tiles k .. k+S-1 land
  // (bounded) before the CTA's shared memory is released.
  __device__ __forceinline__ void drain(int64_t k) const {
    for (int64_t j = k; j < k + S; ++j)
      if (has(j)) mbar_wait(bars + 8u * static_cast<uint32_t>(j % S),
                            static_cast<uint32_t>((j / S) & 1), kWaitLimitNs);
  }
};

}  // namespace qz
