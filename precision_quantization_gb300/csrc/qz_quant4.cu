// qz_quant4.cu -- quantize to MXFP4 / NVFP4 (blog post "浅谈低精度浮点数", section
// "FP4 / MXFP4 / NVFP4"), optionally with the error statistics fused into the same pass.
//
// Data path: each lane owns one 32-byte chunk of a row of x (16 bf16 or 8 fp32 values),
// read with one 256-bit load, so a warp streams 1 KiB of contiguous input per load.  A
// scale block is 1 (NVFP4 bf16), 2 (NVFP4 fp32, MXFP4 bf16) or 4 (MXFP4 fp32) neighbouring
// lanes; its amax is a max-shuffle among them.  Codes are cast two at a time with
// cvt.rn.satfinite.e2m1x2, packed low-nibble-first, and stored as one 8- or 4-byte word
// per lane (coalesced); the first lane of every block stores its scale byte.
#include "qz_device.cuh"
#include "qz_internal.h"
#include "qz_pipe.cuh"

namespace qz {
namespace {

constexpr int kUnroll = 2;

struct Q4Args {
  const void* x;
  Geom g;
  uint8_t* codes;
  uint8_t* scales;
  const float* amax;  // NVFP4 BLOCK: alpha on the device; else unused
  float* tscale_out;  // may be null
  qz_stats* stats;
  void* ws;
  int scale_round;
  bool reverse;  // pipelined path: walk the tiles from the end of the tensor
  float zero;    // 0.0f, opaque to the assembler (see mul2_rounded)
  float* amax_out = nullptr;  // staged path: this tensor's max |x| (for the next call's scale)
};

// fl32(a / b) for scalar scale arithmetic: the FMA-corrected quotient where it is exact
// (normal operands, normal quotient), IEEE division otherwise.
__device__ __forceinline__ float div_scalar(float a, float b, float rb) {
  if (a >= 0x1p-100f && fast_div_ok(b)) {
    const float q = div_by(a, b, rb);
    if (q >= 0x1p-120f) return q;
  }
  return __fdiv_rn(a, b);
}

template <int FMT, int DT, bool UNIT, bool STATS, bool VEC>
__global__ void __launch_bounds__(kThreads) quant4_kernel(Q4Args a) {
  constexpr int EPC = Elem<DT>::kPer32B;     // elements per lane-chunk
  constexpr int BS = FMT == QZ_MXFP4 ? 32 : 16;
  constexpr int L = BS / EPC;                // lanes per scale block
  constexpr int CB = EPC / 2;                // code bytes per chunk
  const Geom& g = a.g;
  const int lane = threadIdx.x & 31;

  // per-tensor scale (NVFP4): s_g = fl32(alpha / (6 * 448)), 1 when 0
  float sg = 1.0f, rg = 1.0f;
  if constexpr (FMT == QZ_NVFP4 && !UNIT) {
    const float alpha = *a.amax;
    if (!(alpha >= 0.0f) || !is_finite_f(alpha)) {
      if (blockIdx.x == 0 && threadIdx.x == 0) flag_status(a.ws, QZ_FLAG_BAD_AMAX);
    }
    sg = __fdiv_rn(alpha, 2688.0f);
    if (sg == 0.0f) sg = 1.0f;
    rg = __frcp_rn(sg);
  }
  if (a.tscale_out && blockIdx.x == 0 && threadIdx.x == 0) *a.tscale_out = sg;

  StatAcc acc;
  const int64_t warp_id = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarps * 32 * kUnroll;
  for (int64_t base = warp_id * 32 * kUnroll; base < g.n_chunks; base += stride) {
    uint32_t w[kUnroll][8];
    int64_t row[kUnroll], col[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const int64_t u = base + k * 32 + lane;
      if (g.dense) {
        row[k] = 0;
        col[k] = u * EPC;  // flat element index
      } else {
        row[k] = u / g.cpr;
        col[k] = (u - row[k] * g.cpr) * EPC;
      }
      if (u < g.n_chunks) {
        const int64_t e0 = row[k] * g.ld + col[k];
        if constexpr (VEC) {
          ld32B(w[k], static_cast<const char*>(a.x) + e0 * Elem<DT>::kBytes);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            if constexpr (DT == QZ_BF16) {
              const uint32_t lo = __float_as_uint(load_elem<DT>(a.x, e0 + 2 * i)) >> 16;
              const uint32_t hi = __float_as_uint(load_elem<DT>(a.x, e0 + 2 * i + 1));
              w[k][i] = (hi & 0xffff0000u) | lo;
            } else {
              w[k][i] = __float_as_uint(load_elem<DT>(a.x, e0 + i));
            }
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) w[k][i] = 0u;
      }
    }
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const int64_t u = base + k * 32 + lane;
      const bool valid = u < g.n_chunks;
      float xs[EPC];
#pragma unroll
      for (int i = 0; i < EPC; ++i) xs[i] = chunk_elem<DT>(w[k], i);
      float A = 0.0f;
#pragma unroll
      for (int i = 0; i < EPC; ++i) A = absmax_nan(A, xs[i]);
      if constexpr (L >= 2) A = absmax_nan(A, __shfl_xor_sync(kFull, A, 1));
      if constexpr (L >= 4) A = absmax_nan(A, __shfl_xor_sync(kFull, A, 2));
      if (valid && !is_finite_f(A)) flag_status(a.ws, QZ_FLAG_NONFINITE_INPUT);

      // block scale and the element quotients v = fl32(x / s)
      uint32_t scode;
      float s;
      float v[EPC];
      if constexpr (FMT == QZ_MXFP4) {
        const int kexp = UNIT ? 0 : mx_exponent(div6(A), a.scale_round);
        scode = static_cast<uint32_t>(kexp + 127);
        s = exp2_pos(kexp);
        const float inv = exp2_neg(kexp);  // x / 2^k == x * 2^-k exactly
#pragma unroll
        for (int i = 0; i < EPC; ++i) v[i] = __fmul_rn(xs[i], inv);
      } else {
        if constexpr (UNIT) {
          scode = 0x38u;  // E4M3 1.0
        } else {
          const float t = div_scalar(div6(A), sg, rg);  // (block_amax / 6) / s_global
          scode = nv_block_code(t, a.scale_round);
        }
        s = __fmul_rn(sg, dec_e4m3(scode));
        if (s == 0.0f) {
#pragma unroll
          for (int i = 0; i < EPC; ++i) v[i] = copysignf(0.0f, xs[i]);
        } else {
          const float r = __frcp_rn(s);
          if (fast_div_ok(s) && __fmul_rn(A, r) <= 0x1p126f) {
#pragma unroll
            for (int i = 0; i < EPC; ++i) v[i] = div_by(xs[i], s, r);
          } else {
#pragma unroll
            for (int i = 0; i < EPC; ++i) v[i] = __fdiv_rn(xs[i], s);
          }
        }
      }

      // cast, pack (element 2i -> low nibble of byte i), store
      uint32_t cw[CB / 4];
#pragma unroll
      for (int j = 0; j < CB / 4; ++j) {
        cw[j] = cvt_e2m1x2(v[8 * j + 0], v[8 * j + 1]) | (cvt_e2m1x2(v[8 * j + 2], v[8 * j + 3]) << 8) |
                (cvt_e2m1x2(v[8 * j + 4], v[8 * j + 5]) << 16) |
                (cvt_e2m1x2(v[8 * j + 6], v[8 * j + 7]) << 24);
      }
      if (valid) {
        const int64_t cofs = g.dense ? col[k] / 2 : row[k] * (g.cols / 2) + col[k] / 2;
        uint8_t* cp = a.codes + cofs;
        if constexpr (VEC) {
          if constexpr (CB == 8) {
            asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(cp), "r"(cw[0]), "r"(cw[1]) : "memory");
          } else {
            asm volatile("st.global.u32 [%0], %1;" ::"l"(cp), "r"(cw[0]) : "memory");
          }
        } else {
#pragma unroll
          for (int j = 0; j < CB; ++j) cp[j] = static_cast<uint8_t>(cw[j / 4] >> (8 * (j % 4)));
        }
        if (lane % L == 0) {
          const int64_t sofs = g.dense ? col[k] / BS : row[k] * (g.cols / BS) + col[k] / BS;
          a.scales[sofs] = static_cast<uint8_t>(scode);
        }
      }

      if constexpr (STATS) {
        // x^ = fl32(decode(q) * s).  Invalid lanes hold x = 0 and code 0 -> e = 0.
        float xh[EPC];
#pragma unroll
        for (int j = 0; j < EPC / 2; ++j) {
          float q0, q1;
          dec_e2m1x2((cw[j / 4] >> (8 * (j % 4))) & 0xffu, q0, q1);
          xh[2 * j] = __fmul_rn(q0, s);
          xh[2 * j + 1] = __fmul_rn(q1, s);
        }
        acc_chunk(acc, xs, xh);
      }
    }
  }
  if constexpr (STATS) stats_finish(acc, a.ws, a.stats, static_cast<uint64_t>(g.rows * g.cols));
}

// ---------------------------------------------------------------------------------------
// Dense tensors (rows back to back, 16-byte aligned): the input is streamed through shared
// memory by 1-D bulk copies, 32 KiB per tile, 2 tiles in flight per CTA, so the memory
// latency is covered by the pipeline instead of by registers.  The element arithmetic is
// done on fp32 pairs (f32x2), which halves the FMA-pipe instructions, and the integer /
// compare work is kept to 3-input max, the casts and the per-block scale.
// ---------------------------------------------------------------------------------------
constexpr int kCPT = kPipeCPT;
constexpr int kTileChunks = kPipeTileChunks;
constexpr int kTileBytes = kPipeTileBytes;
// tiles in flight and resident CTAs per SM of the staged quantizer (the same for both
// formats since the 32 KiB tiles; with 16 KiB tiles MXFP4 had run 4 CTAs x 3 stages)
template <int FMT>
struct PipeShape {
  static constexpr int kStages = kPipeStages;
  static constexpr int kCtas = 3;
  static constexpr int kUnroll = FMT == QZ_MXFP4 ? 2 : 1;  // chunks of the tile loop unrolled
};

// Largest magnitude of 2*NP values held as fp32 pairs, as a tree of 3-input maxima (short
// dependency chains); NAN_PROP selects the NaN-propagating maximum.
template <int NP, bool NAN_PROP>
__device__ __forceinline__ float pairs_absmax(const uint64_t (&xp)[NP]) {
  float v[2 * NP];
#pragma unroll
  for (int p = 0; p < NP; ++p) upk(xp[p], v[2 * p], v[2 * p + 1]);
  float t[(2 * NP + 2) / 3];
#pragma unroll
  for (int i = 0; i < (2 * NP + 2) / 3; ++i) {
    const float a0 = v[3 * i];
    const float a1 = 3 * i + 1 < 2 * NP ? v[3 * i + 1] : 0.0f;
    const float a2 = 3 * i + 2 < 2 * NP ? v[3 * i + 2] : 0.0f;
    t[i] = NAN_PROP ? absmax3(fabsf(a0), a1, a2) : max3(fabsf(a0), fabsf(a1), fabsf(a2));
  }
  constexpr int T = (2 * NP + 2) / 3;
  float u[(T + 2) / 3];
#pragma unroll
  for (int i = 0; i < (T + 2) / 3; ++i) {
    const float a0 = t[3 * i];
    const float a1 = 3 * i + 1 < T ? t[3 * i + 1] : 0.0f;
    const float a2 = 3 * i + 2 < T ? t[3 * i + 2] : 0.0f;
    u[i] = NAN_PROP ? absmax3(a0, a1, a2) : max3(a0, a1, a2);
  }
  constexpr int U = (T + 2) / 3;
  float m = u[0];
#pragma unroll
  for (int i = 1; i < U; ++i) m = NAN_PROP ? absmax_nan(m, u[i]) : fmaxf(m, u[i]);
  return m;
}

// Per-CTA constants of the pipelined quantizer.
struct Q4Ctx {
  float sg, rg;   // NVFP4 s_global and RN(1/s_global)
  bool sg_fast;   // s_global inside the FMA-quotient range
  const float2* tab;
  float zero;     // opaque 0.0f (see mul2_rounded)
  float c6;       // NVFP4: RN(1 / RN(6 * s_global))
  bool c6_ok;     // s_global in [2^-100, 2^100]: 6 * s_global and c6 normal
};

// One 32-byte chunk: block amax, scale, quotients, cast, stores, and (STATS) the error of
// the chunk.  REL: the exact max |e|/|x| search is still open for this warp (T < 1).
// am: running max of the block amaxes' bits (the tensor amax, for amax_out).
template <int FMT, int DT, bool UNIT, bool STATS, int SR, bool REL, bool AMAX>
__device__ __forceinline__ void q4_chunk(const Q4Args& a, const Q4Ctx& cx, const uint32_t (&w)[8],
                                         int64_t u, bool valid, int lane, StatAcc& acc,
                                         float& tpart, uint32_t& am) {
  constexpr int EPC = Elem<DT>::kPer32B;
  constexpr int BS = FMT == QZ_MXFP4 ? 32 : 16;
  constexpr int L = BS / EPC;
  constexpr int NP = EPC / 2;
  // widen to fp32 pairs; block amax (NaN propagates)
  uint64_t xp[NP];
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    if constexpr (DT == QZ_BF16) xp[p] = widen_bf16x2(w[p]);
    else xp[p] = pk(__uint_as_float(w[2 * p]), __uint_as_float(w[2 * p + 1]));
  }
  float A;
  if constexpr (DT == QZ_BF16) A = bf16x16_absmax(w);  // packed bf16x2 maxima: fewer ALU slots
  else A = pairs_absmax<NP, true>(xp);
  if constexpr (L >= 2) A = absmax_nan(A, __shfl_xor_sync(kFull, A, 1));
  if constexpr (L >= 4) A = absmax_nan(A, __shfl_xor_sync(kFull, A, 2));
  // A NaN / Inf block amax is flagged here for UNIT and MXFP4 NEAREST; the MXFP4 UP and
  // NVFP4 scale paths send it to their out-of-line branch and flag it there
  constexpr bool kFlagHere = UNIT || (FMT == QZ_MXFP4 && SR != QZ_SCALE_UP);
  if (kFlagHere && valid && !is_finite_f(A)) flag_status(a.ws, QZ_FLAG_NONFINITE_INPUT);
  if constexpr (AMAX) am = max(am, __float_as_uint(A));  // A >= 0; lanes without data hold 0

  // block scale s and the quotients v = fl32(x / s), as fp32 pairs
  uint32_t scode;
  float s;
  uint64_t vp[NP];
  bool mul_exact = false;  // MXFP4: decode(q) * 2^k exact, so e = fma(-q, s, x)
  int kexp = 0;
  float inv = 1.0f;        // MXFP4: 2^-k
  float nv_ns = 0.0f;      // NVFP4: -s
  if constexpr (FMT == QZ_MXFP4) {
    if constexpr (UNIT) {
      kexp = 0;
    } else if constexpr (SR == QZ_SCALE_UP) {
      // With A = m * 2^e (m in [1,2)), A/6 = (m/1.5) * 2^(e-2): fl32(A/6) <= 2^(e-2) exactly
      // when m <= 1.5, and lies in (2^(e-2), 2^(e-1)) otherwise, so the smallest k with
      // 2^k >= fl32(A/6) is e - 2 + [m > 1.5] -- read off A's fields, valid while A/6 is
      // normal.  The [m > 1.5] is the carry of the fraction field plus (2^22 - 1) into the
      // exponent field, so the code k + 127 is ((bits + 2^22 - 1) >> 23) - 2, in [2, 253]
      // for A in [2^-125, 2^128); there s = 2^k and 1/s are plain exponent fields.  Zero,
      // tiny and non-finite A take the general route.
      const uint32_t b = __float_as_uint(A);
      if (b - 0x02000000u < 0x7d800000u) {
        scode = ((b + 0x3fffffu) >> 23) - 2u;
        kexp = static_cast<int>(scode) - 127;
        s = __uint_as_float(scode << 23);
        inv = __uint_as_float((254u - scode) << 23);
      } else {
        if (valid && b >= 0x7f800000u) flag_status(a.ws, QZ_FLAG_NONFINITE_INPUT);
        kexp = mx_exponent(div6(A), SR);
        scode = static_cast<uint32_t>(kexp + 127);
        s = exp2_pos(kexp);
        inv = exp2_neg(kexp);
      }
    } else {
      kexp = mx_exponent(div6(A), SR);
    }
    if constexpr (UNIT || SR != QZ_SCALE_UP) {
      scode = static_cast<uint32_t>(kexp + 127);
      s = exp2_pos(kexp);
      inv = exp2_neg(kexp);
    }
    const uint64_t inv2 = pk(inv, inv);
#pragma unroll
    for (int p = 0; p < NP; ++p) vp[p] = mul2(xp[p], inv2);
    mul_exact = kexp >= -125 && kexp <= 125;
  } else {
    if constexpr (UNIT) {
      scode = 0x38u;
    } else {
      // The ideal scale t = fl32(fl32(A/6) / s_global) decides the block code only through
      // the E4M3 value (UP) or midpoint (NEAREST) it falls beside.  t' = RN(A * c6) is five
      // roundings of 2^-24 from t (normal operands: c6_ok, A and t' >= 2^-100, or A = 0),
      // so t lies within 6 ulp of t'.  E4M3 values have at most 4 significant bits and
      // their midpoints 5, i.e. fraction fields that are multiples of 2^20 (2^19): when
      // t' is not within 8 ulp of such a multiple, t and t' get the same code; otherwise
      // (rare) t is computed as written.
      float t = __fmul_rn(A, cx.c6);
      constexpr uint32_t kMask = SR == QZ_SCALE_NEAREST ? 0x7ffffu : 0xfffffu;
      const uint32_t tb = __float_as_uint(t);
      const bool near = ((tb + 8u) & kMask) < 16u;
      if (!cx.c6_ok || near || (A != 0.0f && !(A >= 0x1p-100f && t >= 0x1p-100f))) {
        // NaN fails the range test and +Inf makes t' = Inf, whose fraction field is "near"
        if (valid && !is_finite_f(A)) flag_status(a.ws, QZ_FLAG_NONFINITE_INPUT);
        const float a6 = div6(A);  // (block_amax / 6) / s_global
        if (a6 >= 0x1p-100f && cx.sg_fast) {
          t = div_pos(a6, cx.sg, cx.rg);
          if (t < 0x1p-120f) t = __fdiv_rn(a6, cx.sg);
        } else {
          t = __fdiv_rn(a6, cx.sg);
        }
      }
      scode = nv_block_code(t, SR);
    }
    const float2 sr = cx.tab[scode];  // (-s, RN(1/s))
    s = -sr.x;
    nv_ns = sr.x;
    if (UNIT) {  // s = 1: fl32(x / 1) = x
#pragma unroll
      for (int p = 0; p < NP; ++p) vp[p] = xp[p];
    } else if (__fmul_rn(A, sr.y) <= 0x1p126f) {  // NaN 1/s (no exact FMA quotient) fails
      const uint64_t r2 = pk(sr.y, sr.y), ns2 = pk(sr.x, sr.x);
#pragma unroll
      for (int p = 0; p < NP; ++p) vp[p] = div2(xp[p], r2, ns2);
    } else if (s == 0.0f) {
      const uint64_t z2 = pk(0.0f, 0.0f);
#pragma unroll
      for (int p = 0; p < NP; ++p) vp[p] = mul2(xp[p], z2);  // signed zeros
    } else {
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        float lo, hi;
        upk(xp[p], lo, hi);
        vp[p] = pk(__fdiv_rn(lo, s), __fdiv_rn(hi, s));
      }
    }
  }

  // cast and pack 8 at a time; store the codes and the block scale
  uint32_t cw[EPC / 8];
  uint32_t h[EPC / 8][4];
#pragma unroll
  for (int g8 = 0; g8 < EPC / 8; ++g8) {
    float v[8];
#pragma unroll
    for (int p = 0; p < 4; ++p) upk(vp[4 * g8 + p], v[2 * p], v[2 * p + 1]);
    if constexpr (STATS) cw[g8] = e2m1x8(v, h[g8]);
    else cw[g8] = e2m1x8_codes(v);
  }
  if (valid) {
    uint8_t* cp = a.codes + u * (EPC / 2);
    if constexpr (EPC == 16) {
      asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(cp), "r"(cw[0]), "r"(cw[1]) : "memory");
    } else {
      asm volatile("st.global.u32 [%0], %1;" ::"l"(cp), "r"(cw[0]) : "memory");
    }
    if (lane % L == 0) a.scales[u / L] = static_cast<uint8_t>(scode);
  }
  if constexpr (!STATS) return;

  // x^ = fl32(decode(q) * s), e = fl32(x - x^); lanes without data hold x = 0, q = 0
  Pairs<NP> e;
  if (FMT == QZ_MXFP4 && __all_sync(kFull, kexp >= -24 && kexp <= 15)) {
    const uint16_t ns16 = f16_neg_pow2(kexp);  // -s exactly, as an f16 operand
#pragma unroll
    for (int p = 0; p < NP; ++p) e.v[p] = fma_f16_pair(h[p / 4][p % 4], ns16, xp[p]);
  } else if (FMT == QZ_MXFP4 && __all_sync(kFull, mul_exact)) {
    const uint64_t ns2 = pk(-s, -s);
#pragma unroll
    for (int p = 0; p < NP; ++p) e.v[p] = fma2(f16x2_to_f32x2(h[p / 4][p % 4]), ns2, xp[p]);
  } else {
    // x + fl32(q * -s) = x - fl32(q * s)
    const float ns = FMT == QZ_NVFP4 ? nv_ns : -s;
    const uint64_t ns2 = pk(ns, ns), z2 = pk(cx.zero, cx.zero);
#pragma unroll
    for (int p = 0; p < NP; ++p) e.v[p] = add2(xp[p], mul2_rounded(f16x2_to_f32x2(h[p / 4][p % 4]), ns2, z2));
  }
  acc_pairs<NP, REL>(acc, xp, e, tpart);
}

template <int FMT, int DT, bool UNIT, bool STATS, int SR, bool AMAX>
__global__ void __launch_bounds__(kThreads, PipeShape<FMT>::kCtas) quant4_pipe_kernel(Q4Args a) {
  constexpr int S = PipeShape<FMT>::kStages;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[S];
  __shared__ float2 tab[128];  // NVFP4: (-s, RN(1/s)) for every E4M3 block code; NaN 1/s: divide
  __shared__ int s_abort;
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t n_chunks = a.g.n_chunks;

  Q4Ctx cx{1.0f, 1.0f, true, tab, a.zero, 0.0f, false};
  if constexpr (FMT == QZ_NVFP4) {
    if constexpr (!UNIT) {
      const float alpha = *a.amax;
      if ((!(alpha >= 0.0f) || !is_finite_f(alpha)) && blockIdx.x == 0 && tid == 0)
        flag_status(a.ws, QZ_FLAG_BAD_AMAX);
      cx.sg = __fdiv_rn(alpha, 2688.0f);  // global_amax / (6 * 448)
      if (cx.sg == 0.0f) cx.sg = 1.0f;
      cx.rg = __frcp_rn(cx.sg);
    }
    cx.sg_fast = fast_div_ok(cx.sg);
    cx.c6_ok = cx.sg >= 0x1p-100f && cx.sg <= 0x1p100f;
    cx.c6 = __frcp_rn(__fmul_rn(6.0f, cx.sg));
    for (int c = tid; c < 128; c += kThreads) {
      const float s = __fmul_rn(cx.sg, dec_e4m3(static_cast<uint32_t>(c)));
      tab[c] = make_float2(-s, (s > 0.0f && fast_div_ok(s)) ? __frcp_rn(s) : __uint_as_float(0x7fc00000u));
    }
  }
  if (a.tscale_out && blockIdx.x == 0 && tid == 0) *a.tscale_out = cx.sg;
  if (tid == 0) {
    for (int i = 0; i < S; ++i) mbar_init(smem_addr(&bars[i]), 1);
    mbar_init_fence();
    s_abort = 0;
  }
  __syncthreads();
  const BulkPipe<S, kTileBytes> P{smem_addr(smem), smem_addr(&bars[0]),
                                        static_cast<const char*>(a.x), n_chunks * 32,
                                        (n_chunks + kTileChunks - 1) / kTileChunks, a.reverse};
  if (tid == 0) P.prologue();

  StatAcc acc;
  uint32_t am = 0u;
  for (int64_t k = 0; P.has(k); ++k) {
    const int64_t tile = P.tile_of(k);
    if (!P.wait(k)) s_abort = 1;
    float tpart = 0.0f;  // in-range chunk sums of squares of this tile
    const uint32_t stage = P.stage(k);
    // MXFP4: two chunks in flight per thread (measured 127.6 -> 125.6 us with statistics on
    // a 32768 x 8192 bf16 tensor); NVFP4: one, which keeps its larger chunk code from
    // running out of registers (148 -> 154 us when unrolled by two).
    // A tile wholly inside the tensor takes a loop in which every chunk is valid: no bounds
    // test, zero fill or guarded store per chunk (NVFP4 with statistics 148 -> 146 us).
    if ((tile + 1) * kTileChunks <= n_chunks) {
#pragma unroll(PipeShape<FMT>::kUnroll)
      for (int c = 0; c < kCPT; ++c) {
        const int j = c * kThreads + tid;
        const int64_t u = tile * kTileChunks + j;
        uint32_t w[8];
        lds32B(w, stage + 32u * j);
        if (!STATS || acc.T >= 1.0f)
          q4_chunk<FMT, DT, UNIT, STATS, SR, false, AMAX>(a, cx, w, u, true, lane, acc, tpart, am);
        else
          q4_chunk<FMT, DT, UNIT, STATS, SR, true, AMAX>(a, cx, w, u, true, lane, acc, tpart, am);
      }
    } else
#pragma unroll(PipeShape<FMT>::kUnroll)
    for (int c = 0; c < kCPT; ++c) {
      const int j = c * kThreads + tid;
      const int64_t u = tile * kTileChunks + j;  // global 32-byte chunk
      const bool valid = u < n_chunks;
      uint32_t w[8];
      if (valid) {
        lds32B(w, stage + 32u * j);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = 0u;
      }
      if (!STATS || acc.T >= 1.0f)  // warp-uniform: the relative-error search is settled
        q4_chunk<FMT, DT, UNIT, STATS, SR, false, AMAX>(a, cx, w, u, valid, lane, acc, tpart, am);
      else
        q4_chunk<FMT, DT, UNIT, STATS, SR, true, AMAX>(a, cx, w, u, valid, lane, acc, tpart, am);
    }
    if constexpr (STATS) acc_add_sum(acc, tpart);
    __syncthreads();  // every thread is done with this stage
    if (s_abort) {
      if (tid == 0) {
        flag_status(a.ws, QZ_FLAG_PIPELINE_TIMEOUT);
        P.drain(k);
      }
      return;
    }
    if (tid == 0) P.issue(k + S);
  }
  if constexpr (AMAX) amax_finish<QZ_F32>(am, a.amax_out, a.ws);
  if constexpr (STATS) stats_finish(acc, a.ws, a.stats, static_cast<uint64_t>(a.g.rows * a.g.cols));
}

template <int FMT, int DT, bool UNIT, bool STATS, bool AMAX>
qz_status run_pipe_k(const Q4Args& args, cudaStream_t s) {
  auto kern = args.scale_round == QZ_SCALE_NEAREST ? &quant4_pipe_kernel<FMT, DT, UNIT, STATS, QZ_SCALE_NEAREST, AMAX>
                                                    : &quant4_pipe_kernel<FMT, DT, UNIT, STATS, QZ_SCALE_UP, AMAX>;
  constexpr size_t smem = static_cast<size_t>(PipeShape<FMT>::kStages) * kTileBytes;
  if (!set_dyn_smem(reinterpret_cast<const void*>(kern), static_cast<int>(smem)))
    return QZ_ERR_CUDA;
  const int grid = grid_for(reinterpret_cast<const void*>(kern),
                            (args.g.n_chunks + kTileChunks - 1) / kTileChunks, s, smem);
  kern<<<grid, kThreads, smem, s>>>(args);
  return launch_status();
}

// AMAX: also fold this tensor's amax into amax_out (the delayed-scaling call)
template <int FMT, int DT, bool UNIT, bool STATS>
qz_status run_pipe(const Q4Args& args, cudaStream_t s) {
  return args.amax_out ? run_pipe_k<FMT, DT, UNIT, STATS, true>(args, s)
                       : run_pipe_k<FMT, DT, UNIT, STATS, false>(args, s);
}

// With amax_out, the staged kernel folds the tensor amax in; the direct path leaves it to
// the caller (fused: returned true).
template <int FMT, int DT, bool UNIT, bool STATS, bool VEC>
qz_status run(const Q4Args& args, cudaStream_t s, bool& fused) {
  if constexpr (VEC) {
    if (args.g.dense && reinterpret_cast<uintptr_t>(args.x) % 16 == 0) {
      fused = true;
      return run_pipe<FMT, DT, UNIT, STATS>(args, s);
    }
  }
  auto kern = &quant4_kernel<FMT, DT, UNIT, STATS, VEC>;
  const int64_t per_cta = static_cast<int64_t>(kThreads) * kUnroll;
  const int grid = grid_for(reinterpret_cast<const void*>(kern), (args.g.n_chunks + per_cta - 1) / per_cta, s);
  kern<<<grid, kThreads, 0, s>>>(args);
  return launch_status();
}

template <int FMT, int DT>
qz_status dispatch(const Q4Args& args, bool unit, bool stats, cudaStream_t s, bool& f) {
  const bool vec = args.g.vec;
  if (unit) {
    if (stats) return vec ? run<FMT, DT, true, true, true>(args, s, f) : run<FMT, DT, true, true, false>(args, s, f);
    return vec ? run<FMT, DT, true, false, true>(args, s, f) : run<FMT, DT, true, false, false>(args, s, f);
  }
  if (stats) return vec ? run<FMT, DT, false, true, true>(args, s, f) : run<FMT, DT, false, true, false>(args, s, f);
  return vec ? run<FMT, DT, false, false, true>(args, s, f) : run<FMT, DT, false, false, false>(args, s, f);
}

}  // namespace

qz_status launch_quant4(const qz_desc& d, const void* x, void* codes, void* scales,
                        float* tscale_out, const float* amax, bool /*amax_supplied*/,
                        qz_stats* stats, void* ws, cudaStream_t s, float* amax_out) {
  const int eb = d.in_dtype == QZ_BF16 ? 2 : 4;
  Q4Args args;
  args.x = x;
  args.g = make_geom(d, x, eb, 32);
  // codes must allow the 8- / 4-byte word stores of the vector path
  if (reinterpret_cast<uintptr_t>(codes) % 16 != 0) {
    args.g.vec = false;
    args.g.dense = false;
  }
  args.codes = static_cast<uint8_t*>(codes);
  args.scales = static_cast<uint8_t*>(scales);
  args.amax = amax;
  args.tscale_out = tscale_out;
  args.stats = stats;
  args.ws = ws;
  args.scale_round = d.scale_round;
  // NVFP4 with a per-tensor scale is normally preceded by a full read of x for its amax;
  // starting from the end of x picks up what that read left in L2
  args.reverse = d.format == QZ_NVFP4 && d.granularity == QZ_GRAN_BLOCK;
  args.zero = 0.0f;
  args.amax_out = amax_out;
  const bool unit = d.granularity == QZ_GRAN_UNIT;
  const bool st = stats != nullptr;
  bool fused = false;
  qz_status rc;
  if (d.format == QZ_MXFP4)
    rc = d.in_dtype == QZ_BF16 ? dispatch<QZ_MXFP4, QZ_BF16>(args, unit, st, s, fused)
                               : dispatch<QZ_MXFP4, QZ_F32>(args, unit, st, s, fused);
  else
    rc = d.in_dtype == QZ_BF16 ? dispatch<QZ_NVFP4, QZ_BF16>(args, unit, st, s, fused)
                               : dispatch<QZ_NVFP4, QZ_F32>(args, unit, st, s, fused);
  if (rc == QZ_OK && amax_out && !fused) rc = launch_amax(d, x, amax_out, ws, s);
  return rc;
}

}  // namespace qz
