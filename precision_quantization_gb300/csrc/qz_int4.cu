// qz_int4.cu -- grouped symmetric INT4 (blog post "浅谈低精度浮点数", section "FP4 / MXFP4 /
// NVFP4", closing paragraph: q in [-7, 7], s = A / 7, analysed like INT8) and the
// asymmetric 4-bit group dequantization sc * (w - sh) of the "Puzzles 12 Quantized Matrix
// Mult" section of the blog's "Triton" post.
//
// INT4 keeps one fp32 scale per group of G values along cols (G = 16, 32, 64, 128) and
// stores the codes as 4-bit two's complement nibbles, element 2i in the low nibble of byte
// i.  Each lane owns one 32-byte chunk of x (16 bf16 / 8 fp32 values); a group spans
// L = G / chunk lanes of one warp, which finish the group amax with shuffles.
//
// Integer rounding: after clamping v to [-7, 7], t = v + 1.5 * 2^23 lies in [2^23, 2^24),
// where binary32 has unit spacing, so the addition rounds v to the nearest integer with
// ties to even, and the low bits of t's encoding are q in two's complement (t's field is
// 0x4B400000 + q): the nibble is those bits, and q itself is t - 1.5 * 2^23 (exact).
#include <type_traits>

#include "qz_device.cuh"
#include "qz_internal.h"
#include "qz_pipe.cuh"

namespace qz {
namespace {

constexpr int kUnroll = 2;               // chunks in flight per lane
constexpr float kMagic = 12582912.0f;    // 1.5 * 2^23
constexpr float kRcp7 = 0x1.24924ap-3f;  // RN(1/7)

struct I4Args {
  const void* x;
  Geom g;
  uint8_t* codes;
  float* scales;
  float* tscale_out;  // may be null: written 1 (INT4 has no per-tensor scale)
  qz_stats* stats;
  void* ws;
};

// fl32(A / 7), A >= 0: the FMA-corrected quotient where it is exact, IEEE division below
__device__ __forceinline__ float div7(float A) {
  return A >= 0x1p-100f ? div_pos(A, 7.0f, kRcp7) : __fdiv_rn(A, 7.0f);
}

// q (as the nibble and as a float) of the quotient v
__device__ __forceinline__ uint32_t int4_round(float v, float& qf) {
  const float t = __fadd_rn(fminf(fmaxf(v, -7.0f), 7.0f), kMagic);
  qf = __fsub_rn(t, kMagic);
  return __float_as_uint(t) & 0xFu;
}

// the value of a two's complement nibble, exactly
__device__ __forceinline__ float int4_value(uint32_t nib) {
  const uint32_t sext = (nib ^ 8u) - 8u;  // -8..7 as a 32-bit two's complement integer
  return __fsub_rn(__uint_as_float(0x4B400000u + sext), kMagic);
}

// 32-byte chunk u of x: its row, its first column, the element offset in x
struct ChunkPos {
  int64_t row, col, e0;
};
template <int EPC>
__device__ __forceinline__ ChunkPos chunk_pos(const Geom& g, int64_t u) {
  ChunkPos p;
  p.row = u / g.cpr;
  p.col = (u - p.row * g.cpr) * EPC;
  p.e0 = p.row * g.ld + p.col;
  return p;
}

template <int DT, bool VEC>
__device__ __forceinline__ void load_x_chunk(uint32_t (&w)[8], const void* x, int64_t e0) {
  if constexpr (VEC) {
    ld32B(w, static_cast<const char*>(x) + e0 * Elem<DT>::kBytes);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if constexpr (DT == QZ_BF16) {
        const uint32_t lo = __float_as_uint(load_elem<DT>(x, e0 + 2 * i)) >> 16;
        const uint32_t hi = __float_as_uint(load_elem<DT>(x, e0 + 2 * i + 1));
        w[i] = (hi & 0xffff0000u) | lo;
      } else {
        w[i] = __float_as_uint(load_elem<DT>(x, e0 + i));
      }
    }
  }
}

// Quantize (and optionally reduce the error of) every chunk; G values per group.
template <int DT, int G, bool STATS, bool VEC>
__global__ void __launch_bounds__(kThreads) int4_quant_kernel(I4Args a) {
  constexpr int EPC = Elem<DT>::kPer32B;
  constexpr int L = G / EPC;   // lanes per group
  constexpr int CB = EPC / 2;  // code bytes per chunk
  const Geom& g = a.g;
  const int lane = threadIdx.x & 31;
  const int64_t ng = g.cols / G;
  if (a.tscale_out && blockIdx.x == 0 && threadIdx.x == 0) *a.tscale_out = 1.0f;
  StatAcc acc;
  const int64_t warp_id = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarps * 32 * kUnroll;
  for (int64_t base = warp_id * 32 * kUnroll; base < g.n_chunks; base += stride) {
    uint32_t w[kUnroll][8];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const int64_t u = base + k * 32 + lane;
      if (u < g.n_chunks) {
        load_x_chunk<DT, VEC>(w[k], a.x, chunk_pos<EPC>(g, u).e0);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) w[k][i] = 0u;
      }
    }
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const int64_t u = base + k * 32 + lane;
      const bool valid = u < g.n_chunks;
      const ChunkPos p = chunk_pos<EPC>(g, valid ? u : 0);
      float xs[EPC];
#pragma unroll
      for (int i = 0; i < EPC; ++i) xs[i] = chunk_elem<DT>(w[k], i);
      float A = 0.0f;
#pragma unroll
      for (int i = 0; i < EPC; ++i) A = absmax_nan(A, xs[i]);
#pragma unroll
      for (int o = 1; o < L; o <<= 1) A = absmax_nan(A, __shfl_xor_sync(kFull, A, o));
      if (valid && !is_finite_f(A)) flag_status(a.ws, QZ_FLAG_NONFINITE_INPUT);

      float s = div7(A);
      if (s == 0.0f) s = 1.0f;
      const float r = __frcp_rn(s);
      const bool fast = fast_div_ok(s) && __fmul_rn(A, r) <= 0x1p126f;
      float qf[EPC];
      uint32_t nib[EPC];
#pragma unroll
      for (int i = 0; i < EPC; ++i) {
        const float v = fast ? div_by(xs[i], s, r) : __fdiv_rn(xs[i], s);
        nib[i] = int4_round(v, qf[i]);
      }
      uint32_t cw[CB / 4];
#pragma unroll
      for (int j = 0; j < CB / 4; ++j) {
        uint32_t word = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) word |= nib[8 * j + i] << (4 * i);
        cw[j] = word;
      }
      if (valid) {
        uint8_t* cp = a.codes + p.row * (g.cols / 2) + p.col / 2;
        if constexpr (CB == 8) {
          if (reinterpret_cast<uintptr_t>(cp) % 8 == 0) {
            asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(cp), "r"(cw[0]), "r"(cw[1]) : "memory");
          } else {
#pragma unroll
            for (int j = 0; j < CB; ++j) cp[j] = static_cast<uint8_t>(cw[j / 4] >> (8 * (j % 4)));
          }
        } else {
          if (reinterpret_cast<uintptr_t>(cp) % 4 == 0) {
            *reinterpret_cast<uint32_t*>(cp) = cw[0];
          } else {
#pragma unroll
            for (int j = 0; j < CB; ++j) cp[j] = static_cast<uint8_t>(cw[0] >> (8 * j));
          }
        }
        if (lane % L == 0) a.scales[p.row * ng + p.col / G] = s;
      }
      if constexpr (STATS) {
        float xh[EPC];
#pragma unroll
        for (int i = 0; i < EPC; ++i) xh[i] = __fmul_rn(qf[i], s);  // invalid lanes: x = 0, q = 0
        acc_chunk(acc, xs, xh);
      }
    }
  }
  if constexpr (STATS) stats_finish(acc, a.ws, a.stats, static_cast<uint64_t>(g.rows * g.cols));
}

// ---- staged path (dense, 16-byte aligned x): the quant4 tile pipeline ---------------
// One 32-byte chunk: group amax, scale, quotients (fp32 pairs), integer rounding, nibble
// packing, stores, and (STATS) the error.  |x| <= A and s = fl32(A/7) keep |fl32(x/s)|
// within 7 (1 + 2^-22) whenever A is normal, so the rounded q already lies in [-7, 7];
// groups with a subnormal A (or a zero scale replaced by 1) clamp first.
template <int DT, int G, bool STATS, bool REL>
__device__ __forceinline__ void i4_chunk(const I4Args& a, const uint32_t (&w)[8], int64_t u,
                                         bool valid, int lane, StatAcc& acc, float& tpart,
                                         float zero) {
  constexpr int EPC = Elem<DT>::kPer32B;
  constexpr int L = G / EPC;
  constexpr int NP = EPC / 2;
  uint64_t xp[NP];
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    if constexpr (DT == QZ_BF16) xp[p] = widen_bf16x2(w[p]);
    else xp[p] = pk(__uint_as_float(w[2 * p]), __uint_as_float(w[2 * p + 1]));
  }
  float A;
  if constexpr (DT == QZ_BF16) {
    A = bf16x16_absmax(w);  // packed bf16x2 maxima: fewer ALU slots than fp32 maxima
  } else {
    A = 0.0f;
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      float x0, x1;
      upk(xp[p], x0, x1);
      A = absmax3(A, x0, x1);
    }
  }
#pragma unroll
  for (int o = 1; o < L; o <<= 1) A = absmax_nan(A, __shfl_xor_sync(kFull, A, o));

  float s = div7(A);
  if (s == 0.0f) s = 1.0f;
  const float r = __frcp_rn(s);
  const bool fast = fast_div_ok(s) && __fmul_rn(A, r) <= 0x1p126f;
  uint64_t vp[NP];
  if (__all_sync(kFull, fast)) {  // a NaN / Inf amax makes s non-finite: never fast
    const uint64_t r2 = pk(r, r), ns2 = pk(-s, -s);
#pragma unroll
    for (int p = 0; p < NP; ++p) vp[p] = div2(xp[p], r2, ns2);
  } else {
    if (valid && !is_finite_f(A)) flag_status(a.ws, QZ_FLAG_NONFINITE_INPUT);
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      float x0, x1;
      upk(xp[p], x0, x1);
      vp[p] = fast ? div2(xp[p], pk(r, r), pk(-s, -s)) : pk(__fdiv_rn(x0, s), __fdiv_rn(x1, s));
    }
  }
  if (!__all_sync(kFull, A >= 0x1p-100f || A == 0.0f)) {
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      float v0, v1;
      upk(vp[p], v0, v1);
      vp[p] = pk(fminf(fmaxf(v0, -7.0f), 7.0f), fminf(fmaxf(v1, -7.0f), 7.0f));
    }
  }
  // t = v + 1.5 * 2^23: RNE to an integer; its low field bits are q (two's complement)
  const uint64_t magic2 = pk(kMagic, kMagic);
  uint64_t tp[NP];
#pragma unroll
  for (int p = 0; p < NP; ++p) tp[p] = add2(vp[p], magic2);
  uint32_t cw[EPC / 8];
#pragma unroll
  for (int g8 = 0; g8 < EPC / 8; ++g8) {
    uint32_t by[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float t0, t1;
      upk(tp[4 * g8 + i], t0, t1);
      // bits [0,4) from t0, bits [4,8) from t1 (the other bits are discarded below)
      by[i] = (__float_as_uint(t0) & 0x0Fu) | (__float_as_uint(t1) << 4 & ~0x0Fu);
    }
    cw[g8] = __byte_perm(__byte_perm(by[0], by[1], 0x0040), __byte_perm(by[2], by[3], 0x0040), 0x5410);
  }
  {  // predicated stores
    uint8_t* cp = a.codes + u * (EPC / 2);
    const uint32_t pv = valid ? 1u : 0u, ps = (valid && lane % L == 0) ? 1u : 0u;
    if constexpr (EPC == 16) {
      asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %3, 0;\n\t@p st.global.v2.u32 [%0], {%1, %2};\n\t}"
                   ::"l"(cp), "r"(cw[0]), "r"(cw[1]), "r"(pv) : "memory");
    } else {
      asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %2, 0;\n\t@p st.global.u32 [%0], %1;\n\t}"
                   ::"l"(cp), "r"(cw[0]), "r"(pv) : "memory");
    }
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %2, 0;\n\t@p st.global.f32 [%0], %1;\n\t}"
                 ::"l"(a.scales + u / L), "f"(s), "r"(ps) : "memory");
  }
  if constexpr (STATS) {
    const uint64_t s2 = pk(s, s), z2 = pk(zero, zero);
    Pairs<NP> e;
#pragma unroll
    for (int p = 0; p < NP; ++p) e.v[p] = sub2(xp[p], mul2_rounded(sub2(tp[p], magic2), s2, z2));
    acc_pairs<NP, REL>(acc, xp, e, tpart);
  }
}

template <int DT, int G, bool STATS>
__global__ void __launch_bounds__(kThreads, 3) int4_pipe_kernel(I4Args a, float zero) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kPipeStages];
  __shared__ int s_abort;
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t n_chunks = a.g.n_chunks;
  if (a.tscale_out && blockIdx.x == 0 && tid == 0) *a.tscale_out = 1.0f;
  if (tid == 0) {
    for (int i = 0; i < kPipeStages; ++i) mbar_init(smem_addr(&bars[i]), 1);
    mbar_init_fence();
    s_abort = 0;
  }
  __syncthreads();
  const BulkPipe<kPipeStages, kPipeTileBytes> P{smem_addr(smem), smem_addr(&bars[0]),
                                                static_cast<const char*>(a.x), n_chunks * 32,
                                                (n_chunks + kPipeTileChunks - 1) / kPipeTileChunks,
                                                false};
  if (tid == 0) P.prologue();
  StatAcc acc;
  for (int64_t k = 0; P.has(k); ++k) {
    const int64_t tile = P.tile_of(k);
    if (!P.wait(k)) s_abort = 1;
    float tpart = 0.0f;
    const uint32_t stage = P.stage(k);
#pragma unroll 1  // not unrolled: a smaller loop body (measured 160 -> 152 us, 32768 x 8192 bf16)
    for (int c = 0; c < kPipeCPT; ++c) {
      const int j = c * kThreads + tid;
      const int64_t u = tile * kPipeTileChunks + j;
      const bool valid = u < n_chunks;
      uint32_t w[8];
      if (valid) {
        lds32B(w, stage + 32u * j);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = 0u;
      }
      if (!STATS || acc.T >= 1.0f)  // warp-uniform: the relative-error search is settled
        i4_chunk<DT, G, STATS, false>(a, w, u, valid, lane, acc, tpart, zero);
      else
        i4_chunk<DT, G, STATS, true>(a, w, u, valid, lane, acc, tpart, zero);
    }
    if constexpr (STATS) acc_add_sum(acc, tpart);
    __syncthreads();
    if (s_abort) {
      if (tid == 0) {
        flag_status(a.ws, QZ_FLAG_PIPELINE_TIMEOUT);
        P.drain(k);
      }
      return;
    }
    if (tid == 0) P.issue(k + kPipeStages);
  }
  if constexpr (STATS) stats_finish(acc, a.ws, a.stats, static_cast<uint64_t>(a.g.rows * a.g.cols));
}

// x^ of one chunk from its codes and group scale
template <int EPC>
__device__ __forceinline__ void int4_chunk_values(const uint8_t* codes, const float* scales,
                                                  const Geom& g, int G, const ChunkPos& p,
                                                  float (&xh)[EPC]) {
  constexpr int CB = EPC / 2;
  const uint8_t* cp = codes + p.row * (g.cols / 2) + p.col / 2;
  uint32_t cw[CB / 4];
  if (reinterpret_cast<uintptr_t>(cp) % 4 == 0) {
#pragma unroll
    for (int j = 0; j < CB / 4; ++j) cw[j] = reinterpret_cast<const uint32_t*>(cp)[j];
  } else {
#pragma unroll
    for (int j = 0; j < CB / 4; ++j) {
      cw[j] = 0u;
#pragma unroll
      for (int b = 0; b < 4; ++b) cw[j] |= static_cast<uint32_t>(cp[4 * j + b]) << (8 * b);
    }
  }
  const float s = scales[p.row * (g.cols / G) + p.col / G];
#pragma unroll
  for (int i = 0; i < EPC; ++i) xh[i] = __fmul_rn(int4_value((cw[i / 8] >> (4 * (i % 8))) & 0xFu), s);
}

template <int ODT, int G>
__global__ void __launch_bounds__(kThreads) int4_dequant_kernel(const uint8_t* codes, const float* scales,
                                                                void* y, Geom g, bool vec) {
  constexpr int EPC = Elem<ODT>::kPer32B;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t nthr = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t u = tid; u < g.n_chunks; u += nthr) {
    const ChunkPos p = chunk_pos<EPC>(g, u);
    float xh[EPC];
    int4_chunk_values<EPC>(codes, scales, g, G, p, xh);
    if (vec) {
      uint32_t o[8];
      if constexpr (ODT == QZ_BF16) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o[i]) : "f"(xh[2 * i + 1]), "f"(xh[2 * i]));
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = __float_as_uint(xh[i]);
      }
      st32B(static_cast<char*>(y) + p.e0 * Elem<ODT>::kBytes, o);
    } else {
#pragma unroll
      for (int i = 0; i < EPC; ++i) store_elem<ODT>(y, p.e0 + i, xh[i]);
    }
  }
}

template <int DT, int G, bool VEC>
__global__ void __launch_bounds__(kThreads) int4_stats_kernel(I4Args a) {
  constexpr int EPC = Elem<DT>::kPer32B;
  const Geom& g = a.g;
  StatAcc acc;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t nthr = static_cast<int64_t>(gridDim.x) * kThreads;
  // warp-uniform trip count (the relative-error vote in acc_chunk)
  for (int64_t ub = tid - (threadIdx.x & 31); ub < g.n_chunks; ub += nthr) {
    const int64_t u = ub + (threadIdx.x & 31);
    float xs[EPC], xh[EPC];
    if (u < g.n_chunks) {
      const ChunkPos p = chunk_pos<EPC>(g, u);
      uint32_t w[8];
      load_x_chunk<DT, VEC>(w, a.x, p.e0);
#pragma unroll
      for (int i = 0; i < EPC; ++i) {
        xs[i] = chunk_elem<DT>(w, i);
        if (!is_finite_f(xs[i])) flag_status(a.ws, QZ_FLAG_NONFINITE_INPUT);
      }
      int4_chunk_values<EPC>(a.codes, a.scales, g, G, p, xh);
    } else {
#pragma unroll
      for (int i = 0; i < EPC; ++i) xs[i] = xh[i] = 0.0f;
    }
    acc_chunk(acc, xs, xh);
  }
  stats_finish(acc, a.ws, a.stats, static_cast<uint64_t>(g.rows * g.cols));
}

// ---- asymmetric 4-bit group dequantization ---------------------------------------------
struct A4Args {
  const uint32_t* w;
  const float* scales;
  const uint32_t* shifts;
  void* y;
  int64_t rows, cols, group, ld;
};

template <int ODT, bool GROUP8>
__global__ void __launch_bounds__(kThreads) asym4_dequant_kernel(A4Args a) {
  const int64_t wpr = a.cols / 8;                  // code words per row
  const int64_t ng = a.cols / a.group;             // groups per row
  const int64_t sw = (ng + 7) / 8;                 // shift words per row
  const int64_t nwords = a.rows * wpr;
  const bool vec = (reinterpret_cast<uintptr_t>(a.y) % (8 * Elem<ODT>::kBytes) == 0) &&
                   (a.ld % 8 == 0);
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t nthr = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t wi = tid; wi < nwords; wi += nthr) {
    const int64_t row = wi / wpr, c0 = (wi - row * wpr) * 8;
    const uint32_t word = a.w[wi];
    float out[8];
    if constexpr (GROUP8) {  // the 8 codes share one group
      const int64_t j = c0 / a.group;
      const float sc = a.scales[row * ng + j];
      const uint32_t sh = (a.shifts[row * sw + j / 8] >> (4 * (j % 8))) & 0xFu;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t d = ((word >> (4 * i)) & 0xFu) - sh;  // w - sh, two's complement
        out[i] = __fmul_rn(sc, __fsub_rn(__uint_as_float(0x4B400000u + d), kMagic));
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int64_t j = (c0 + i) / a.group;
        const float sc = a.scales[row * ng + j];
        const uint32_t sh = (a.shifts[row * sw + j / 8] >> (4 * (j % 8))) & 0xFu;
        const uint32_t d = ((word >> (4 * i)) & 0xFu) - sh;
        out[i] = __fmul_rn(sc, __fsub_rn(__uint_as_float(0x4B400000u + d), kMagic));
      }
    }
    const int64_t e0 = row * a.ld + c0;
    if (vec) {
      if constexpr (ODT == QZ_BF16) {
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o[i]) : "f"(out[2 * i + 1]), "f"(out[2 * i]));
        asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(static_cast<uint16_t*>(a.y) + e0),
                     "r"(o[0]), "r"(o[1]), "r"(o[2]), "r"(o[3])
                     : "memory");
      } else {
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = __float_as_uint(out[i]);
        st32B(static_cast<float*>(a.y) + e0, o);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) store_elem<ODT>(a.y, e0 + i, out[i]);
    }
  }
}

template <typename K>
int grid_of(K kern, int64_t work_items, int per_thread, cudaStream_t s) {
  const int64_t per_cta = static_cast<int64_t>(kThreads) * per_thread;
  return grid_for(reinterpret_cast<const void*>(kern), (work_items + per_cta - 1) / per_cta, s);
}

template <int DT, int G>
qz_status quant_g(const I4Args& a, bool stats, cudaStream_t s) {
  const int64_t chunks = a.g.n_chunks;
  if (a.g.vec && a.g.dense && reinterpret_cast<uintptr_t>(a.x) % 16 == 0 &&
      reinterpret_cast<uintptr_t>(a.codes) % 8 == 0) {
    auto k = stats ? &int4_pipe_kernel<DT, G, true> : &int4_pipe_kernel<DT, G, false>;
    if (!set_dyn_smem(reinterpret_cast<const void*>(k), static_cast<int>(kPipeSmem))) return QZ_ERR_CUDA;
    const int grid = grid_for(reinterpret_cast<const void*>(k),
                              (chunks + kPipeTileChunks - 1) / kPipeTileChunks, s, kPipeSmem);
    k<<<grid, kThreads, kPipeSmem, s>>>(a, 0.0f);
    return launch_status();
  }
  if (stats) {
    if (a.g.vec) {
      auto k = &int4_quant_kernel<DT, G, true, true>;
      k<<<grid_of(k, chunks, kUnroll, s), kThreads, 0, s>>>(a);
    } else {
      auto k = &int4_quant_kernel<DT, G, true, false>;
      k<<<grid_of(k, chunks, kUnroll, s), kThreads, 0, s>>>(a);
    }
  } else {
    if (a.g.vec) {
      auto k = &int4_quant_kernel<DT, G, false, true>;
      k<<<grid_of(k, chunks, kUnroll, s), kThreads, 0, s>>>(a);
    } else {
      auto k = &int4_quant_kernel<DT, G, false, false>;
      k<<<grid_of(k, chunks, kUnroll, s), kThreads, 0, s>>>(a);
    }
  }
  return launch_status();
}

template <int DT, int G>
qz_status stats_g(const I4Args& a, cudaStream_t s) {
  if (a.g.vec) {
    auto k = &int4_stats_kernel<DT, G, true>;
    k<<<grid_of(k, a.g.n_chunks, 1, s), kThreads, 0, s>>>(a);
  } else {
    auto k = &int4_stats_kernel<DT, G, false>;
    k<<<grid_of(k, a.g.n_chunks, 1, s), kThreads, 0, s>>>(a);
  }
  return launch_status();
}

template <int ODT, int G>
qz_status dequant_g(const uint8_t* codes, const float* scales, void* y, const Geom& g, cudaStream_t s) {
  auto k = &int4_dequant_kernel<ODT, G>;
  k<<<grid_of(k, g.n_chunks, 1, s), kThreads, 0, s>>>(codes, scales, y, g, g.vec);
  return launch_status();
}

// G = 16, 32, 64, 128 (validated by the caller)
template <typename F>
qz_status by_group(int G, F&& f) {
  switch (G) {
    case 16: return f(std::integral_constant<int, 16>{});
    case 32: return f(std::integral_constant<int, 32>{});
    case 64: return f(std::integral_constant<int, 64>{});
    default: return f(std::integral_constant<int, 128>{});
  }
}

}  // namespace

qz_status launch_quant_int4(const qz_desc& d, const void* x, void* codes, void* scales,
                            float* tscale_out, qz_stats* stats, void* ws, cudaStream_t s) {
  I4Args a;
  a.x = x;
  a.g = make_geom(d, x, d.in_dtype == QZ_BF16 ? 2 : 4, 32);
  a.codes = static_cast<uint8_t*>(codes);
  a.scales = static_cast<float*>(scales);
  a.tscale_out = tscale_out;
  a.stats = stats;
  a.ws = ws;
  return by_group(d.block_size, [&](auto G) {
    return d.in_dtype == QZ_BF16 ? quant_g<QZ_BF16, decltype(G)::value>(a, stats != nullptr, s)
                                 : quant_g<QZ_F32, decltype(G)::value>(a, stats != nullptr, s);
  });
}

qz_status launch_stats_int4(const qz_desc& d, const void* x, const void* codes, const void* scales,
                            qz_stats* stats, void* ws, cudaStream_t s) {
  I4Args a;
  a.x = x;
  a.g = make_geom(d, x, d.in_dtype == QZ_BF16 ? 2 : 4, 32);
  a.codes = static_cast<uint8_t*>(const_cast<void*>(codes));
  a.scales = static_cast<float*>(const_cast<void*>(scales));
  a.tscale_out = nullptr;
  a.stats = stats;
  a.ws = ws;
  return by_group(d.block_size, [&](auto G) {
    return d.in_dtype == QZ_BF16 ? stats_g<QZ_BF16, decltype(G)::value>(a, s)
                                 : stats_g<QZ_F32, decltype(G)::value>(a, s);
  });
}

qz_status launch_dequant_int4(const qz_desc& d, const void* codes, const void* scales, void* y,
                              int out_dtype, cudaStream_t s) {
  const Geom g = make_geom(d, y, out_dtype == QZ_BF16 ? 2 : 4, 32);
  const uint8_t* c = static_cast<const uint8_t*>(codes);
  const float* sc = static_cast<const float*>(scales);
  return by_group(d.block_size, [&](auto G) {
    return out_dtype == QZ_BF16 ? dequant_g<QZ_BF16, decltype(G)::value>(c, sc, y, g, s)
                                : dequant_g<QZ_F32, decltype(G)::value>(c, sc, y, g, s);
  });
}

qz_status launch_dequant_asym4(const uint32_t* w, const float* scales, const uint32_t* shifts,
                               int64_t rows, int64_t cols, int64_t group, void* y, int64_t ld,
                               int out_dtype, cudaStream_t s) {
  const A4Args a{w, scales, shifts, y, rows, cols, group, ld};
  const int64_t words = rows * (cols / 8);
  const bool g8 = group % 8 == 0;
  if (out_dtype == QZ_BF16) {
    if (g8) {
      auto k = &asym4_dequant_kernel<QZ_BF16, true>;
      k<<<grid_of(k, words, 1, s), kThreads, 0, s>>>(a);
    } else {
      auto k = &asym4_dequant_kernel<QZ_BF16, false>;
      k<<<grid_of(k, words, 1, s), kThreads, 0, s>>>(a);
    }
  } else {
    if (g8) {
      auto k = &asym4_dequant_kernel<QZ_F32, true>;
      k<<<grid_of(k, words, 1, s), kThreads, 0, s>>>(a);
    } else {
      auto k = &asym4_dequant_kernel<QZ_F32, false>;
      k<<<grid_of(k, words, 1, s), kThreads, 0, s>>>(a);
    }
  }
  return launch_status();
}

}  // namespace qz
