// qz_quant8.cu -- quantize to symmetric INT8, FP8 E4M3 or FP8 E5M2 with one scale per
// tensor, one per row, or the unit scale (blog post "浅谈低精度浮点数", section "FP8":
// x^ = s * round(x / s), s = alpha / 127 for INT8; FP8 scales map alpha onto the format
// maximum), optionally with the error statistics fused into the same pass.
//
// Each lane owns a 32-byte chunk of a row (16 bf16 / 8 fp32 values -> 16 / 8 code bytes).
// The per-row kernel gives every row to one CTA: the row is read once into registers,
// its amax reduced across the CTA, and the codes produced from the registers.
#include "qz_device.cuh"
#include "qz_internal.h"
#include "qz_pipe.cuh"

namespace qz {
namespace {

enum Mode { kTensorComputed = 0, kTensorSupplied = 1, kUnit = 2 };

struct Q8Args {
  const void* x;
  Geom g;
  uint8_t* codes;
  float* scales;      // ROW
  const float* amax;  // TENSOR
  float* tscale_out;
  qz_stats* stats;
  void* ws;
  float* amax_out = nullptr;  // staged per-tensor-supplied / unit path: this tensor's max |x|
};

// Load chunk u = (row, chunk index j) of x into w (zero-filled past the end of the row).
template <int DT, bool VEC>
__device__ __forceinline__ void load_chunk(uint32_t (&w)[8], const void* x, const Geom& g,
                                           int64_t row, int64_t col) {
  constexpr int EPC = Elem<DT>::kPer32B;
  const int64_t e0 = row * g.ld + col;
  if constexpr (VEC) {
    ld32B(w, static_cast<const char*>(x) + e0 * Elem<DT>::kBytes);
  } else {
    const int64_t nv = g.cols - col;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if constexpr (DT == QZ_BF16) {
        const uint32_t lo = (2 * i < nv) ? (__float_as_uint(load_elem<DT>(x, e0 + 2 * i)) >> 16) : 0u;
        const uint32_t hi = (2 * i + 1 < nv) ? __float_as_uint(load_elem<DT>(x, e0 + 2 * i + 1)) : 0u;
        w[i] = (hi & 0xffff0000u) | lo;
      } else {
        w[i] = (i < nv) ? __float_as_uint(load_elem<DT>(x, e0 + i)) : 0u;
      }
    }
    (void)EPC;
  }
}

// Quantize one chunk with scale s (r = RN(1/s)); `exact` selects the Markstein quotient,
// otherwise IEEE division; unit scale skips the division.  Stores the codes and, with
// STATS, accumulates the error of the chunk.
template <int FMT, int DT, bool STATS, bool VEC, bool UNIT>
__device__ __forceinline__ void quant_chunk(const uint32_t (&w)[8], bool valid, int64_t nv,
                                            float s, float r, bool fast, uint8_t* cp,
                                            StatAcc& acc) {
  constexpr int EPC = Elem<DT>::kPer32B;
  float xs[EPC];
#pragma unroll
  for (int i = 0; i < EPC; ++i) xs[i] = chunk_elem<DT>(w, i);
  float v[EPC];
#pragma unroll
  for (int i = 0; i < EPC; ++i) {
    if constexpr (UNIT) v[i] = xs[i];
    else v[i] = fast ? div_by(xs[i], s, r) : __fdiv_rn(xs[i], s);
  }
  uint32_t cw[EPC / 4];
#pragma unroll
  for (int j = 0; j < EPC / 4; ++j)
    cw[j] = cvt8x2<FMT>(v[4 * j], v[4 * j + 1]) | (cvt8x2<FMT>(v[4 * j + 2], v[4 * j + 3]) << 16);
  if (valid) {
    if constexpr (VEC) {
      if constexpr (EPC == 16) {
        asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(cp), "r"(cw[0]), "r"(cw[1]),
                     "r"(cw[2]), "r"(cw[3])
                     : "memory");
      } else {
        asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(cp), "r"(cw[0]), "r"(cw[1]) : "memory");
      }
    } else {
#pragma unroll
      for (int j = 0; j < EPC; ++j)
        if (j < nv) cp[j] = static_cast<uint8_t>(cw[j / 4] >> (8 * (j % 4)));
    }
  }
  if constexpr (STATS) {
    // elements past the end of a row hold x = 0 and code 0 -> e = 0
    float xh[EPC];
#pragma unroll
    for (int j = 0; j < EPC / 2; ++j) {
      float q0, q1;
      dec8x2<FMT>((cw[j / 2] >> (16 * (j % 2))) & 0xffffu, q0, q1);
      xh[2 * j] = __fmul_rn(q0, s);
      xh[2 * j + 1] = __fmul_rn(q1, s);
    }
    acc_chunk(acc, xs, xh);
  }
}

constexpr int kUnroll = 2;

template <int FMT, int DT, int MODE, bool STATS, bool VEC>
__global__ void __launch_bounds__(kThreads) quant8_kernel(Q8Args a) {
  constexpr int EPC = Elem<DT>::kPer32B;
  const Geom& g = a.g;
  const int lane = threadIdx.x & 31;
  float s = 1.0f, r = 1.0f;
  bool fast = true;
  if constexpr (MODE != kUnit) {
    const float alpha = *a.amax;
    if (MODE == kTensorSupplied && (!(alpha >= 0.0f) || !is_finite_f(alpha)) && blockIdx.x == 0 &&
        threadIdx.x == 0)
      flag_status(a.ws, QZ_FLAG_BAD_AMAX);
    s = __fdiv_rn(alpha, Fmt8<FMT>::kMax);
    if (s == 0.0f) s = 1.0f;
    r = __frcp_rn(s);
    fast = fast_div_ok(s);
  }
  if (a.tscale_out && blockIdx.x == 0 && threadIdx.x == 0) *a.tscale_out = s;

  StatAcc acc;
  const int64_t warp_id = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarps * 32 * kUnroll;
  for (int64_t base = warp_id * 32 * kUnroll; base < g.n_chunks; base += stride) {
    uint32_t w[kUnroll][8];
    int64_t row[kUnroll], col[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const int64_t u = base + k * 32 + lane;
      if (g.dense) {  // full chunks, rows back to back: flat element index
        row[k] = 0;
        col[k] = u * EPC;
      } else {
        row[k] = u / g.cpr;
        col[k] = (u - row[k] * g.cpr) * EPC;
      }
      if (u < g.n_chunks) {
        load_chunk<DT, VEC>(w[k], a.x, g, row[k], col[k]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) w[k][i] = 0u;
      }
    }
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const int64_t u = base + k * 32 + lane;
      const bool valid = u < g.n_chunks;
      bool f = fast;
      if constexpr (MODE != kTensorComputed) {
        // no earlier pass has looked at these values: check finiteness here, and keep the
        // FMA quotient only where |x| / s cannot overflow (a supplied amax may be too small)
        float A = 0.0f;
#pragma unroll
        for (int i = 0; i < EPC; ++i) A = absmax_nan(A, chunk_elem<DT>(w[k], i));
        if (valid && !is_finite_f(A)) flag_status(a.ws, QZ_FLAG_NONFINITE_INPUT);
        if constexpr (MODE == kTensorSupplied) f = f && (__fmul_rn(A, r) <= 0x1p126f);
      }
      uint8_t* cp = a.codes + row[k] * g.cols + col[k];
      const int64_t nv = g.dense ? EPC : g.cols - col[k];
      quant_chunk<FMT, DT, STATS, VEC, MODE == kUnit>(w[k], valid, nv, s, r, f, cp, acc);
    }
  }
  if constexpr (STATS) stats_finish(acc, a.ws, a.stats, static_cast<uint64_t>(g.rows * g.cols));
}

// One CTA per row.  RCH > 0: the row is at most RCH chunks per thread and stays in
// registers between the amax and the quantize pass (vector path).  RCH == 0: any row
// length, x is read twice (the second read mostly hits L2).
template <int FMT, int DT, bool STATS, bool VEC, int RCH>
__global__ void __launch_bounds__(kThreads) quant8_row_kernel(Q8Args a) {
  constexpr int EPC = Elem<DT>::kPer32B;
  const Geom& g = a.g;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __shared__ float s_red[kWarps];
  if (a.tscale_out && blockIdx.x == 0 && threadIdx.x == 0) *a.tscale_out = 1.0f;
  StatAcc acc;
  for (int64_t row = blockIdx.x; row < g.rows; row += gridDim.x) {
    constexpr int NR = RCH > 0 ? RCH : 1;
    uint32_t w[NR][8];
    float A = 0.0f;
    if constexpr (RCH > 0) {
#pragma unroll
      for (int k = 0; k < RCH; ++k) {
        const int64_t j = threadIdx.x + static_cast<int64_t>(k) * kThreads;
        if (j < g.cpr) {
          load_chunk<DT, VEC>(w[k], a.x, g, row, j * EPC);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) w[k][i] = 0u;
        }
#pragma unroll
        for (int i = 0; i < EPC; ++i) A = absmax_nan(A, chunk_elem<DT>(w[k], i));
      }
    } else {
      for (int64_t j = threadIdx.x; j < g.cpr; j += kThreads) {
        load_chunk<DT, VEC>(w[0], a.x, g, row, j * EPC);
#pragma unroll
        for (int i = 0; i < EPC; ++i) A = absmax_nan(A, chunk_elem<DT>(w[0], i));
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) A = absmax_nan(A, __shfl_xor_sync(kFull, A, o));
    if (lane == 0) s_red[warp] = A;
    __syncthreads();
    A = s_red[0];
#pragma unroll
    for (int i = 1; i < kWarps; ++i) A = absmax_nan(A, s_red[i]);
    __syncthreads();  // s_red is reused by the next row
    float s = __fdiv_rn(A, Fmt8<FMT>::kMax);
    if (s == 0.0f) s = 1.0f;
    const float r = __frcp_rn(s);
    const bool fast = fast_div_ok(s);
    if (threadIdx.x == 0) {
      a.scales[row] = s;
      if (!is_finite_f(A)) flag_status(a.ws, QZ_FLAG_NONFINITE_INPUT);
    }
    uint8_t* crow = a.codes + row * g.cols;
    if constexpr (RCH > 0) {
#pragma unroll
      for (int k = 0; k < RCH; ++k) {
        const int64_t j = threadIdx.x + static_cast<int64_t>(k) * kThreads;
        if (static_cast<int64_t>(k) * kThreads + (threadIdx.x & ~31) < g.cpr)  // warp-uniform
          quant_chunk<FMT, DT, STATS, VEC, false>(w[k], j < g.cpr, g.cols - j * EPC, s, r, fast,
                                                   crow + j * EPC, acc);
      }
    } else {
      for (int64_t jb = threadIdx.x & ~31; jb < g.cpr; jb += kThreads) {  // warp-uniform trip
        const int64_t j = jb + lane;
        const bool valid = j < g.cpr;
        if (valid) {
          load_chunk<DT, VEC>(w[0], a.x, g, row, j * EPC);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) w[0][i] = 0u;
        }
        quant_chunk<FMT, DT, STATS, VEC, false>(w[0], valid, g.cols - j * EPC, s, r, fast,
                                                 crow + j * EPC, acc);
      }
    }
  }
  if constexpr (STATS) stats_finish(acc, a.ws, a.stats, static_cast<uint64_t>(g.rows * g.cols));
}

// ---------------------------------------------------------------------------------------
// Staged (shared-memory) paths, see qz_pipe.cuh
// ---------------------------------------------------------------------------------------
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23: fl(v + kMagic) - kMagic = RNE(v), |v| < 2^22

// Cast the quotients of one chunk (NP fp32 pairs) to codes.  Writes the EPC code bytes
// (element 0 in the lowest byte of cw[0]) and, with STATS, the code values q as fp32 pairs.
// INT8 rounds with the magic-number addition, which leaves RNE(v) in the low byte of the
// sum's bits and needs no float-to-int conversion; CLAMP limits v to [-127, 127] first
// (only needed when |v| can exceed 127.5: a supplied amax or the unit scale).
template <int FMT, int NP, bool STATS, bool CLAMP>
__device__ __forceinline__ void q8_cast(const uint64_t (&vp)[NP], uint32_t (&cw)[NP / 2],
                                        uint64_t (&qf)[NP]) {
  if constexpr (FMT == QZ_INT8) {
    const uint64_t m2 = pk(kMagic, kMagic);
    uint32_t lo[NP], hi[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      uint64_t v2 = vp[p];
      if constexpr (CLAMP) {
        float a, b;
        upk(v2, a, b);
        v2 = pk(fminf(fmaxf(a, -127.0f), 127.0f), fminf(fmaxf(b, -127.0f), 127.0f));
      }
      const uint64_t t2 = add2(v2, m2);
      if constexpr (STATS) qf[p] = sub2(t2, m2);
      float tl, th;
      upk(t2, tl, th);
      lo[p] = __float_as_uint(tl);
      hi[p] = __float_as_uint(th);
    }
#pragma unroll
    for (int p = 0; p < NP; p += 2) {
      const uint32_t u01 = __byte_perm(lo[p], hi[p], 0x0040);
      const uint32_t u23 = __byte_perm(lo[p + 1], hi[p + 1], 0x0040);
      cw[p / 2] = __byte_perm(u01, u23, 0x5410);
    }
  } else {
    uint32_t h16[NP];
#pragma unroll
    for (int p = 0; p < NP; ++p) {
      float a, b;
      upk(vp[p], a, b);
      h16[p] = cvt8x2<FMT>(a, b);
      if constexpr (STATS) {
        uint32_t hh;
        const uint16_t c = static_cast<uint16_t>(h16[p]);
        if constexpr (FMT == QZ_FP8_E4M3) asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hh) : "h"(c));
        else asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(hh) : "h"(c));
        qf[p] = f16x2_to_f32x2(hh);
      }
    }
#pragma unroll
    for (int p = 0; p < NP; p += 2) cw[p / 2] = (h16[p] & 0xffffu) | (h16[p + 1] << 16);
  }
}

// One chunk of the per-tensor / unit-scale path: quotients, cast, store, stats.  am: running
// max of the chunk amaxes' bits (MODE != kTensorComputed; the tensor amax for amax_out).
template <int FMT, int DT, int MODE, bool STATS, bool REL, bool AMAX = true>
__device__ __forceinline__ void q8_chunk(const uint32_t (&w)[8], bool valid, uint8_t* cp, float s,
                                         uint64_t r2, uint64_t ns2, uint64_t s2, uint64_t z2, bool fast,
                                         void* ws, StatAcc& acc, float& tpart, uint32_t& am) {
  constexpr int EPC = Elem<DT>::kPer32B;
  constexpr int NP = EPC / 2;
  uint64_t xp[NP];
#pragma unroll
  for (int p = 0; p < NP; ++p) {
    if constexpr (DT == QZ_BF16) xp[p] = widen_bf16x2(w[p]);
    else xp[p] = pk(__uint_as_float(w[2 * p]), __uint_as_float(w[2 * p + 1]));
  }
  bool f = fast;
  if constexpr (MODE != kTensorComputed) {
    // no earlier pass has looked at these values: check finiteness here, and keep the FMA
    // quotient only where |x| / s cannot overflow (a supplied amax may be too small)
    float A;
    if constexpr (DT == QZ_BF16) {
      A = bf16x16_absmax(w);  // packed bf16x2 maxima: fewer ALU slots than fp32 maxima
    } else {
      A = 0.0f;
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        float a, b;
        upk(xp[p], a, b);
        A = absmax3(A, a, b);
      }
    }
    // UNIT checks finiteness here; with a supplied scale a NaN / Inf A fails the quotient
    // range test and is flagged on the division path below
    if (MODE == kUnit && valid && !is_finite_f(A)) flag_status(ws, QZ_FLAG_NONFINITE_INPUT);
    if constexpr (AMAX) am = max(am, __float_as_uint(A));
    if constexpr (MODE == kTensorSupplied) {
      float r, rr;
      upk(r2, r, rr);
      f = f && (__fmul_rn(A, r) <= 0x1p126f);
      if (!f && valid && !is_finite_f(A)) flag_status(ws, QZ_FLAG_NONFINITE_INPUT);
    }
  }
  uint64_t vp[NP];
  if constexpr (MODE == kUnit) {
#pragma unroll
    for (int p = 0; p < NP; ++p) vp[p] = xp[p];
  } else {
    if (f) {
#pragma unroll
      for (int p = 0; p < NP; ++p) vp[p] = div2(xp[p], r2, ns2);
    } else {
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        float a, b;
        upk(xp[p], a, b);
        vp[p] = pk(__fdiv_rn(a, s), __fdiv_rn(b, s));
      }
    }
  }
  uint32_t cw[NP / 2];
  uint64_t qf[NP];
  q8_cast<FMT, NP, STATS, MODE != kTensorComputed>(vp, cw, qf);
  if (valid) {
    if constexpr (EPC == 16) {
      asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(cp), "r"(cw[0]), "r"(cw[1]),
                   "r"(cw[2]), "r"(cw[3])
                   : "memory");
    } else {
      asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(cp), "r"(cw[0]), "r"(cw[1]) : "memory");
    }
  }
  if constexpr (STATS) {
    // x^ = fl32(q * s) (= q for the unit scale), e = fl32(x - x^)
    Pairs<NP> e;
#pragma unroll
    for (int p = 0; p < NP; ++p) e.v[p] = sub2(xp[p], MODE == kUnit ? qf[p] : mul2_rounded(qf[p], s2, z2));
    acc_pairs<NP, REL>(acc, xp, e, tpart);
  }
}

// Dense tensors, per-tensor or unit scale: the quant4 pipeline (32 KiB tiles streamed
// through shared memory by bulk copies, four 32-byte chunks per lane per tile).
template <int FMT, int DT, int MODE, bool STATS, bool AMAX>
__global__ void __launch_bounds__(kThreads, 3) quant8_pipe_kernel(Q8Args a, float zero) {
  constexpr int EPC = Elem<DT>::kPer32B;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kPipeStages];
  __shared__ int s_abort;
  const int tid = threadIdx.x;
  const int64_t n_chunks = a.g.n_chunks;
  float s = 1.0f, r = 1.0f;
  bool fast = true;
  if constexpr (MODE != kUnit) {
    const float alpha = *a.amax;
    if (MODE == kTensorSupplied && (!(alpha >= 0.0f) || !is_finite_f(alpha)) && blockIdx.x == 0 &&
        tid == 0)
      flag_status(a.ws, QZ_FLAG_BAD_AMAX);
    s = __fdiv_rn(alpha, Fmt8<FMT>::kMax);
    if (s == 0.0f) s = 1.0f;
    r = __frcp_rn(s);
    fast = fast_div_ok(s);
  }
  if (a.tscale_out && blockIdx.x == 0 && tid == 0) *a.tscale_out = s;
  const uint64_t r2 = pk(r, r), ns2 = pk(-s, -s), s2 = pk(s, s), z2 = pk(zero, zero);
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
  uint32_t am = 0u;
  for (int64_t k = 0; P.has(k); ++k) {
    const int64_t tile = P.tile_of(k);
    if (!P.wait(k)) s_abort = 1;
    float tpart = 0.0f;
    const uint32_t stage = P.stage(k);
#pragma unroll
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
      uint8_t* cp = a.codes + u * EPC;
      if (!STATS || acc.T >= 1.0f)  // warp-uniform: the relative-error search is settled
        q8_chunk<FMT, DT, MODE, STATS, false, AMAX>(w, valid, cp, s, r2, ns2, s2, z2, fast, a.ws, acc, tpart, am);
      else
        q8_chunk<FMT, DT, MODE, STATS, true, AMAX>(w, valid, cp, s, r2, ns2, s2, z2, fast, a.ws, acc, tpart, am);
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
  if constexpr (MODE != kTensorComputed) {
    if constexpr (AMAX) amax_finish<QZ_F32>(am, a.amax_out, a.ws);
  }
  if constexpr (STATS) stats_finish(acc, a.ws, a.stats, static_cast<uint64_t>(a.g.rows * a.g.cols));
}

// Per-row scale with rows of at most kRowPipeMaxBytes: each row arrives in shared memory
// with one bulk copy (two rows in flight per CTA); the row amax and the codes are both
// computed from shared memory, so x is read from HBM once.
constexpr int kRowPipeMaxBytes = 64 * 1024;

template <int FMT, int DT, bool STATS>
__global__ void __launch_bounds__(kThreads) quant8_rowpipe_kernel(Q8Args a, float zero, uint32_t stage_bytes) {
  constexpr int EPC = Elem<DT>::kPer32B;
  constexpr int NP = EPC / 2;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[2];
  __shared__ float s_red[kWarps];
  __shared__ int s_abort;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const Geom& g = a.g;
  const uint32_t row_bytes = static_cast<uint32_t>(g.cols) * Elem<DT>::kBytes;
  if (a.tscale_out && blockIdx.x == 0 && tid == 0) *a.tscale_out = 1.0f;
  if (tid == 0) {
    mbar_init(smem_addr(&bars[0]), 1);
    mbar_init(smem_addr(&bars[1]), 1);
    mbar_init_fence();
    s_abort = 0;
  }
  __syncthreads();
  const uint32_t base = smem_addr(smem);
  auto issue = [&](int64_t k) {  // thread 0: row blockIdx.x + k * gridDim.x into stage k % 2
    const int64_t row = blockIdx.x + k * gridDim.x;
    if (row >= g.rows) return;
    const uint32_t st = static_cast<uint32_t>(k & 1), bar = smem_addr(&bars[st]);
    mbar_expect_tx(bar, row_bytes);
    bulk_g2s(base + st * stage_bytes, static_cast<const char*>(a.x) + row * g.ld * Elem<DT>::kBytes,
             row_bytes, bar);
  };
  if (tid == 0) {
    issue(0);
    issue(1);
  }
  const uint64_t z2 = pk(zero, zero);
  StatAcc acc;
  for (int64_t k = 0; blockIdx.x + k * gridDim.x < g.rows; ++k) {
    const int64_t row = blockIdx.x + k * gridDim.x;
    const uint32_t st = static_cast<uint32_t>(k & 1);
    if (!mbar_wait(smem_addr(&bars[st]), static_cast<uint32_t>((k >> 1) & 1), kWaitLimitNs)) s_abort = 1;
    const uint32_t rbase = base + st * stage_bytes;
    // pass 1: row amax (NaN propagates)
    float A = 0.0f;
    for (int64_t j = tid; j < g.cpr; j += kThreads) {
      uint32_t w[8];
      lds32B(w, rbase + 32u * static_cast<uint32_t>(j));
#pragma unroll
      for (int p = 0; p < NP; ++p) {
        float lo, hi;
        if constexpr (DT == QZ_BF16) {
          lo = __uint_as_float(w[p] << 16);
          hi = __uint_as_float(w[p] & 0xffff0000u);
        } else {
          lo = __uint_as_float(w[2 * p]);
          hi = __uint_as_float(w[2 * p + 1]);
        }
        A = absmax3(A, lo, hi);
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) A = absmax_nan(A, __shfl_xor_sync(kFull, A, o));
    if (lane == 0) s_red[warp] = A;
    __syncthreads();
    A = s_red[0];
#pragma unroll
    for (int i = 1; i < kWarps; ++i) A = absmax_nan(A, s_red[i]);
    float s = __fdiv_rn(A, Fmt8<FMT>::kMax);  // alpha / qmax
    if (s == 0.0f) s = 1.0f;
    const float r = __frcp_rn(s);
    const bool fast = fast_div_ok(s);
    if (tid == 0) {
      a.scales[row] = s;
      if (!is_finite_f(A)) flag_status(a.ws, QZ_FLAG_NONFINITE_INPUT);
    }
    const uint64_t r2 = pk(r, r), ns2 = pk(-s, -s), s2 = pk(s, s);
    // pass 2: codes (warp-uniform trip count: the stats vote)
    float tpart = 0.0f;
    uint32_t am_unused = 0u;
    uint8_t* crow = a.codes + row * g.cols;
    for (int64_t jb = tid & ~31; jb < g.cpr; jb += kThreads) {
      const int64_t j = jb + lane;
      const bool valid = j < g.cpr;
      uint32_t w[8];
      if (valid) {
        lds32B(w, rbase + 32u * static_cast<uint32_t>(j));
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = 0u;
      }
      if (!STATS || acc.T >= 1.0f)
        q8_chunk<FMT, DT, kTensorComputed, STATS, false>(w, valid, crow + j * EPC, s, r2, ns2, s2, z2,
                                                         fast, a.ws, acc, tpart, am_unused);
      else
        q8_chunk<FMT, DT, kTensorComputed, STATS, true>(w, valid, crow + j * EPC, s, r2, ns2, s2, z2,
                                                        fast, a.ws, acc, tpart, am_unused);
    }
    if constexpr (STATS) acc_add_sum(acc, tpart);
    __syncthreads();  // stage and s_red free again
    if (s_abort) {
      if (tid == 0) {
        flag_status(a.ws, QZ_FLAG_PIPELINE_TIMEOUT);
        for (int64_t j = k; j < k + 2; ++j)
          if (blockIdx.x + j * gridDim.x < g.rows)
            mbar_wait(smem_addr(&bars[j & 1]), static_cast<uint32_t>((j >> 1) & 1), kWaitLimitNs);
      }
      return;
    }
    if (tid == 0) issue(k + 2);
  }
  if constexpr (STATS) stats_finish(acc, a.ws, a.stats, static_cast<uint64_t>(g.rows * g.cols));
}

// Per-row scale with short rows (at most 32 * RCH chunks, full 32-byte chunks): one warp
// per row.  Each lane loads its RCH chunks of the row with 256-bit loads into registers,
// the row amax is a warp reduction (no block-wide synchronisation, so the warps of a CTA
// run their rows independently and the per-row latency overlaps across warps), and the
// codes come from the registers, so x is read once.
template <int FMT, int DT, bool STATS, int RCH>
__global__ void __launch_bounds__(kThreads) quant8_rowwarp_kernel(Q8Args a, float zero) {
  constexpr int EPC = Elem<DT>::kPer32B;
  const Geom& g = a.g;
  const int lane = threadIdx.x & 31;
  if (a.tscale_out && blockIdx.x == 0 && threadIdx.x == 0) *a.tscale_out = 1.0f;
  const uint64_t z2 = pk(zero, zero);
  StatAcc acc;
  uint32_t am_unused = 0u;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); row < g.rows;
       row += nwarps) {  // warp-uniform
    const char* xrow = static_cast<const char*>(a.x) + row * g.ld * Elem<DT>::kBytes;
    uint32_t w[RCH][8];
    float A = 0.0f;
#pragma unroll
    for (int k = 0; k < RCH; ++k) {
      const int64_t j = lane + 32 * k;
      if (j < g.cpr) {
        ld32B(w[k], xrow + j * 32);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) w[k][i] = 0u;
      }
    }
#pragma unroll
    for (int k = 0; k < RCH; ++k) {
      if constexpr (DT == QZ_BF16) {
        A = absmax_nan(A, bf16x16_absmax(w[k]));
      } else {
#pragma unroll
        for (int i = 0; i < 8; i += 2) A = absmax3(A, __uint_as_float(w[k][i]), __uint_as_float(w[k][i + 1]));
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) A = absmax_nan(A, __shfl_xor_sync(kFull, A, o));
    float s = __fdiv_rn(A, Fmt8<FMT>::kMax);  // alpha / qmax
    if (s == 0.0f) s = 1.0f;
    const float r = __frcp_rn(s);
    const bool fast = fast_div_ok(s);
    if (lane == 0) {
      a.scales[row] = s;
      if (!is_finite_f(A)) flag_status(a.ws, QZ_FLAG_NONFINITE_INPUT);
    }
    const uint64_t r2 = pk(r, r), ns2 = pk(-s, -s), s2 = pk(s, s);
    float tpart = 0.0f;
    uint8_t* crow = a.codes + row * g.cols;
#pragma unroll
    for (int k = 0; k < RCH; ++k) {
      if (32 * k < g.cpr) {  // warp-uniform
        const int64_t j = lane + 32 * k;
        if (!STATS || acc.T >= 1.0f)
          q8_chunk<FMT, DT, kTensorComputed, STATS, false, false>(w[k], j < g.cpr, crow + j * EPC, s, r2,
                                                                  ns2, s2, z2, fast, a.ws, acc, tpart,
                                                                  am_unused);
        else
          q8_chunk<FMT, DT, kTensorComputed, STATS, true, false>(w[k], j < g.cpr, crow + j * EPC, s, r2,
                                                                 ns2, s2, z2, fast, a.ws, acc, tpart,
                                                                 am_unused);
      }
    }
    if constexpr (STATS) acc_add_sum(acc, tpart);
  }
  if constexpr (STATS) stats_finish(acc, a.ws, a.stats, static_cast<uint64_t>(g.rows * g.cols));
}

// Per-row scale with the fused statistics, rows of at most kRowSlotMaxBytes: one warp per
// row and a shared-memory slot per warp.  Lane 0 brings the row in with one bulk copy (on
// the warp's own barrier), the warp takes the row amax from the slot, then quantizes the
// row chunk by chunk from the slot with the statistics -- a loop that is not unrolled, so
// the chunk code exists once per variant of the relative-error search.  Warps never wait
// for one another, so the per-row latency of one warp overlaps with the work of the rest.
constexpr int kRowSlotMaxBytes = 16 * 1024;

template <int FMT, int DT>
__global__ void __launch_bounds__(kThreads) quant8_rowslot_kernel(Q8Args a, float zero, uint32_t slot_bytes) {
  constexpr int EPC = Elem<DT>::kPer32B;
  constexpr int NP = EPC / 2;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const Geom& g = a.g;
  const uint32_t row_bytes = static_cast<uint32_t>(g.cols) * Elem<DT>::kBytes;  // whole chunks
  if (a.tscale_out && blockIdx.x == 0 && tid == 0) *a.tscale_out = 1.0f;
  const uint32_t bar = smem_addr(&bars[warp]);
  const uint32_t slot = smem_addr(smem) + static_cast<uint32_t>(warp) * slot_bytes;
  if (lane == 0) {
    mbar_init(bar, 1);
    mbar_init_fence();
  }
  __syncwarp();
  const uint64_t z2 = pk(zero, zero);
  StatAcc acc;
  uint32_t am_unused = 0u, phase = 0u;
  const int cpr = static_cast<int>(g.cpr);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + warp; row < g.rows; row += nwarps) {  // warp-uniform
    if (lane == 0) {
      mbar_expect_tx(bar, row_bytes);
      bulk_g2s(slot, static_cast<const char*>(a.x) + row * g.ld * Elem<DT>::kBytes, row_bytes, bar);
    }
    if (!__all_sync(kFull, mbar_wait(bar, phase, kWaitLimitNs))) {
      // the copy did not land within the limit: flag it, let it land (bounded), stop
      if (lane == 0) {
        flag_status(a.ws, QZ_FLAG_PIPELINE_TIMEOUT);
        mbar_wait(bar, phase, kWaitLimitNs);
      }
      __syncwarp();
      break;
    }
    phase ^= 1u;
    // pass 1: row amax (NaN propagates)
    float A = 0.0f;
#pragma unroll 1
    for (int j = lane; j < cpr; j += 32) {
      uint32_t w[8];
      lds32B(w, slot + 32u * static_cast<uint32_t>(j));
      if constexpr (DT == QZ_BF16) {
        A = absmax_nan(A, bf16x16_absmax(w));
      } else {
#pragma unroll
        for (int i = 0; i < 8; i += 2) A = absmax3(A, __uint_as_float(w[i]), __uint_as_float(w[i + 1]));
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) A = absmax_nan(A, __shfl_xor_sync(kFull, A, o));
    float s = __fdiv_rn(A, Fmt8<FMT>::kMax);  // alpha / qmax
    if (s == 0.0f) s = 1.0f;
    const float r = __frcp_rn(s);
    const bool fast = fast_div_ok(s);
    if (lane == 0) {
      a.scales[row] = s;
      if (!is_finite_f(A)) flag_status(a.ws, QZ_FLAG_NONFINITE_INPUT);
    }
    const uint64_t r2 = pk(r, r), ns2 = pk(-s, -s), s2 = pk(s, s);
    // pass 2: codes and statistics, one chunk per lane per step (warp-uniform trip count:
    // the relative-error search votes)
    float tpart = 0.0f;
    uint8_t* crow = a.codes + row * g.cols;
#pragma unroll 1
    for (int jb = 0; jb < cpr; jb += 32) {
      const int j = jb + lane;
      const bool valid = j < cpr;
      uint32_t w[8];
      if (valid) {
        lds32B(w, slot + 32u * static_cast<uint32_t>(j));
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = 0u;
      }
      if (acc.T >= 1.0f)
        q8_chunk<FMT, DT, kTensorComputed, true, false, false>(w, valid, crow + static_cast<int64_t>(j) * EPC, s,
                                                               r2, ns2, s2, z2, fast, a.ws, acc, tpart, am_unused);
      else
        q8_chunk<FMT, DT, kTensorComputed, true, true, false>(w, valid, crow + static_cast<int64_t>(j) * EPC, s,
                                                              r2, ns2, s2, z2, fast, a.ws, acc, tpart, am_unused);
    }
    acc_add_sum(acc, tpart);
    __syncwarp();  // every lane is done with the slot before the next copy refills it
  }
  (void)NP;
  stats_finish(acc, a.ws, a.stats, static_cast<uint64_t>(g.rows * g.cols));
}

// Per-row scale with the fused statistics, rows of whole 32-byte chunks whose chunk count is
// a multiple of 4 (at most kRowQuadMaxBytes): a group of four warps per row, each warp a
// quarter of it.  Each warp owns two shared-memory slots of a quarter row: lane 0 copies its
// quarter of the group's next row into one (a bulk copy on the warp's own barrier) while the
// warp works on the other, so the copies overlap the arithmetic.  The quarter amaxes meet in
// shared memory behind a named barrier of the group's 128 threads; then each warp quantizes
// its quarter with the statistics.  Rows are dealt to groups in turn, so the work is even to
// a quarter of a row per warp (with a warp per row, 4096 rows on 3648 warps left a second,
// nearly empty round paying a whole row's latency).  Every warp of a group takes the same
// rows and reaches every barrier, whatever its copies do.
constexpr int kQuadWarps = 4;
constexpr int kRowQuadMaxBytes = 48 * 1024;

template <int FMT, int DT>
__global__ void __launch_bounds__(kThreads, 3) quant8_rowquad_kernel(Q8Args a, float zero, uint32_t slot_bytes) {
  constexpr int EPC = Elem<DT>::kPer32B;
  constexpr int kGroups = kWarps / kQuadWarps;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kWarps][2];
  __shared__ float s_am[2][kWarps];  // quarter amaxes, by the parity of the row iteration
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int grp = warp / kQuadWarps, q = warp % kQuadWarps;
  const Geom& g = a.g;
  const int cpq = static_cast<int>(g.cpr) / kQuadWarps;  // chunks per quarter
  const uint32_t qbytes = static_cast<uint32_t>(cpq) * 32u;
  if (a.tscale_out && blockIdx.x == 0 && tid == 0) *a.tscale_out = 1.0f;
  const uint32_t slots = smem_addr(smem) + static_cast<uint32_t>(warp) * 2u * slot_bytes;
  const uint32_t bar0 = smem_addr(&bars[warp][0]), bar1 = smem_addr(&bars[warp][1]);
  if (lane == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar1, 1);
    mbar_init_fence();
  }
  __syncwarp();
  const int64_t step = static_cast<int64_t>(gridDim.x) * kGroups;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kGroups + grp;
  const char* xq = static_cast<const char*>(a.x) + static_cast<int64_t>(q) * cpq * 32;
  const auto issue = [&](int64_t row, int b) {  // lane 0: this warp's quarter of `row` into slot b
    const uint32_t bar = b ? bar1 : bar0;
    mbar_expect_tx(bar, qbytes);
    bulk_g2s(slots + static_cast<uint32_t>(b) * slot_bytes, xq + row * g.ld * Elem<DT>::kBytes, qbytes, bar);
  };
  if (lane == 0 && first < g.rows) issue(first, 0);
  const uint64_t z2 = pk(zero, zero);
  StatAcc acc;
  uint32_t am_unused = 0u, phase = 0u;  // bit b: parity of the next wait on slot b
  int k = 0;
  for (int64_t row = first; row < g.rows; row += step, ++k) {  // the same rows for the whole group
    const int b = k & 1;
    if (lane == 0 && row + step < g.rows) issue(row + step, b ^ 1);  // slot b ^ 1: read in iteration k - 1
    const uint32_t bar = b ? bar1 : bar0;
    if (!__all_sync(kFull, mbar_wait(bar, (phase >> b) & 1u, kWaitLimitNs))) {
      // the copy did not land within the limit: flag it and let it land (bounded); the warp
      // goes on with whatever the slot holds, so that the group's barriers stay matched
      if (lane == 0) {
        flag_status(a.ws, QZ_FLAG_PIPELINE_TIMEOUT);
        mbar_wait(bar, (phase >> b) & 1u, kWaitLimitNs);
      }
      __syncwarp();
    }
    phase ^= 1u << b;
    const uint32_t slot = slots + static_cast<uint32_t>(b) * slot_bytes;
    // pass 1: the quarter's amax (NaN propagates), then the row's from the group
    float A = 0.0f;
#pragma unroll 1
    for (int j = lane; j < cpq; j += 32) {
      uint32_t w[8];
      lds32B(w, slot + 32u * static_cast<uint32_t>(j));
      if constexpr (DT == QZ_BF16) {
        A = absmax_nan(A, bf16x16_absmax(w));
      } else {
#pragma unroll
        for (int i = 0; i < 8; i += 2) A = absmax3(A, __uint_as_float(w[i]), __uint_as_float(w[i + 1]));
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) A = absmax_nan(A, __shfl_xor_sync(kFull, A, o));
    if (lane == 0) s_am[b][warp] = A;
    asm volatile("bar.sync %0, %1;" ::"r"(1 + grp), "r"(32 * kQuadWarps) : "memory");
#pragma unroll
    for (int i = 0; i < kQuadWarps; ++i) A = absmax_nan(A, s_am[b][grp * kQuadWarps + i]);
    float s = __fdiv_rn(A, Fmt8<FMT>::kMax);  // alpha / qmax
    if (s == 0.0f) s = 1.0f;
    const float r = __frcp_rn(s);
    const bool fast = fast_div_ok(s);
    if (q == 0 && lane == 0) {
      a.scales[row] = s;
      if (!is_finite_f(A)) flag_status(a.ws, QZ_FLAG_NONFINITE_INPUT);
    }
    const uint64_t r2 = pk(r, r), ns2 = pk(-s, -s), s2 = pk(s, s);
    // pass 2: codes and statistics of the quarter, one chunk per lane per step
    float tpart = 0.0f;
    uint8_t* crow = a.codes + row * g.cols + static_cast<int64_t>(q) * cpq * EPC;
#pragma unroll 1
    for (int jb = 0; jb < cpq; jb += 32) {
      const int j = jb + lane;
      const bool valid = j < cpq;
      uint32_t w[8];
      if (valid) {
        lds32B(w, slot + 32u * static_cast<uint32_t>(j));
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i] = 0u;
      }
      if (acc.T >= 1.0f)
        q8_chunk<FMT, DT, kTensorComputed, true, false, false>(w, valid, crow + static_cast<int64_t>(j) * EPC, s,
                                                               r2, ns2, s2, z2, fast, a.ws, acc, tpart, am_unused);
      else
        q8_chunk<FMT, DT, kTensorComputed, true, true, false>(w, valid, crow + static_cast<int64_t>(j) * EPC, s,
                                                              r2, ns2, s2, z2, fast, a.ws, acc, tpart, am_unused);
    }
    acc_add_sum(acc, tpart);
    __syncwarp();  // every lane is done with the slot before it is refilled
  }
  stats_finish(acc, a.ws, a.stats, static_cast<uint64_t>(g.rows * g.cols));
}

template <typename K>
qz_status go(K kern, const Q8Args& args, int64_t work_ctas, cudaStream_t s) {
  const int grid = grid_for(reinterpret_cast<const void*>(kern), work_ctas, s);
  kern<<<grid, kThreads, 0, s>>>(args);
  return launch_status();
}

template <typename K>
qz_status go2(K kern, const Q8Args& args, int64_t work_ctas, cudaStream_t s) {  // (args, 0.0f) kernels
  const int grid = grid_for(reinterpret_cast<const void*>(kern), work_ctas, s);
  kern<<<grid, kThreads, 0, s>>>(args, 0.0f);
  return launch_status();
}

template <int FMT, int DT, bool STATS>
qz_status run_row(const Q8Args& args, cudaStream_t s) {
  const Geom& g = args.g;
  const int64_t rows = g.rows;
  const int64_t row_bytes = g.cols * Elem<DT>::kBytes;
  // short rows of whole 32-byte chunks (vector path: aligned, cols a multiple of a chunk),
  // without statistics: one warp per row, the row in registers.  (With statistics the
  // row pipeline below measured faster on the weight-like rows: 8 unrolled chunks per lane,
  // each in two variants of the relative-error search, make a large loop body.)
  if (!STATS && g.vec && g.cpr <= 256 && reinterpret_cast<uintptr_t>(args.x) % 32 == 0 &&
      (g.ld * Elem<DT>::kBytes) % 32 == 0 && g.cols % Elem<DT>::kPer32B == 0) {
    const int64_t work = (rows + kWarps - 1) / kWarps;
    if (g.cpr <= 64) return go2(&quant8_rowwarp_kernel<FMT, DT, STATS, 2>, args, work, s);
    if (g.cpr <= 128) return go2(&quant8_rowwarp_kernel<FMT, DT, STATS, 4>, args, work, s);
    return go2(&quant8_rowwarp_kernel<FMT, DT, STATS, 8>, args, work, s);
  }
  // with statistics, rows of whole chunks whose chunk count is a multiple of 4: four warps
  // per row, double-buffered quarter rows
  if (STATS && g.vec && row_bytes <= kRowQuadMaxBytes && row_bytes % (32 * kQuadWarps) == 0 &&
      reinterpret_cast<uintptr_t>(args.x) % 16 == 0 && (g.ld * Elem<DT>::kBytes) % 16 == 0) {
    auto kern = &quant8_rowquad_kernel<FMT, DT>;
    const uint32_t slot = static_cast<uint32_t>((row_bytes / kQuadWarps + 127) / 128 * 128);
    const size_t smem = static_cast<size_t>(kWarps) * 2 * slot;
    if (!set_dyn_smem(reinterpret_cast<const void*>(kern), static_cast<int>(smem))) return QZ_ERR_CUDA;
    const int grid = grid_for(reinterpret_cast<const void*>(kern), (rows + kWarps / kQuadWarps - 1) / (kWarps / kQuadWarps),
                              s, smem);
    kern<<<grid, kThreads, smem, s>>>(args, 0.0f, slot);
    return launch_status();
  }
  // with statistics, rows of whole chunks up to 16 KiB: a warp and a shared-memory slot per row
  if (STATS && g.vec && row_bytes <= kRowSlotMaxBytes && row_bytes % 32 == 0 &&
      reinterpret_cast<uintptr_t>(args.x) % 16 == 0 && (g.ld * Elem<DT>::kBytes) % 16 == 0) {
    auto kern = &quant8_rowslot_kernel<FMT, DT>;
    const uint32_t slot = static_cast<uint32_t>((row_bytes + 127) / 128 * 128);
    const size_t smem = static_cast<size_t>(kWarps) * slot;
    if (!set_dyn_smem(reinterpret_cast<const void*>(kern), static_cast<int>(smem))) return QZ_ERR_CUDA;
    const int grid = grid_for(reinterpret_cast<const void*>(kern), (rows + kWarps - 1) / kWarps, s, smem);
    kern<<<grid, kThreads, smem, s>>>(args, 0.0f, slot);
    return launch_status();
  }
  if (g.vec && row_bytes <= kRowPipeMaxBytes && reinterpret_cast<uintptr_t>(args.x) % 16 == 0 &&
      (g.ld * Elem<DT>::kBytes) % 16 == 0) {
    auto kern = &quant8_rowpipe_kernel<FMT, DT, STATS>;
    const uint32_t stage = static_cast<uint32_t>((row_bytes + 127) / 128 * 128);
    const size_t smem = 2 * static_cast<size_t>(stage);
    if (!set_dyn_smem(reinterpret_cast<const void*>(kern), static_cast<int>(smem)))
      return QZ_ERR_CUDA;
    const int grid = grid_for(reinterpret_cast<const void*>(kern), rows, s, smem);
    kern<<<grid, kThreads, smem, s>>>(args, 0.0f, stage);
    return launch_status();
  }
  if (g.vec) {
    if (g.cpr <= kThreads) return go(&quant8_row_kernel<FMT, DT, STATS, true, 1>, args, rows, s);
    if (g.cpr <= 2 * kThreads) return go(&quant8_row_kernel<FMT, DT, STATS, true, 2>, args, rows, s);
    if (g.cpr <= 4 * kThreads) return go(&quant8_row_kernel<FMT, DT, STATS, true, 4>, args, rows, s);
    if (g.cpr <= 8 * kThreads) return go(&quant8_row_kernel<FMT, DT, STATS, true, 8>, args, rows, s);
    return go(&quant8_row_kernel<FMT, DT, STATS, true, 0>, args, rows, s);
  }
  return go(&quant8_row_kernel<FMT, DT, STATS, false, 0>, args, rows, s);
}

template <int FMT, int DT, int MODE, bool STATS>
qz_status run_flat(const Q8Args& args, cudaStream_t s, bool& fused) {
  if (args.g.vec && args.g.dense && reinterpret_cast<uintptr_t>(args.x) % 16 == 0) {
    fused = MODE != kTensorComputed;
    // AMAX: also fold this tensor's amax into amax_out (the delayed-scaling call)
    auto kern = args.amax_out ? &quant8_pipe_kernel<FMT, DT, MODE, STATS, true>
                              : &quant8_pipe_kernel<FMT, DT, MODE, STATS, false>;
    if (!set_dyn_smem(reinterpret_cast<const void*>(kern), static_cast<int>(kPipeSmem)))
      return QZ_ERR_CUDA;
    const int grid = grid_for(reinterpret_cast<const void*>(kern),
                              (args.g.n_chunks + kPipeTileChunks - 1) / kPipeTileChunks, s, kPipeSmem);
    kern<<<grid, kThreads, kPipeSmem, s>>>(args, 0.0f);
    return launch_status();
  }
  const int64_t per_cta = static_cast<int64_t>(kThreads) * kUnroll;
  const int64_t work = (args.g.n_chunks + per_cta - 1) / per_cta;
  if (args.g.vec) return go(&quant8_kernel<FMT, DT, MODE, STATS, true>, args, work, s);
  return go(&quant8_kernel<FMT, DT, MODE, STATS, false>, args, work, s);
}

template <int FMT, int DT>
qz_status dispatch(const Q8Args& args, int gran, bool supplied, bool stats, cudaStream_t s, bool& f) {
  if (gran == QZ_GRAN_ROW) return stats ? run_row<FMT, DT, true>(args, s) : run_row<FMT, DT, false>(args, s);
  if (gran == QZ_GRAN_UNIT)
    return stats ? run_flat<FMT, DT, kUnit, true>(args, s, f) : run_flat<FMT, DT, kUnit, false>(args, s, f);
  if (supplied)
    return stats ? run_flat<FMT, DT, kTensorSupplied, true>(args, s, f)
                 : run_flat<FMT, DT, kTensorSupplied, false>(args, s, f);
  return stats ? run_flat<FMT, DT, kTensorComputed, true>(args, s, f)
               : run_flat<FMT, DT, kTensorComputed, false>(args, s, f);
}

template <int FMT>
qz_status dispatch_dt(const qz_desc& d, const Q8Args& args, bool supplied, bool stats, cudaStream_t s,
                      bool& f) {
  return d.in_dtype == QZ_BF16 ? dispatch<FMT, QZ_BF16>(args, d.granularity, supplied, stats, s, f)
                               : dispatch<FMT, QZ_F32>(args, d.granularity, supplied, stats, s, f);
}

}  // namespace

qz_status launch_quant8(const qz_desc& d, const void* x, void* codes, void* scales,
                        float* tscale_out, const float* amax, bool amax_supplied,
                        qz_stats* stats, void* ws, cudaStream_t s, float* amax_out) {
  const int eb = d.in_dtype == QZ_BF16 ? 2 : 4;
  Q8Args args;
  args.x = x;
  args.g = make_geom(d, x, eb, 32);
  // the vector path stores EPC code bytes per chunk at row * cols + col
  if (reinterpret_cast<uintptr_t>(codes) % 16 != 0) {
    args.g.vec = false;
    args.g.dense = false;
  }
  args.codes = static_cast<uint8_t*>(codes);
  args.scales = static_cast<float*>(scales);
  args.amax = amax;
  args.tscale_out = tscale_out;
  args.stats = stats;
  args.ws = ws;
  args.amax_out = amax_out;
  const bool st = stats != nullptr;
  bool fused = false;
  qz_status rc;
  switch (d.format) {
    case QZ_INT8: rc = dispatch_dt<QZ_INT8>(d, args, amax_supplied, st, s, fused); break;
    case QZ_FP8_E4M3: rc = dispatch_dt<QZ_FP8_E4M3>(d, args, amax_supplied, st, s, fused); break;
    default: rc = dispatch_dt<QZ_FP8_E5M2>(d, args, amax_supplied, st, s, fused); break;
  }
  if (rc == QZ_OK && amax_out && !fused) rc = launch_amax(d, x, amax_out, ws, s);
  return rc;
}

}  // namespace qz
