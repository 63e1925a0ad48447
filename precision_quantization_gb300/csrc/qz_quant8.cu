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
        if constexpr (MODE == kTensorSupplied) f = f && (__fmul_rn(A, r) <= 0x1p100f);
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

template <typename K>
qz_status go(K kern, const Q8Args& args, int64_t work_ctas, cudaStream_t s) {
  const int grid = grid_for(reinterpret_cast<const void*>(kern), work_ctas, s);
  kern<<<grid, kThreads, 0, s>>>(args);
  return launch_status();
}

template <int FMT, int DT, bool STATS>
qz_status run_row(const Q8Args& args, cudaStream_t s) {
  const Geom& g = args.g;
  const int64_t rows = g.rows;
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
qz_status run_flat(const Q8Args& args, cudaStream_t s) {
  const int64_t per_cta = static_cast<int64_t>(kThreads) * kUnroll;
  const int64_t work = (args.g.n_chunks + per_cta - 1) / per_cta;
  if (args.g.vec) return go(&quant8_kernel<FMT, DT, MODE, STATS, true>, args, work, s);
  return go(&quant8_kernel<FMT, DT, MODE, STATS, false>, args, work, s);
}

template <int FMT, int DT>
qz_status dispatch(const Q8Args& args, int gran, bool supplied, bool stats, cudaStream_t s) {
  if (gran == QZ_GRAN_ROW) return stats ? run_row<FMT, DT, true>(args, s) : run_row<FMT, DT, false>(args, s);
  if (gran == QZ_GRAN_UNIT)
    return stats ? run_flat<FMT, DT, kUnit, true>(args, s) : run_flat<FMT, DT, kUnit, false>(args, s);
  if (supplied)
    return stats ? run_flat<FMT, DT, kTensorSupplied, true>(args, s)
                 : run_flat<FMT, DT, kTensorSupplied, false>(args, s);
  return stats ? run_flat<FMT, DT, kTensorComputed, true>(args, s)
               : run_flat<FMT, DT, kTensorComputed, false>(args, s);
}

template <int FMT>
qz_status dispatch_dt(const qz_desc& d, const Q8Args& args, bool supplied, bool stats, cudaStream_t s) {
  return d.in_dtype == QZ_BF16 ? dispatch<FMT, QZ_BF16>(args, d.granularity, supplied, stats, s)
                               : dispatch<FMT, QZ_F32>(args, d.granularity, supplied, stats, s);
}

}  // namespace

qz_status launch_quant8(const qz_desc& d, const void* x, void* codes, void* scales,
                        float* tscale_out, const float* amax, bool amax_supplied,
                        qz_stats* stats, void* ws, cudaStream_t s) {
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
  const bool st = stats != nullptr;
  switch (d.format) {
    case QZ_INT8: return dispatch_dt<QZ_INT8>(d, args, amax_supplied, st, s);
    case QZ_FP8_E4M3: return dispatch_dt<QZ_FP8_E4M3>(d, args, amax_supplied, st, s);
    default: return dispatch_dt<QZ_FP8_E5M2>(d, args, amax_supplied, st, s);
  }
}

}  // namespace qz
