// qz_stats.cu -- error statistics of existing codes against x (the error measures of the
// blog post "浅谈低精度浮点数": |x - x^| and |x - x^| / |x|, here reduced to the sum of
// squares / MSE, the largest absolute and the largest relative error).
//
// Reads x and the codes (+ scales) once; x^ is rebuilt exactly as the dequantize kernels
// build it, and the reduction is the same one the fused quantize path uses.
#include "qz_device.cuh"
#include "qz_internal.h"

namespace qz {
namespace {

struct StArgs {
  const void* x;
  Geom g;  // over x
  const uint8_t* codes;
  const void* scales;
  const float* tscale;
  qz_stats* stats;
  void* ws;
};

template <int DT, bool VEC>
__device__ __forceinline__ void load_x_chunk(uint32_t (&w)[8], const void* x, const Geom& g,
                                             int64_t row, int64_t col, int64_t nv) {
  const int64_t e0 = row * g.ld + col;
  if constexpr (VEC) {
    ld32B(w, static_cast<const char*>(x) + e0 * Elem<DT>::kBytes);
  } else {
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
  }
}

// FMT: any format; GRAN: QZ_GRAN_TENSOR / ROW / UNIT for INT8 / FP8, BLOCK / UNIT for FP4.
template <int FMT, int DT, int GRAN, bool VEC>
__global__ void __launch_bounds__(kThreads) stats_kernel(StArgs a) {
  constexpr int EPC = Elem<DT>::kPer32B;
  constexpr bool FP4 = FMT == QZ_MXFP4 || FMT == QZ_NVFP4;
  constexpr int BS = FMT == QZ_MXFP4 ? 32 : 16;
  const Geom& g = a.g;
  const int lane = threadIdx.x & 31;
  float st = 1.0f;
  if constexpr ((FMT == QZ_NVFP4 && GRAN == QZ_GRAN_BLOCK) || (!FP4 && GRAN == QZ_GRAN_TENSOR)) st = *a.tscale;
  StatAcc acc;
  const int64_t warp_id = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarps * 32;
  for (int64_t base = warp_id * 32; base < g.n_chunks; base += stride) {  // warp-uniform trip
    const int64_t u = base + lane;
    const bool valid = u < g.n_chunks;
    int64_t row = 0, col = 0;
    if (g.dense) {
      col = u * EPC;
    } else {
      row = u / g.cpr;
      col = (u - row * g.cpr) * EPC;
    }
    const int64_t nv = valid ? (g.dense ? EPC : g.cols - col) : 0;
    uint32_t w[8];
    if (valid) {
      load_x_chunk<DT, VEC>(w, a.x, g, row, col, nv);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = 0u;
    }
    float xs[EPC], xh[EPC];
#pragma unroll
    for (int i = 0; i < EPC; ++i) xs[i] = chunk_elem<DT>(w, i);
    if (valid) {
      float A = 0.0f;
#pragma unroll
      for (int i = 0; i < EPC; ++i) A = absmax_nan(A, xs[i]);
      if (!is_finite_f(A)) flag_status(a.ws, QZ_FLAG_NONFINITE_INPUT);
    }
    if constexpr (FP4) {
      // codes: EPC/2 bytes of this chunk; scale: one byte per block
      float s = 0.0f;
      uint32_t cw[2] = {0u, 0u};
      if (valid) {
        const int64_t cofs = g.dense ? col / 2 : row * (g.cols / 2) + col / 2;
        const int64_t sofs = g.dense ? col / BS : row * (g.cols / BS) + col / BS;
#pragma unroll
        for (int j = 0; j < EPC / 2; ++j) cw[j / 4] |= static_cast<uint32_t>(a.codes[cofs + j]) << (8 * (j % 4));
        if constexpr (FMT == QZ_MXFP4) {
          const uint32_t c = GRAN == QZ_GRAN_UNIT ? 127u : static_cast<const uint8_t*>(a.scales)[sofs];
          s = c == 255u ? __uint_as_float(0x7fc00000u) : exp2_pos(static_cast<int>(c) - 127);
        } else {
          s = GRAN == QZ_GRAN_UNIT ? 1.0f : __fmul_rn(st, dec_e4m3(static_cast<const uint8_t*>(a.scales)[sofs]));
        }
      }
#pragma unroll
      for (int j = 0; j < EPC / 2; ++j) {
        float q0, q1;
        dec_e2m1x2((cw[j / 4] >> (8 * (j % 4))) & 0xffu, q0, q1);
        xh[2 * j] = __fmul_rn(q0, s);
        xh[2 * j + 1] = __fmul_rn(q1, s);
      }
    } else {
      float s = st;
      uint32_t cw[EPC / 4];
#pragma unroll
      for (int j = 0; j < EPC / 4; ++j) cw[j] = 0u;
      if (valid) {
        const uint8_t* cp = a.codes + (g.dense ? col : row * g.cols + col);
#pragma unroll
        for (int j = 0; j < EPC; ++j)
          if (j < nv) cw[j / 4] |= static_cast<uint32_t>(cp[j]) << (8 * (j % 4));
        if constexpr (GRAN == QZ_GRAN_ROW) s = static_cast<const float*>(a.scales)[g.dense ? col / g.cols : row];
      }
#pragma unroll
      for (int j = 0; j < EPC / 2; ++j) {
        float q0, q1;
        dec8x2<FMT>((cw[j / 2] >> (16 * (j % 2))) & 0xffffu, q0, q1);
        xh[2 * j] = __fmul_rn(q0, s);
        xh[2 * j + 1] = __fmul_rn(q1, s);
      }
      // lanes or elements without data: x = 0 and code 0 give x^ = 0 * s = 0 -> e = 0
    }
    acc_chunk(acc, xs, xh);
  }
  stats_finish(acc, a.ws, a.stats, static_cast<uint64_t>(g.rows * g.cols));
}

template <int FMT, int DT, int GRAN>
qz_status go(const StArgs& a, cudaStream_t s) {
  const void* k = a.g.vec ? reinterpret_cast<const void*>(&stats_kernel<FMT, DT, GRAN, true>)
                          : reinterpret_cast<const void*>(&stats_kernel<FMT, DT, GRAN, false>);
  const int grid = grid_for(k, (a.g.n_chunks + kThreads - 1) / kThreads, s);
  if (a.g.vec) stats_kernel<FMT, DT, GRAN, true><<<grid, kThreads, 0, s>>>(a);
  else stats_kernel<FMT, DT, GRAN, false><<<grid, kThreads, 0, s>>>(a);
  return launch_status();
}

template <int FMT, int DT>
qz_status by_gran(const StArgs& a, int gran, cudaStream_t s) {
  if constexpr (FMT == QZ_MXFP4 || FMT == QZ_NVFP4) {
    return gran == QZ_GRAN_UNIT ? go<FMT, DT, QZ_GRAN_UNIT>(a, s) : go<FMT, DT, QZ_GRAN_BLOCK>(a, s);
  } else {
    if (gran == QZ_GRAN_TENSOR) return go<FMT, DT, QZ_GRAN_TENSOR>(a, s);
    if (gran == QZ_GRAN_ROW) return go<FMT, DT, QZ_GRAN_ROW>(a, s);
    return go<FMT, DT, QZ_GRAN_UNIT>(a, s);
  }
}

template <int FMT>
qz_status by_dt(const qz_desc& d, const StArgs& a, cudaStream_t s) {
  return d.in_dtype == QZ_BF16 ? by_gran<FMT, QZ_BF16>(a, d.granularity, s) : by_gran<FMT, QZ_F32>(a, d.granularity, s);
}

qz_status launch(const qz_desc& d, const void* x, const void* codes, const void* scales,
                 const float* tscale, qz_stats* stats, void* ws, cudaStream_t s) {
  StArgs a;
  a.x = x;
  a.g = make_geom(d, x, d.in_dtype == QZ_BF16 ? 2 : 4, 32);
  a.codes = static_cast<const uint8_t*>(codes);
  a.scales = scales;
  a.tscale = tscale;
  a.stats = stats;
  a.ws = ws;
  switch (d.format) {
    case QZ_INT8: return by_dt<QZ_INT8>(d, a, s);
    case QZ_FP8_E4M3: return by_dt<QZ_FP8_E4M3>(d, a, s);
    case QZ_FP8_E5M2: return by_dt<QZ_FP8_E5M2>(d, a, s);
    case QZ_MXFP4: return by_dt<QZ_MXFP4>(d, a, s);
    default: return by_dt<QZ_NVFP4>(d, a, s);
  }
}

// One CTA folds `count` statistics records of disjoint parts of a tensor: sums of squares
// and element counts add (fp64, fixed order: thread t takes records t, t + 256, ..., then
// the warp and CTA folds in lane and warp order, so a given count always sums alike), the
// largest errors take their maximum.  Every record is read before thread 0 writes `out`,
// so `out` may be one of the parts.
__global__ void __launch_bounds__(kThreads) stats_merge_kernel(const qz_stats* parts, int64_t count,
                                                               qz_stats* out) {
  __shared__ double s_sum[kWarps];
  __shared__ unsigned long long s_n[kWarps];
  __shared__ float s_abs[kWarps], s_rel[kWarps];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double t = 0.0;
  unsigned long long n = 0;
  float ma = 0.0f, mr = 0.0f;
  for (int64_t i = threadIdx.x; i < count; i += kThreads) {
    t += parts[i].sum_sq_err;
    n += parts[i].n;
    ma = fmaxf(ma, parts[i].max_abs_err);
    mr = fmaxf(mr, parts[i].max_rel_err);
  }
  t = warp_sum(t);
  ma = warp_max(ma);
  mr = warp_max(mr);
#pragma unroll
  for (int o = 16; o; o >>= 1) n += __shfl_xor_sync(kFull, n, o);
  if (lane == 0) {
    s_sum[warp] = t;
    s_n[warp] = n;
    s_abs[warp] = ma;
    s_rel[warp] = mr;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double tot = 0.0;
    unsigned long long nt = 0;
    for (int w = 0; w < kWarps; ++w) {
      tot += s_sum[w];
      nt += s_n[w];
      ma = fmaxf(ma, s_abs[w]);
      mr = fmaxf(mr, s_rel[w]);
    }
    out->sum_sq_err = tot;
    out->mse = nt ? tot / static_cast<double>(nt) : 0.0;
    out->max_abs_err = ma;
    out->max_rel_err = mr;
    out->n = nt;
  }
}

}  // namespace

qz_status launch_stats_merge(const qz_stats* parts, int64_t count, qz_stats* out, cudaStream_t s) {
  stats_merge_kernel<<<1, kThreads, 0, s>>>(parts, count, out);
  return launch_status();
}

qz_status launch_stats8(const qz_desc& d, const void* x, const void* codes, const void* scales,
                        const float* tscale, qz_stats* stats, void* ws, cudaStream_t s) {
  return launch(d, x, codes, scales, tscale, stats, ws, s);
}
qz_status launch_stats4(const qz_desc& d, const void* x, const void* codes, const void* scales,
                        const float* tscale, qz_stats* stats, void* ws, cudaStream_t s) {
  return launch(d, x, codes, scales, tscale, stats, ws, s);
}

}  // namespace qz
