// qz_amax.cu -- largest |x| of a tensor: the alpha of the per-tensor INT8 / FP8 scale and
// the global amax of NVFP4's fp32 tensor scale (blog post "浅谈低精度浮点数", sections "FP8"
// and "FP4 / MXFP4 / NVFP4").
//
// One streaming read of x.  The maximum is taken on the magnitude bits as unsigned
// integers, which orders finite values like floats and puts Inf and NaN above every finite
// value, so a single comparison at the end detects non-finite input.
#include "qz_device.cuh"
#include "qz_internal.h"

namespace qz {
namespace {

constexpr int kUnroll = 4;

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads)
amax_kernel(const void* __restrict__ x, Geom g, float* __restrict__ out, void* ws) {
  constexpr int EPC = Elem<DT>::kPer32B;
  uint32_t m = 0;  // bf16: two 16-bit maxima side by side; fp32: one
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t nthr = static_cast<int64_t>(gridDim.x) * kThreads;
  if constexpr (VEC) {
    for (int64_t base = tid; base < g.n_chunks; base += nthr * kUnroll) {
      uint32_t w[kUnroll][8];
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        const int64_t u = base + k * nthr;
        if (u < g.n_chunks) {
          const char* p;
          if (g.dense) {
            p = static_cast<const char*>(x) + u * 32;
          } else {
            const int64_t r = u / g.cpr, j = u - r * g.cpr;
            p = static_cast<const char*>(x) + (r * g.ld + j * EPC) * Elem<DT>::kBytes;
          }
          ld32B(w[k], p);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) w[k][i] = 0u;
        }
      }
#pragma unroll
      for (int k = 0; k < kUnroll; ++k)
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if constexpr (DT == QZ_BF16) m = __vmaxu2(m, w[k][i] & 0x7fff7fffu);
          else m = max(m, w[k][i] & 0x7fffffffu);
        }
    }
  } else {
    const int64_t n = g.rows * g.cols;
    for (int64_t i = tid; i < n; i += nthr) {
      const int64_t r = i / g.cols, c = i - r * g.cols;
      const uint32_t b = __float_as_uint(load_elem<DT>(x, r * g.ld + c)) & 0x7fffffffu;
      if constexpr (DT == QZ_BF16) m = __vmaxu2(m, b >> 16);
      else m = max(m, b);
    }
  }
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

template <int DT>
qz_status run(const qz_desc& d, const void* x, float* out, void* ws, cudaStream_t s) {
  const Geom g = make_geom(d, x, Elem<DT>::kBytes, 32);
  if (g.vec) {
    const void* k = reinterpret_cast<const void*>(&amax_kernel<DT, true>);
    const int grid = grid_for(k, (g.n_chunks + kThreads * kUnroll - 1) / (kThreads * kUnroll), s);
    amax_kernel<DT, true><<<grid, kThreads, 0, s>>>(x, g, out, ws);
  } else {
    const void* k = reinterpret_cast<const void*>(&amax_kernel<DT, false>);
    const int grid = grid_for(k, (g.rows * g.cols + kThreads - 1) / kThreads, s);
    amax_kernel<DT, false><<<grid, kThreads, 0, s>>>(x, g, out, ws);
  }
  return launch_status();
}

}  // namespace

qz_status launch_amax(const qz_desc& d, const void* x, float* out, void* ws, cudaStream_t s) {
  if (out == nullptr) out = &static_cast<WsHeader*>(ws)->amax;
  return d.in_dtype == QZ_BF16 ? run<QZ_BF16>(d, x, out, ws, s) : run<QZ_F32>(d, x, out, ws, s);
}

}  // namespace qz
