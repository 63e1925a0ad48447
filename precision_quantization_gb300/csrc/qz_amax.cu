// qz_amax.cu -- largest |x| of a tensor: the alpha of the per-tensor INT8 / FP8 scale and
// the global amax of NVFP4's fp32 tensor scale (blog post "浅谈低精度浮点数", sections "FP8"
// and "FP4 / MXFP4 / NVFP4").
//
// One streaming read of x.  The maximum is taken on the magnitude bits as unsigned
// integers, which orders finite values like floats and puts Inf and NaN above every finite
// value, so a single comparison at the end detects non-finite input.
#include "qz_device.cuh"
#include "qz_internal.h"
#include "qz_pipe.cuh"

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
  amax_finish<DT>(m, out, ws);
}

// Dense tensors: x streamed through shared memory by 1-D bulk copies (32 KiB tiles, two
// in flight per CTA), so the read runs at the copy engine's pace whatever the occupancy.
constexpr int kAmaxStages = kPipeStages;
constexpr int kAmaxCPT = kPipeCPT;
constexpr int kAmaxTileChunks = kThreads * kAmaxCPT;
constexpr int kAmaxTileBytes = kAmaxTileChunks * 32;
constexpr size_t kAmaxSmem = static_cast<size_t>(kAmaxStages) * kAmaxTileBytes;

template <int DT>
__global__ void __launch_bounds__(kThreads)
amax_pipe_kernel(const void* __restrict__ x, int64_t n_chunks, float* __restrict__ out, void* ws) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kAmaxStages];
  __shared__ int s_abort;
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int i = 0; i < kAmaxStages; ++i) mbar_init(smem_addr(&bars[i]), 1);
    mbar_init_fence();
    s_abort = 0;
  }
  __syncthreads();
  const BulkPipe<kAmaxStages, kAmaxTileBytes> P{smem_addr(smem), smem_addr(&bars[0]),
                                                static_cast<const char*>(x), n_chunks * 32,
                                                (n_chunks + kAmaxTileChunks - 1) / kAmaxTileChunks,
                                                false};
  if (tid == 0) P.prologue();
  uint32_t m = 0;
  for (int64_t k = 0; P.has(k); ++k) {
    const int64_t tile = P.tile_of(k);
    if (!P.wait(k)) s_abort = 1;
    const uint32_t stage = P.stage(k);
#pragma unroll
    for (int c = 0; c < kAmaxCPT; ++c) {
      const int j = c * kThreads + tid;
      if (tile * kAmaxTileChunks + j < n_chunks) {
        uint32_t w[8];
        lds32B(w, stage + 32u * j);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if constexpr (DT == QZ_BF16) m = __vmaxu2(m, w[i] & 0x7fff7fffu);
          else m = max(m, w[i] & 0x7fffffffu);
        }
      }
    }
    __syncthreads();
    if (s_abort) {
      if (tid == 0) {
        flag_status(ws, QZ_FLAG_PIPELINE_TIMEOUT);
        P.drain(k);
      }
      return;
    }
    if (tid == 0) P.issue(k + kAmaxStages);
  }
  amax_finish<DT>(m, out, ws);
}

template <int DT>
qz_status run(const qz_desc& d, const void* x, float* out, void* ws, cudaStream_t s) {
  const Geom g = make_geom(d, x, Elem<DT>::kBytes, 32);
  if (g.vec && g.dense) {
    auto kern = &amax_pipe_kernel<DT>;
    if (!set_dyn_smem(reinterpret_cast<const void*>(kern), static_cast<int>(kAmaxSmem)))
      return QZ_ERR_CUDA;
    const int grid = grid_for(reinterpret_cast<const void*>(kern),
                              (g.n_chunks + kAmaxTileChunks - 1) / kAmaxTileChunks, s, kAmaxSmem);
    kern<<<grid, kThreads, kAmaxSmem, s>>>(x, g.n_chunks, out, ws);
    return launch_status();
  }
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
