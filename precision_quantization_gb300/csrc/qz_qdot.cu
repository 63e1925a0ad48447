// qz_qdot.cu -- the quantized matrix product of the blog's "Puzzles 12 Quantized Matrix Mult"
// (section of its "Triton" post): z[j][k] = sum_l sc[j][l/g] (w[j][l] - sh[j][l/g]) y[l][k],
// with 4-bit weights w packed 8 per 32-bit word (low nibble first), one fp32 scale and one
// 4-bit shift per group of g weights along l, and bf16 activations y.
//
// For a few activation columns (n1 <= 8: decoding, small batches) the product streams the
// packed weights once and does 2 * n1 flops per 4-bit weight, so it runs on the FMA pipe
// without tensor cores: a warp takes a block of weight rows, its lanes the rows' 32-bit
// code words (coalesced 128-byte reads), the weights are dequantized in registers exactly
// as qz_dequantize_asym4 does (fl32(sc * (w - sh))), accumulation is fp32 by paired FMA,
// and a shuffle reduction across the warp finishes each output.
#include <algorithm>

#include "qz_device.cuh"
#include "qz_internal.h"
#include "qz_pipe.cuh"

namespace qz {
namespace {

constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23: 0x4B400000 + d is the float d + kMagic

struct QdArgs {
  const uint32_t* w;
  const float* scales;
  const uint32_t* shifts;
  const uint16_t* y;  // bf16 bits [mid, ld_y]
  float* z;
  int64_t n0, mid, group, ld_y, ld_z;
  int64_t ksplit;     // slices of the code words per row (> 1: z zeroed, partial sums added)
  int64_t wps;        // code words per slice, a multiple of 32
};

__device__ __forceinline__ float bf16_value(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

// x + 1.5 * 2^23 read back as a float minus 1.5 * 2^23: the small integer d, exactly
__device__ __forceinline__ float small_int(uint32_t d) {
  return __fsub_rn(__uint_as_float(0x4B400000u + d), kMagic);
}

// A warp takes R weight rows at once (R even) and one slice of their code words: the
// activations of each l are loaded and widened once for the R rows, the dequantized
// weights of rows (2p, 2p+1) form an fp32 pair, and every FMA is a paired one
// (fma.rn.f32x2) over two rows of one column k.  With several slices per row (rows too
// few to fill the GPU) the warps add their partial sums into the zeroed z.
template <int N1, int R>
__global__ void __launch_bounds__(kThreads) quant_dot_kernel(QdArgs a, bool yvec) {
  static_assert(R % 2 == 0, "rows are paired");
  constexpr int P = R / 2;
  const int lane = threadIdx.x & 31;
  const int64_t wpr = a.mid / 8;            // code words per weight row
  const int64_t ng = a.mid / a.group;       // groups per row
  const int64_t sw = (ng + 7) / 8;          // shift words per row
  const bool g8 = a.group % 8 == 0;         // a code word lies in one group
  const int64_t warp = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
  const int64_t nblocks = (a.n0 + R - 1) / R;
  for (int64_t item = warp; item < nblocks * a.ksplit; item += nwarps) {
    const int64_t r0 = (item / a.ksplit) * R;
    const int64_t w_begin = (item % a.ksplit) * a.wps;
    const int64_t w_end = min(w_begin + a.wps, wpr);
    int64_t row[R];
#pragma unroll
    for (int i = 0; i < R; ++i) row[i] = min(r0 + i, a.n0 - 1);  // rows past the end: repeat the last
    uint64_t acc[P][N1];
#pragma unroll
    for (int p = 0; p < P; ++p)
#pragma unroll
      for (int k = 0; k < N1; ++k) acc[p][k] = pk(0.0f, 0.0f);
    for (int64_t wi = w_begin + lane; wi < w_end; wi += 32) {
      const int64_t l0 = wi * 8;
      uint32_t word[R];
#pragma unroll
      for (int i = 0; i < R; ++i) word[i] = __ldg(a.w + row[i] * wpr + wi);
      float sc[R];
      uint32_t sh[R];
      if (g8) {
        const int64_t g = l0 / a.group;
#pragma unroll
        for (int i = 0; i < R; ++i) {
          sc[i] = __ldg(a.scales + row[i] * ng + g);
          sh[i] = (__ldg(a.shifts + row[i] * sw + g / 8) >> (4 * (g % 8))) & 0xFu;
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (!g8) {
          const int64_t g = (l0 + e) / a.group;
#pragma unroll
          for (int i = 0; i < R; ++i) {
            sc[i] = __ldg(a.scales + row[i] * ng + g);
            sh[i] = (__ldg(a.shifts + row[i] * sw + g / 8) >> (4 * (g % 8))) & 0xFu;
          }
        }
        // activations y[l0 + e][0 .. N1), widened to fp32
        float yv[N1];
        const uint16_t* yr = a.y + (l0 + e) * a.ld_y;
        if (N1 == 8 && yvec) {
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(yr));
          const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int k = 0; k < N1 / 2; ++k) {
            yv[2 * k] = __uint_as_float(u[k] << 16);
            yv[2 * k + 1] = __uint_as_float(u[k] & 0xffff0000u);
          }
        } else {
#pragma unroll
          for (int k = 0; k < N1; ++k) yv[k] = bf16_value(__ldg(yr + k));
        }
#pragma unroll
        for (int p = 0; p < P; ++p) {
          // fl32(sc * (w - sh)) of rows 2p and 2p+1, element e
          const uint32_t da = ((word[2 * p] >> (4 * e)) & 0xFu) - sh[2 * p];
          const uint32_t db = ((word[2 * p + 1] >> (4 * e)) & 0xFu) - sh[2 * p + 1];
          const uint64_t deq = mul2(pk(sc[2 * p], sc[2 * p + 1]), pk(small_int(da), small_int(db)));
#pragma unroll
          for (int k = 0; k < N1; ++k) acc[p][k] = fma2(deq, pk(yv[k], yv[k]), acc[p][k]);
        }
      }
    }
    // warp sums; lane 0 writes the rows that exist
#pragma unroll
    for (int p = 0; p < P; ++p) {
#pragma unroll
      for (int k = 0; k < N1; ++k) {
        float lo, hi;
        upk(acc[p][k], lo, hi);
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          lo = __fadd_rn(lo, __shfl_xor_sync(kFull, lo, o));
          hi = __fadd_rn(hi, __shfl_xor_sync(kFull, hi, o));
        }
        if (lane == 0) {
          float* za = a.z + (r0 + 2 * p) * a.ld_z + k;
          if (a.ksplit > 1) {
            if (r0 + 2 * p < a.n0) atomicAdd(za, lo);
            if (r0 + 2 * p + 1 < a.n0) atomicAdd(za + a.ld_z, hi);
          } else {
            if (r0 + 2 * p < a.n0) *za = lo;
            if (r0 + 2 * p + 1 < a.n0) za[a.ld_z] = hi;
          }
        }
      }
    }
  }
}

template <int N1>
qz_status run(QdArgs a, bool yvec, cudaStream_t s) {
  constexpr int R = N1 <= 2 ? 8 : 4;  // rows per warp: more for few columns
  auto k = &quant_dot_kernel<N1, R>;
  // enough (row block, slice) items for every SM to hold several warps busy
  const int64_t wpr = a.mid / 8, nblocks = (a.n0 + R - 1) / R;
  const int64_t want = static_cast<int64_t>(sm_count()) * 4 * kWarps;
  int64_t ks = nblocks >= want ? 1 : (want + nblocks - 1) / nblocks;
  ks = std::max<int64_t>(1, std::min<int64_t>(ks, wpr / 32));
  a.wps = ((wpr + ks - 1) / ks + 31) / 32 * 32;
  a.ksplit = (wpr + a.wps - 1) / a.wps;
  if (a.ksplit > 1 &&
      cudaMemset2DAsync(a.z, static_cast<size_t>(a.ld_z) * 4, 0, static_cast<size_t>(N1) * 4,
                        static_cast<size_t>(a.n0), s) != cudaSuccess)
    return QZ_ERR_CUDA;
  const int grid = grid_for(reinterpret_cast<const void*>(k),
                            (nblocks * a.ksplit + kWarps - 1) / kWarps, s);
  k<<<grid, kThreads, 0, s>>>(a, yvec);
  return launch_status();
}

}  // namespace

qz_status launch_quant_dot(const uint32_t* w, const float* scales, const uint32_t* shifts,
                           int64_t n0, int64_t mid, int64_t group, const void* y, int64_t ld_y,
                           int64_t n1, float* z, int64_t ld_z, cudaStream_t s) {
  const QdArgs a{w, scales, shifts, static_cast<const uint16_t*>(y), z, n0, mid, group, ld_y, ld_z, 1, 0};
  const bool yvec = reinterpret_cast<uintptr_t>(y) % 16 == 0 && ld_y % 8 == 0;
  switch (n1) {
    case 1: return run<1>(a, yvec, s);
    case 2: return run<2>(a, yvec, s);
    case 3: return run<3>(a, yvec, s);
    case 4: return run<4>(a, yvec, s);
    case 5: return run<5>(a, yvec, s);
    case 6: return run<6>(a, yvec, s);
    case 7: return run<7>(a, yvec, s);
    default: return run<8>(a, yvec, s);
  }
}

}  // namespace qz
