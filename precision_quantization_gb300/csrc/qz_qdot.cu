// qz_qdot.cu -- the quantized matrix product of the blog's "Puzzles 12 Quantized Matrix Mult"
// (section of its "Triton" post): z[j][k] = sum_l sc[j][l/g] (w[j][l] - sh[j][l/g]) y[l][k],
// with 4-bit weights w packed 8 per 32-bit word (low nibble first), one fp32 scale and one
// 4-bit shift per group of g weights along l, and bf16 activations y.
//
// For a few activation columns (n1 <= 8: decoding, small batches) the product streams the
// packed weights once and does 2 * n1 flops per 4-bit weight: it is bound by HBM, not by
// arithmetic, so it runs on the FMA pipe without tensor cores -- a warp per weight row,
// lanes over the row's 32-bit code words (coalesced 128-byte reads), the weights
// dequantized in registers exactly as qz_dequantize_asym4 does (fl32(sc * (w - sh))),
// fp32 accumulation by FMA, a shuffle reduction across the warp.
#include "qz_device.cuh"
#include "qz_internal.h"

namespace qz {
namespace {

constexpr int kWordsInFlight = 4;  // code words per lane per iteration
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23: 0x4B400000 + d is the float d + kMagic

struct QdArgs {
  const uint32_t* w;
  const float* scales;
  const uint32_t* shifts;
  const uint16_t* y;  // bf16 bits [mid, ld_y]
  float* z;
  int64_t n0, mid, group, ld_y, ld_z;
};

__device__ __forceinline__ float bf16_value(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

template <int N1>
__global__ void __launch_bounds__(kThreads) quant_dot_kernel(QdArgs a, bool yvec) {
  const int lane = threadIdx.x & 31;
  const int64_t wpr = a.mid / 8;            // code words per weight row
  const int64_t ng = a.mid / a.group;       // groups per row
  const int64_t sw = (ng + 7) / 8;          // shift words per row
  const bool g8 = a.group % 8 == 0;         // a code word lies in one group
  const int64_t warp = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
  for (int64_t j = warp; j < a.n0; j += nwarps) {
    const uint32_t* wr = a.w + j * wpr;
    float acc[N1];
#pragma unroll
    for (int k = 0; k < N1; ++k) acc[k] = 0.0f;
    for (int64_t base = 0; base < wpr; base += 32 * kWordsInFlight) {
      uint32_t word[kWordsInFlight];
#pragma unroll
      for (int i = 0; i < kWordsInFlight; ++i) {
        const int64_t wi = base + i * 32 + lane;
        word[i] = wi < wpr ? __ldg(wr + wi) : 0u;
      }
#pragma unroll
      for (int i = 0; i < kWordsInFlight; ++i) {
        const int64_t wi = base + i * 32 + lane;
        if (wi >= wpr) break;
        const int64_t l0 = wi * 8;
        float deq[8];
        if (g8) {
          const int64_t g = l0 / a.group;
          const float sc = __ldg(a.scales + j * ng + g);
          const uint32_t sh = (__ldg(a.shifts + j * sw + g / 8) >> (4 * (g % 8))) & 0xFu;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint32_t d = ((word[i] >> (4 * e)) & 0xFu) - sh;  // w - sh, two's complement
            deq[e] = __fmul_rn(sc, __fsub_rn(__uint_as_float(0x4B400000u + d), kMagic));
          }
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int64_t g = (l0 + e) / a.group;
            const float sc = __ldg(a.scales + j * ng + g);
            const uint32_t sh = (__ldg(a.shifts + j * sw + g / 8) >> (4 * (g % 8))) & 0xFu;
            const uint32_t d = ((word[i] >> (4 * e)) & 0xFu) - sh;
            deq[e] = __fmul_rn(sc, __fsub_rn(__uint_as_float(0x4B400000u + d), kMagic));
          }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const uint16_t* yr = a.y + (l0 + e) * a.ld_y;
          if constexpr (N1 == 8) {
            if (yvec) {
              const uint4 v = __ldg(reinterpret_cast<const uint4*>(yr));
              const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                acc[2 * k] = __fmaf_rn(deq[e], __uint_as_float(u[k] << 16), acc[2 * k]);
                acc[2 * k + 1] = __fmaf_rn(deq[e], __uint_as_float(u[k] & 0xffff0000u), acc[2 * k + 1]);
              }
              continue;
            }
          }
#pragma unroll
          for (int k = 0; k < N1; ++k) acc[k] = __fmaf_rn(deq[e], bf16_value(__ldg(yr + k)), acc[k]);
        }
      }
    }
#pragma unroll
    for (int k = 0; k < N1; ++k) {
      float v = acc[k];
#pragma unroll
      for (int o = 16; o; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(kFull, v, o));
      acc[k] = v;
    }
    if (lane == 0) {
#pragma unroll
      for (int k = 0; k < N1; ++k) a.z[j * a.ld_z + k] = acc[k];
    }
  }
}

template <int N1>
qz_status run(const QdArgs& a, bool yvec, cudaStream_t s) {
  auto k = &quant_dot_kernel<N1>;
  const int grid = grid_for(reinterpret_cast<const void*>(k), (a.n0 + kWarps - 1) / kWarps, s);
  k<<<grid, kThreads, 0, s>>>(a, yvec);
  return launch_status();
}

}  // namespace

qz_status launch_quant_dot(const uint32_t* w, const float* scales, const uint32_t* shifts,
                           int64_t n0, int64_t mid, int64_t group, const void* y, int64_t ld_y,
                           int64_t n1, float* z, int64_t ld_z, cudaStream_t s) {
  const QdArgs a{w, scales, shifts, static_cast<const uint16_t*>(y), z, n0, mid, group, ld_y, ld_z};
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
