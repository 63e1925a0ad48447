// qz_dequant.cu -- x^ = fl32(decode(q) * s), written as bf16 (round to nearest even) or
// fp32 (blog post "浅谈低精度浮点数": x^ = s * Q(x / s) for INT8 / FP8, and
// x^ = s * Q_E2M1(...) with s the E8M0 scale for MXFP4 or s_global * s_block for NVFP4).
//
// Each lane produces one 32-byte chunk of y (16 bf16 / 8 fp32 values): it reads that
// chunk's codes (one 16/8/4-byte load), its block scale byte (FP4) or row scale (ROW),
// decodes two codes per cvt, multiplies, and writes the chunk with one 256-bit store.
#include "qz_device.cuh"
#include "qz_internal.h"

namespace qz {
namespace {

constexpr int kUnroll = 4;  // chunks per thread in flight

struct DqArgs {
  const uint8_t* codes;
  const void* scales;
  const float* tscale;
  void* y;
  Geom g;  // over y
};

template <int ODT>
__device__ __forceinline__ void put_chunk(void* y, const Geom& g, int64_t row, int64_t col,
                                          int64_t nv, const float* xh, bool vec) {
  constexpr int EPC = Elem<ODT>::kPer32B;
  const int64_t e0 = row * g.ld + col;
  if (vec) {
    uint32_t w[8];
    if constexpr (ODT == QZ_BF16) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(w[i]) : "f"(xh[2 * i + 1]), "f"(xh[2 * i]));
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = __float_as_uint(xh[i]);
    }
    st32B(static_cast<char*>(y) + e0 * Elem<ODT>::kBytes, w);
  } else {
#pragma unroll
    for (int i = 0; i < EPC; ++i)
      if (i < nv) store_elem<ODT>(y, e0 + i, xh[i]);
  }
}

// MXFP4 / NVFP4
template <int FMT, int ODT, bool UNIT, bool VEC>
__global__ void __launch_bounds__(kThreads) dequant4_kernel(DqArgs a) {
  constexpr int EPC = Elem<ODT>::kPer32B;
  constexpr int BS = FMT == QZ_MXFP4 ? 32 : 16;
  constexpr int CB = EPC / 2;
  const Geom& g = a.g;
  float sg = 1.0f;
  if constexpr (FMT == QZ_NVFP4 && !UNIT) sg = *a.tscale;
  const uint8_t* sc = static_cast<const uint8_t*>(a.scales);
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t nthr = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t base = tid; base < g.n_chunks; base += nthr * kUnroll) {
    // all loads of the kUnroll chunks first, then the arithmetic and the stores
    uint32_t cw[kUnroll][2];
    uint32_t sc_code[kUnroll];
    int64_t row[kUnroll], col[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const int64_t u = base + k * nthr;
      if (g.dense) {
        row[k] = 0;
        col[k] = u * EPC;
      } else {
        row[k] = u / g.cpr;
        col[k] = (u - row[k] * g.cpr) * EPC;
      }
      cw[k][0] = cw[k][1] = 0u;
      sc_code[k] = 127u;
      if (u < g.n_chunks) {
        const int64_t cofs = g.dense ? col[k] / 2 : row[k] * (g.cols / 2) + col[k] / 2;
        const int64_t sofs = g.dense ? col[k] / BS : row[k] * (g.cols / BS) + col[k] / BS;
        if constexpr (VEC) {
          if constexpr (CB == 8) {
            const uint2 v = ld8B(a.codes + cofs);
            cw[k][0] = v.x;
            cw[k][1] = v.y;
          } else {
            cw[k][0] = ld4B(a.codes + cofs);
          }
        } else {
#pragma unroll
          for (int j = 0; j < CB; ++j) cw[k][j / 4] |= static_cast<uint32_t>(a.codes[cofs + j]) << (8 * (j % 4));
        }
        if constexpr (!UNIT) sc_code[k] = ld1B(sc + sofs);
      }
    }
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      if (base + k * nthr >= g.n_chunks) break;
      float s;
      if constexpr (FMT == QZ_MXFP4) {
        const uint32_t c = UNIT ? 127u : sc_code[k];
        s = c == 255u ? __uint_as_float(0x7fc00000u) : exp2_pos(static_cast<int>(c) - 127);
      } else {
        s = UNIT ? 1.0f : __fmul_rn(sg, dec_e4m3(sc_code[k]));
      }
      float xh[EPC];
#pragma unroll
      for (int j = 0; j < CB; ++j) {
        float q0, q1;
        dec_e2m1x2((cw[k][j / 4] >> (8 * (j % 4))) & 0xffu, q0, q1);
        xh[2 * j] = __fmul_rn(q0, s);
        xh[2 * j + 1] = __fmul_rn(q1, s);
      }
      put_chunk<ODT>(a.y, g, row[k], col[k], EPC, xh, VEC);
    }
  }
}

// INT8 / FP8
template <int FMT, int ODT, int GRAN, bool VEC>
__global__ void __launch_bounds__(kThreads) dequant8_kernel(DqArgs a) {
  constexpr int EPC = Elem<ODT>::kPer32B;
  const Geom& g = a.g;
  float st = 1.0f;
  if constexpr (GRAN == QZ_GRAN_TENSOR) st = *a.tscale;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  const int64_t nthr = static_cast<int64_t>(gridDim.x) * kThreads;
  for (int64_t base = tid; base < g.n_chunks; base += nthr * kUnroll) {
    uint32_t cw[kUnroll][EPC / 4];
    float sk[kUnroll];
    int64_t row[kUnroll], col[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const int64_t u = base + k * nthr;
      if (g.dense) {
        row[k] = 0;
        col[k] = u * EPC;
      } else {
        row[k] = u / g.cpr;
        col[k] = (u - row[k] * g.cpr) * EPC;
      }
#pragma unroll
      for (int j = 0; j < EPC / 4; ++j) cw[k][j] = 0u;
      sk[k] = st;
      if (u < g.n_chunks) {
        const int64_t nv = g.dense ? EPC : g.cols - col[k];
        const uint8_t* cp = a.codes + (g.dense ? col[k] : row[k] * g.cols + col[k]);
        if constexpr (VEC) {
          if constexpr (EPC == 16) {
            const uint4 v = ld16B(cp);
            cw[k][0] = v.x;
            cw[k][1] = v.y;
            cw[k][2] = v.z;
            cw[k][3] = v.w;
          } else {
            const uint2 v = ld8B(cp);
            cw[k][0] = v.x;
            cw[k][1] = v.y;
          }
        } else {
#pragma unroll
          for (int j = 0; j < EPC; ++j)
            if (j < nv) cw[k][j / 4] |= static_cast<uint32_t>(cp[j]) << (8 * (j % 4));
        }
        if constexpr (GRAN == QZ_GRAN_ROW) {
          const int64_t r = g.dense ? (col[k] / g.cols) : row[k];
          sk[k] = static_cast<const float*>(a.scales)[r];
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const int64_t u = base + k * nthr;
      if (u >= g.n_chunks) break;
      const int64_t nv = g.dense ? EPC : g.cols - col[k];
      float xh[EPC];
#pragma unroll
      for (int j = 0; j < EPC / 2; ++j) {
        float q0, q1;
        dec8x2<FMT>((cw[k][j / 2] >> (16 * (j % 2))) & 0xffffu, q0, q1);
        xh[2 * j] = __fmul_rn(q0, sk[k]);
        xh[2 * j + 1] = __fmul_rn(q1, sk[k]);
      }
      put_chunk<ODT>(a.y, g, row[k], col[k], nv, xh, VEC);
    }
  }
}

template <typename K>
qz_status go(K kern, const DqArgs& args, cudaStream_t s) {
  const int64_t work = (args.g.n_chunks + kThreads * kUnroll - 1) / (kThreads * kUnroll);
  const int grid = grid_for(reinterpret_cast<const void*>(kern), work, s);
  kern<<<grid, kThreads, 0, s>>>(args);
  return launch_status();
}

template <int FMT, int ODT>
qz_status run4(const DqArgs& a, bool unit, cudaStream_t s) {
  if (unit) return a.g.vec ? go(&dequant4_kernel<FMT, ODT, true, true>, a, s) : go(&dequant4_kernel<FMT, ODT, true, false>, a, s);
  return a.g.vec ? go(&dequant4_kernel<FMT, ODT, false, true>, a, s) : go(&dequant4_kernel<FMT, ODT, false, false>, a, s);
}

template <int FMT, int ODT, int GRAN>
qz_status run8g(const DqArgs& a, cudaStream_t s) {
  return a.g.vec ? go(&dequant8_kernel<FMT, ODT, GRAN, true>, a, s) : go(&dequant8_kernel<FMT, ODT, GRAN, false>, a, s);
}

template <int FMT, int ODT>
qz_status run8(const DqArgs& a, int gran, cudaStream_t s) {
  if (gran == QZ_GRAN_TENSOR) return run8g<FMT, ODT, QZ_GRAN_TENSOR>(a, s);
  if (gran == QZ_GRAN_ROW) return run8g<FMT, ODT, QZ_GRAN_ROW>(a, s);
  return run8g<FMT, ODT, QZ_GRAN_UNIT>(a, s);
}

DqArgs make_args(const qz_desc& d, const void* codes, const void* scales, const float* tscale,
                 void* y, int out_dtype) {
  DqArgs a;
  a.codes = static_cast<const uint8_t*>(codes);
  a.scales = scales;
  a.tscale = tscale;
  a.y = y;
  a.g = make_geom(d, y, out_dtype == QZ_BF16 ? 2 : 4, 32);
  if (reinterpret_cast<uintptr_t>(codes) % 16 != 0) {
    a.g.vec = false;
    a.g.dense = false;
  }
  return a;
}

}  // namespace

qz_status launch_dequant4(const qz_desc& d, const void* codes, const void* scales,
                          const float* tscale, void* y, int out_dtype, cudaStream_t s) {
  const DqArgs a = make_args(d, codes, scales, tscale, y, out_dtype);
  const bool unit = d.granularity == QZ_GRAN_UNIT;
  if (d.format == QZ_MXFP4)
    return out_dtype == QZ_BF16 ? run4<QZ_MXFP4, QZ_BF16>(a, unit, s) : run4<QZ_MXFP4, QZ_F32>(a, unit, s);
  return out_dtype == QZ_BF16 ? run4<QZ_NVFP4, QZ_BF16>(a, unit, s) : run4<QZ_NVFP4, QZ_F32>(a, unit, s);
}

qz_status launch_dequant8(const qz_desc& d, const void* codes, const void* scales,
                          const float* tscale, void* y, int out_dtype, cudaStream_t s) {
  const DqArgs a = make_args(d, codes, scales, tscale, y, out_dtype);
  const int gr = d.granularity;
  switch (d.format) {
    case QZ_INT8: return out_dtype == QZ_BF16 ? run8<QZ_INT8, QZ_BF16>(a, gr, s) : run8<QZ_INT8, QZ_F32>(a, gr, s);
    case QZ_FP8_E4M3:
      return out_dtype == QZ_BF16 ? run8<QZ_FP8_E4M3, QZ_BF16>(a, gr, s) : run8<QZ_FP8_E4M3, QZ_F32>(a, gr, s);
    default: return out_dtype == QZ_BF16 ? run8<QZ_FP8_E5M2, QZ_BF16>(a, gr, s) : run8<QZ_FP8_E5M2, QZ_F32>(a, gr, s);
  }
}

}  // namespace qz
