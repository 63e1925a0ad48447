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
          if (fast_div_ok(s) && __fmul_rn(A, r) <= 0x1p100f) {
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

template <int FMT, int DT, bool UNIT, bool STATS, bool VEC>
qz_status run(const Q4Args& args, cudaStream_t s) {
  auto kern = &quant4_kernel<FMT, DT, UNIT, STATS, VEC>;
  const int64_t per_cta = static_cast<int64_t>(kThreads) * kUnroll;
  const int grid = grid_for(reinterpret_cast<const void*>(kern), (args.g.n_chunks + per_cta - 1) / per_cta, s);
  kern<<<grid, kThreads, 0, s>>>(args);
  return launch_status();
}

template <int FMT, int DT>
qz_status dispatch(const Q4Args& args, bool unit, bool stats, cudaStream_t s) {
  const bool vec = args.g.vec;
  if (unit) {
    if (stats) return vec ? run<FMT, DT, true, true, true>(args, s) : run<FMT, DT, true, true, false>(args, s);
    return vec ? run<FMT, DT, true, false, true>(args, s) : run<FMT, DT, true, false, false>(args, s);
  }
  if (stats) return vec ? run<FMT, DT, false, true, true>(args, s) : run<FMT, DT, false, true, false>(args, s);
  return vec ? run<FMT, DT, false, false, true>(args, s) : run<FMT, DT, false, false, false>(args, s);
}

}  // namespace

qz_status launch_quant4(const qz_desc& d, const void* x, void* codes, void* scales,
                        float* tscale_out, const float* amax, bool /*amax_supplied*/,
                        qz_stats* stats, void* ws, cudaStream_t s) {
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
  const bool unit = d.granularity == QZ_GRAN_UNIT;
  const bool st = stats != nullptr;
  if (d.format == QZ_MXFP4)
    return d.in_dtype == QZ_BF16 ? dispatch<QZ_MXFP4, QZ_BF16>(args, unit, st, s)
                                 : dispatch<QZ_MXFP4, QZ_F32>(args, unit, st, s);
  return d.in_dtype == QZ_BF16 ? dispatch<QZ_NVFP4, QZ_BF16>(args, unit, st, s)
                               : dispatch<QZ_NVFP4, QZ_F32>(args, unit, st, s);
}

}  // namespace qz
