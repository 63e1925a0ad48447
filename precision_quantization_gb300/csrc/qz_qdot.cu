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

// ---- tensor-core form (group % 16 == 0, mid % 32 == 0) ----------------------------------
// sum_l sc (w - sh) y = sum_groups sc_g * sum_{l in g} (w - sh) y: w - sh is an integer in
// [-15, 15], exact in bf16, and so is every product with a bf16 y in fp32, so the inner
// sums run on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate) and the
// group scale is applied by one FMA per output and group.  The rounding of this order
// stays within the bound qz_quant_dot states for any order of the fp32 terms.
//
// A warp owns 16 weight rows and one slice of l; the 8 warps of a CTA share the slice,
// whose activations are staged in shared memory as yT[n][l] (n < 8, zero past n1, rows
// padded by 8 elements so the fragment reads are conflict-free).
constexpr int kQdSliceMax = 2048;          // l per slice (staged activations: 8 x 2056 bf16)
constexpr int kQdRowsPerCta = 16 * kWarps;

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// bf16 pair (lo, hi) of the nibbles i and i + 1 of `word` minus the shift, exact integers:
// base = 0x4B400000 - sh, so base + nibble is the encoding of 1.5 * 2^23 + (w - sh)
__device__ __forceinline__ uint32_t int_pair_bf16(uint32_t word, int i, uint32_t base) {
  const uint32_t lo = base + ((word >> (4 * i)) & 0xFu);
  const uint32_t hi = base + ((word >> (4 * i + 4)) & 0xFu);
  const uint64_t v = sub2(pk(__uint_as_float(lo), __uint_as_float(hi)), pk(kMagic, kMagic));
  float vl, vh;
  upk(v, vl, vh);
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(vh), "f"(vl));
  return r;
}

__global__ void __launch_bounds__(kThreads) quant_dot_mma_kernel(QdArgs a, int n1) {
  __shared__ uint16_t yT[8][kQdSliceMax + 8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int64_t wpr = a.mid / 8, ng = a.mid / a.group, sw = (ng + 7) / 8;
  const int64_t nrb = (a.n0 + kQdRowsPerCta - 1) / kQdRowsPerCta;
  for (int64_t item = blockIdx.x; item < nrb * a.ksplit; item += gridDim.x) {
    const int64_t r0 = (item / a.ksplit) * kQdRowsPerCta + warp * 16;
    const int64_t l_begin = (item % a.ksplit) * a.wps * 8;
    const int64_t l_len = min(a.wps * 8, a.mid - l_begin);  // a multiple of 32
    __syncthreads();  // the previous item's staged activations are no longer read
    for (int l = threadIdx.x; l < l_len; l += kThreads) {
      const uint16_t* yr = a.y + (l_begin + l) * a.ld_y;
#pragma unroll
      for (int n = 0; n < 8; ++n) yT[n][l] = n < n1 ? yr[n] : static_cast<uint16_t>(0);
    }
    __syncthreads();
    const int64_t ra = min(r0 + g, a.n0 - 1), rb = min(r0 + g + 8, a.n0 - 1);  // rows of this lane
    float z[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // rows g / g+8, columns 2t, 2t+1
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    int64_t cur = -1;  // group of acc
    float sca = 0.0f, scb = 0.0f;
    uint32_t sha = 0u, shb = 0u;  // 0x4B400000 - shift of rows g / g+8
    if (r0 < a.n0) {
      for (int64_t l = 0; l < l_len; l += 32) {
        const int64_t lg = l_begin + l;      // global l of this 32-wide step
        const uint4 wa = __ldg(reinterpret_cast<const uint4*>(a.w + ra * wpr + lg / 8));
        const uint4 wb = __ldg(reinterpret_cast<const uint4*>(a.w + rb * wpr + lg / 8));
        const uint32_t wra[4] = {wa.x, wa.y, wa.z, wa.w}, wrb[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
        for (int s = 0; s < 2; ++s) {       // two k16 steps
          const int64_t k0 = lg + 16 * s;
          const int64_t grp = k0 / a.group;
          if (grp != cur) {                  // close the previous group: z += sc * acc
            z[0] = __fmaf_rn(sca, acc[0], z[0]);
            z[1] = __fmaf_rn(sca, acc[1], z[1]);
            z[2] = __fmaf_rn(scb, acc[2], z[2]);
            z[3] = __fmaf_rn(scb, acc[3], z[3]);
            acc[0] = acc[1] = acc[2] = acc[3] = 0.0f;
            cur = grp;
            sca = __ldg(a.scales + ra * ng + grp);
            scb = __ldg(a.scales + rb * ng + grp);
            sha = 0x4B400000u - ((__ldg(a.shifts + ra * sw + grp / 8) >> (4 * (grp % 8))) & 0xFu);
            shb = 0x4B400000u - ((__ldg(a.shifts + rb * sw + grp / 8) >> (4 * (grp % 8))) & 0xFu);
          }
          uint32_t af[4];
          af[0] = int_pair_bf16(wra[2 * s], 2 * t, sha);      // row g,   k 2t, 2t+1
          af[1] = int_pair_bf16(wrb[2 * s], 2 * t, shb);      // row g+8, k 2t, 2t+1
          af[2] = int_pair_bf16(wra[2 * s + 1], 2 * t, sha);  // row g,   k 2t+8, 2t+9
          af[3] = int_pair_bf16(wrb[2 * s + 1], 2 * t, shb);  // row g+8, k 2t+8, 2t+9
          const int64_t kl = l + 16 * s + 2 * t;               // slice-local k of b0
          const uint32_t b0 = *reinterpret_cast<const uint32_t*>(&yT[g][kl]);
          const uint32_t b1 = *reinterpret_cast<const uint32_t*>(&yT[g][kl + 8]);
          mma_bf16_16816(acc, af, b0, b1);
        }
      }
      z[0] = __fmaf_rn(sca, acc[0], z[0]);
      z[1] = __fmaf_rn(sca, acc[1], z[1]);
      z[2] = __fmaf_rn(scb, acc[2], z[2]);
      z[3] = __fmaf_rn(scb, acc[3], z[3]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t row = r0 + g + (i >= 2 ? 8 : 0);
        const int col = 2 * t + (i & 1);
        if (row < a.n0 && col < n1) {
          float* zp = a.z + row * a.ld_z + col;
          if (a.ksplit > 1) atomicAdd(zp, z[i]);
          else *zp = z[i];
        }
      }
    }
  }
}

qz_status run_mma(QdArgs a, int n1, cudaStream_t s) {
  const int64_t wpr = a.mid / 8, nrb = (a.n0 + kQdRowsPerCta - 1) / kQdRowsPerCta;
  const int64_t want = static_cast<int64_t>(sm_count()) * 2;  // CTAs
  int64_t ks = std::max<int64_t>((want + nrb - 1) / nrb, (a.mid + kQdSliceMax - 1) / kQdSliceMax);
  ks = std::max<int64_t>(1, std::min<int64_t>(ks, wpr / 4));
  a.wps = ((wpr + ks - 1) / ks + 3) / 4 * 4;  // words per slice: l a multiple of 32
  a.ksplit = (wpr + a.wps - 1) / a.wps;
  if (a.ksplit > 1 &&
      cudaMemset2DAsync(a.z, static_cast<size_t>(a.ld_z) * 4, 0, static_cast<size_t>(n1) * 4,
                        static_cast<size_t>(a.n0), s) != cudaSuccess)
    return QZ_ERR_CUDA;
  const int grid = grid_for(reinterpret_cast<const void*>(&quant_dot_mma_kernel), nrb * a.ksplit, s);
  quant_dot_mma_kernel<<<grid, kThreads, 0, s>>>(a, static_cast<int>(n1));
  return launch_status();
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
  if (group % 16 == 0 && mid % 32 == 0 && reinterpret_cast<uintptr_t>(w) % 16 == 0)
    return run_mma(a, static_cast<int>(n1), s);
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
