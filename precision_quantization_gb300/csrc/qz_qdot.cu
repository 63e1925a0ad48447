// qz_qdot.cu -- the quantized matrix product of the blog's "Puzzles 12 Quantized Matrix Mult"
// (section of its "Triton" post): z[j][k] = sum_l sc[j][l/g] (w[j][l] - sh[j][l/g]) y[l][k],
// with 4-bit weights w packed 8 per 32-bit word (low nibble first), one fp32 scale and one
// 4-bit shift per group of g weights along l, and bf16 activations y.
//
// For a few activation columns (n1 <= 8: decoding, small batches) the product streams the
// packed weights once and does 2 * n1 flops per 4-bit weight.  Two forms:
//   - tensor-core form (group % 16 == 0, mid % 64 == 0, 16-byte aligned words): the sum
//     regrouped as sum over groups of sc * sum (w - sh) y; the inner sums, whose factors
//     are exact small integers and bf16 values, run on mma.sync (bf16 in, fp32
//     accumulate), the group scale is one FMA per output and group;
//   - FMA form (any other group): a warp takes a block of weight rows, its lanes the rows'
//     32-bit code words (coalesced 128-byte reads), the weights are dequantized in
//     registers exactly as qz_dequantize_asym4 does (fl32(sc * (w - sh))), accumulation is
//     fp32 by paired FMA, and a shuffle reduction across the warp finishes each output.
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

// z[j][0 .. n1) = 0 for the split sums to add into (a 2-D memset of 4 * n1-byte rows)
__global__ void __launch_bounds__(kThreads) zero_z_kernel(float* z, int64_t ld_z, int64_t n0, int n1) {
  const int64_t n = n0 * n1;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * kThreads)
    z[(i / n1) * ld_z + i % n1] = 0.0f;
}

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

// ---- tensor-core form (group % 16 == 0, mid % 64 == 0) ----------------------------------
// sum_l sc (w - sh) y = sum_groups sc_g * sum_{l in g} (w - sh) y: w - sh is an integer in
// [-15, 15], exact in bf16, and so is every product with a bf16 y in fp32, so the inner
// sums run on the tensor cores (mma.sync m16n8k16, bf16 in, fp32 accumulate) and the
// group scale is applied by one FMA per output and group.  The rounding of this order
// stays within the bound qz_quant_dot states for any order of the fp32 terms.
//
// Work item: 128 weight rows (16 per warp) x one slice of l.  Per item the CTA stages in
// shared memory the slice's activations as rows of 8 bf16 (ys[l][n], zero past n1) and the
// rows' scales and shift words for the groups the slice touches; each warp streams its
// rows' code words through a ring of kQdBatches batches of kQdBatch 64-wide steps (32
// kQdBatch contiguous bytes of each of its 16 rows per batch, 16-byte cp.async), the
// later batches in flight while the first is consumed.  Activations (n1 == 8, aligned
// rows), scales, shifts and code words all move by cp.async.
//
// The k order inside a 16-wide part is permuted, the same way for both operands (a sum
// does not depend on the naming of its index): mma slots (2t, 2t+1, 2t+8, 2t+9) of lane
// t hold l = (t, t+4, 8+t, 12+t).  Then the weight pair a lane needs from one code word is
// its nibbles t and t+4, i.e. (word >> 4t) & 0x000F000F, which OR 0x43004300 turns into the
// bf16 pair (128 + w_t, 128 + w_t+4); one bf16x2 FMA subtracts 128 + sh exactly.  The B
// fragments come from ys by ldmatrix.trans, whose per-lane row addresses apply the same
// permutation (row r of an 8 x 8 tile <-> slot r <-> l = r / 2 + 4 (r % 2)).
constexpr int kQdSlice = 1024;                 // max l per slice
constexpr int kQdBatch = 4;                    // 64-wide steps per batch of code words (2 or 4)
constexpr int kQdBatches = 3;                  // batches in the ring of a warp
constexpr int kQdStages = kQdBatch * kQdBatches;
constexpr int kQdRowsPerCta = 16 * kWarps;
constexpr int kQdGroups = 17;                  // groups a slice may touch (slice <= 16 groups)

struct QdSmem {
  uint4 ys[kQdSlice];  // activation row l: y[l][0 .. 8) as bf16
  uint32_t wbuf[kWarps][kQdStages][16][8];
  float sc[kQdRowsPerCta][kQdGroups];
  uint32_t shw[kQdRowsPerCta][3];  // the shift words covering those groups
};

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// the bf16 pair (w_t - sh, w_t+4 - sh) of a code word already shifted right by 4t;
// nsh = the bf16 pair (-(128 + sh), -(128 + sh))
__device__ __forceinline__ uint32_t weight_pair(uint32_t shifted, uint32_t nsh) {
  uint32_t x, r;
  asm("lop3.b32 %0, %1, 0x000F000F, 0x43004300, 0xEA;" : "=r"(x) : "r"(shifted));  // (a & b) | c
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(x), "r"(0x3F803F80u), "r"(nsh));  // x * 1 + nsh
  return r;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr) : "memory");
}

// Quotient by an invariant divisor d by one multiply (Granlund and Montgomery, "Division
// by invariant integers using multiplication", 1994): with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, n / d = (umulhi(m, n) + n) >> l for 0 <= n < 2^31.
struct FastDiv {
  uint32_t m = 1, l = 0;
  FastDiv() = default;
  explicit FastDiv(uint32_t d) {
    while ((1ull << l) < d) ++l;
    m = static_cast<uint32_t>(((1ull << 32) * ((1ull << l) - d)) / d + 1);
  }
  __device__ __forceinline__ int operator()(int n) const {
    return static_cast<int>((__umulhi(m, static_cast<uint32_t>(n)) + static_cast<uint32_t>(n)) >> l);
  }
};

struct QmArgs {
  const uint32_t* w;
  const float* scales;
  const uint32_t* shifts;
  const uint16_t* y;  // bf16 bits [mid, ld_y]
  float* z;
  int64_t n0, ld_y, ld_z, wpr, ng, sw;  // wpr: code words per row; ng / sw: groups / shift words per row
  int mid, group, lps, ksplit, nitems;  // lps: l per slice (a multiple of 64); items = row blocks x slices
  FastDiv by_ksplit, by_group;
};

// G64: group % 64 == 0, so groups change only between 64-wide steps
template <bool G64>
__global__ void __launch_bounds__(kThreads, 3) quant_dot_mma_kernel(QmArgs a, int n1, bool yvec) {
  extern __shared__ __align__(16) unsigned char qd_smem_raw[];
  QdSmem& sm = *reinterpret_cast<QdSmem*>(qd_smem_raw);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  constexpr uint32_t kStageBytes = 16 * 8 * 4;
  // ldmatrix row address of this lane: tile m = lane / 8 (part m / 2, slots 8 (m % 2) ..),
  // row r = lane % 8 <-> l = 16 (m / 2) + 8 (m % 2) + r / 2 + 4 (r % 2)
  const int mt = lane >> 3, mr = lane & 7;
  const uint32_t yl = static_cast<uint32_t>(__cvta_generic_to_shared(
      &sm.ys[16 * (mt >> 1) + 8 * (mt & 1) + (mr >> 1) + 4 * (mr & 1)]));
  const uint32_t wl = static_cast<uint32_t>(__cvta_generic_to_shared(&sm.wbuf[warp][0][g][0]));
  // the copies of a lane: 16 bytes of row kRowsPerCopy j + lane / kChunks, chunk
  // lane % kChunks of a batch (step chunk / 2, half chunk % 2)
  constexpr int kChunks = 2 * kQdBatch;           // 16-byte chunks of a row in a batch
  constexpr int kRowsPerCopy = 32 / kChunks;      // rows one copy instruction covers
  constexpr int kCopies = 16 / kRowsPerCopy;      // copies per lane and batch
  const int cchunk = lane % kChunks, crow = warp * 16 + lane / kChunks;  // CTA-local row of copy 0
  const uint32_t cdst0 = static_cast<uint32_t>(
      __cvta_generic_to_shared(&sm.wbuf[warp][cchunk >> 1][lane / kChunks][4 * (cchunk & 1)]));
  const int ra = warp * 16 + g, rb = ra + 8;  // CTA-local rows of this lane's outputs

  for (int item = blockIdx.x; item < a.nitems; item += gridDim.x) {
    const int kb = a.by_ksplit(item);
    const int64_t rc = static_cast<int64_t>(kb) * kQdRowsPerCta;  // first row of the CTA
    const int rlast = static_cast<int>(min(static_cast<int64_t>(kQdRowsPerCta - 1), a.n0 - 1 - rc));
    const int l_begin = (item - kb * a.ksplit) * a.lps;
    const int l_len = min(a.lps, a.mid - l_begin);  // a multiple of 64
    const int g_first = a.by_group(l_begin);
    const int ngs = a.by_group(l_begin + l_len - 1) - g_first + 1;  // <= kQdGroups
    const int nsteps = l_len / 64, nbatches = (nsteps + kQdBatch - 1) / kQdBatch;
    const bool live = warp * 16 <= rlast;
    __syncthreads();  // the previous item's staged data is no longer read

    // scales and shift words of the CTA's rows for the groups g_first .. g_first + ngs - 1,
    // by 4-byte asynchronous copies (rows past the end are left as they are: their
    // outputs are not written).  Entry idx -> (row idx / n, idx % n); the quotient by a
    // float reciprocal is exact here: (idx + 1/2) / n lies at least 1 / (2 n) from an
    // integer, and idx < 2^12.
    const int gfo = g_first & 7;                // nibble of g_first in its shift word
    const int nsw = (gfo + ngs + 7) / 8;        // shift words per row, <= 3
    {
      const float* sbase = a.scales + rc * a.ng + g_first;
      const float rcp = 1.0f / static_cast<float>(ngs);
      for (int idx = threadIdx.x; idx < kQdRowsPerCta * ngs; idx += kThreads) {
        const int rr = static_cast<int>((static_cast<float>(idx) + 0.5f) * rcp), gi = idx - rr * ngs;
        if (rr <= rlast)
          cp_async4(static_cast<uint32_t>(__cvta_generic_to_shared(&sm.sc[rr][gi])), sbase + rr * a.ng + gi);
      }
      const uint32_t* hbase = a.shifts + rc * a.sw + (g_first >> 3);
      const float rcpw = 1.0f / static_cast<float>(nsw);
      for (int idx = threadIdx.x; idx < kQdRowsPerCta * nsw; idx += kThreads) {
        const int rr = static_cast<int>((static_cast<float>(idx) + 0.5f) * rcpw), k = idx - rr * nsw;
        if (rr <= rlast)
          cp_async4(static_cast<uint32_t>(__cvta_generic_to_shared(&sm.shw[rr][k])), hbase + rr * a.sw + k);
      }
    }
    // activations of the slice: rows of 16 bytes
    const uint16_t* ybase = a.y + static_cast<int64_t>(l_begin) * a.ld_y;
    if (yvec) {  // n1 == 8, rows 16-byte aligned: copied as they are
      for (int l = threadIdx.x; l < l_len; l += kThreads)
        cp_async16(static_cast<uint32_t>(__cvta_generic_to_shared(&sm.ys[l])), ybase + l * a.ld_y);
    } else {  // zero past n1
      for (int l = threadIdx.x; l < l_len; l += kThreads) {
        const uint16_t* yr = ybase + l * a.ld_y;
        uint32_t v[4];
#pragma unroll
        for (int n = 0; n < 4; ++n) {
          const uint32_t lo = 2 * n < n1 ? __ldg(yr + 2 * n) : 0u;
          const uint32_t hi = 2 * n + 1 < n1 ? __ldg(yr + 2 * n + 1) : 0u;
          v[n] = lo | (hi << 16);
        }
        sm.ys[l] = make_uint4(v[0], v[1], v[2], v[3]);
      }
    }
    cp_async_commit();  // scales, shifts and activations: one group, older than the code words'

    // this warp's code words, a batch at a time (rows past the end are not copied)
    const uint32_t* csrc = a.w + (rc + crow) * a.wpr + l_begin / 8 + 4 * cchunk;
    const int64_t cstride = kRowsPerCopy * a.wpr;
    int ahead = 0;     // batches issued so far
    int bt_issue = 0;  // ring slot of the next one
    const auto issue = [&]() {
      if (ahead < nbatches && kQdBatch * ahead + (cchunk >> 1) < nsteps) {
        const uint32_t dst = cdst0 + bt_issue * (kQdBatch * kStageBytes);
        const uint32_t* src = csrc + 8 * kQdBatch * ahead;
#pragma unroll
        for (int j = 0; j < kCopies; ++j)
          if (crow + kRowsPerCopy * j <= rlast) cp_async16(dst + j * kRowsPerCopy * 32, src + j * cstride);
      }
      cp_async_commit();  // empty groups keep the count uniform
      ++ahead;
      bt_issue = bt_issue == kQdBatches - 1 ? 0 : bt_issue + 1;
    };
    if (live) {
#pragma unroll
      for (int i = 0; i < kQdBatches - 1; ++i) issue();
      cp_async_wait<kQdBatches - 1>();  // the scale group (older than the code words)
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (!live) continue;  // a warp past the last row: nothing below synchronises the CTA

    float z[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // rows g / g+8, columns 2t, 2t+1
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    int gi = 0;  // staged group of acc
    // its l still to come, in 64- or 16-wide units
    int left = ((g_first + 1) * a.group - l_begin) / (G64 ? 64 : 16);
    const int per = a.group / (G64 ? 64 : 16);
    // -(128 + sh) as a bf16 pair, for staged group gi of CTA-local row r
    const auto nshift = [&](int r, int gi) {
      const int p = gfo + gi;
      return 0xC300C300u + 0x00010001u * ((sm.shw[r][p >> 3] >> (4 * (p & 7))) & 0xFu);
    };
    float sca = sm.sc[ra][0], scb = sm.sc[rb][0];
    uint32_t nsa = nshift(ra, 0), nsb = nshift(rb, 0);
    const auto next_group = [&]() {  // z += sc * acc for the group just closed; load the next
      z[0] = __fmaf_rn(sca, acc[0], z[0]);
      z[1] = __fmaf_rn(sca, acc[1], z[1]);
      z[2] = __fmaf_rn(scb, acc[2], z[2]);
      z[3] = __fmaf_rn(scb, acc[3], z[3]);
      acc[0] = acc[1] = acc[2] = acc[3] = 0.0f;
      ++gi;
      sca = sm.sc[ra][gi];
      scb = sm.sc[rb][gi];
      nsa = nshift(ra, gi);
      nsb = nshift(rb, gi);
    };
    int slot = 0;  // ring slot of batch bt
#pragma unroll 1
    for (int bt = 0; bt < nbatches; ++bt) {
      cp_async_wait<kQdBatches - 2>();  // this lane's copies of batch bt have landed
      __syncwarp();                     // ... and every lane's; batch bt - 1 is read
      issue();
      const uint32_t wsl = wl + slot * (kQdBatch * kStageBytes);
      const uint32_t ysl = yl + bt * (kQdBatch * 64 * 16);
      slot = slot == kQdBatches - 1 ? 0 : slot + 1;
      const int nq = min(kQdBatch, nsteps - kQdBatch * bt);
#pragma unroll
      for (int q = 0; q < kQdBatch; ++q) {  // the batch's 64-wide steps
        if (q >= nq) break;
        const uint32_t wst = wsl + q * kStageBytes;
        const uint4 wa0 = lds128(wst), wa1 = lds128(wst + 16);                    // row g
        const uint4 wb0 = lds128(wst + 8 * 32), wb1 = lds128(wst + 8 * 32 + 16);  // row g + 8
        uint32_t yb[8];  // B registers (b0, b1) of parts 0 .. 3
        ldsm_x4_trans(*reinterpret_cast<uint32_t(*)[4]>(&yb[0]), ysl + q * 64 * 16);            // parts 0, 1
        ldsm_x4_trans(*reinterpret_cast<uint32_t(*)[4]>(&yb[4]), ysl + q * 64 * 16 + 32 * 16);  // parts 2, 3
        if (G64) {
          if (left == 0) {
            next_group();
            left = per;
          }
          --left;
        }
        const uint32_t wa[8] = {wa0.x, wa0.y, wa0.z, wa0.w, wa1.x, wa1.y, wa1.z, wa1.w};
        const uint32_t wb[8] = {wb0.x, wb0.y, wb0.z, wb0.w, wb1.x, wb1.y, wb1.z, wb1.w};
#pragma unroll
        for (int s = 0; s < 4; ++s) {  // four k16 parts
          if (!G64) {
            if (left == 0) {
              next_group();
              left = per;
            }
            --left;
          }
          uint32_t af[4];
          af[0] = weight_pair(wa[2 * s] >> (4 * t), nsa);      // row g,   slots 2t, 2t+1
          af[1] = weight_pair(wb[2 * s] >> (4 * t), nsb);      // row g+8, slots 2t, 2t+1
          af[2] = weight_pair(wa[2 * s + 1] >> (4 * t), nsa);  // row g,   slots 2t+8, 2t+9
          af[3] = weight_pair(wb[2 * s + 1] >> (4 * t), nsb);  // row g+8, slots 2t+8, 2t+9
          mma_bf16_16816(acc, af, yb[2 * s], yb[2 * s + 1]);
        }
      }
    }
    cp_async_wait<0>();
    __syncwarp();
    z[0] = __fmaf_rn(sca, acc[0], z[0]);
    z[1] = __fmaf_rn(sca, acc[1], z[1]);
    z[2] = __fmaf_rn(scb, acc[2], z[2]);
    z[3] = __fmaf_rn(scb, acc[3], z[3]);
    float* zr = a.z + (rc + ra) * a.ld_z + 2 * t;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int row = ra + (q >= 2 ? 8 : 0), col = 2 * t + (q & 1);
      if (row <= rlast && col < n1) {
        float* zp = zr + (q >= 2 ? 8 * a.ld_z : 0) + (q & 1);
        if (a.ksplit > 1) atomicAdd(zp, z[q]);
        else *zp = z[q];
      }
    }
  }
}

// false when the sizes leave the 32-bit index range the kernel assumes
bool run_mma(QdArgs in, int n1, bool yvec, cudaStream_t s, qz_status* st) {
  const int64_t wpr = in.mid / 8, nrb = (in.n0 + kQdRowsPerCta - 1) / kQdRowsPerCta;
  // a slice spans at most 16 groups (so it touches at most kQdGroups) and kQdSlice values
  const int64_t lmax = std::min<int64_t>(kQdSlice, 16 * in.group);  // a multiple of 256
  const int64_t want = static_cast<int64_t>(sm_count()) * 2;        // CTAs
  int64_t ks = std::max<int64_t>((want + nrb - 1) / nrb, (in.mid + lmax - 1) / lmax);
  ks = std::max<int64_t>(1, std::min<int64_t>(ks, wpr / 8));
  const int64_t wps = ((wpr + ks - 1) / ks + 7) / 8 * 8;  // words per slice: l a multiple of 64
  const int64_t ksplit = (wpr + wps - 1) / wps;
  if (in.mid + in.group >= (int64_t{1} << 31) || nrb * ksplit >= (int64_t{1} << 31)) return false;
  QmArgs a;
  a.w = in.w;
  a.scales = in.scales;
  a.shifts = in.shifts;
  a.y = in.y;
  a.z = in.z;
  a.n0 = in.n0;
  a.ld_y = in.ld_y;
  a.ld_z = in.ld_z;
  a.wpr = wpr;
  a.ng = in.mid / in.group;
  a.sw = (a.ng + 7) / 8;
  a.mid = static_cast<int>(in.mid);
  a.group = static_cast<int>(in.group);
  a.lps = static_cast<int>(wps * 8);
  a.ksplit = static_cast<int>(ksplit);
  a.nitems = static_cast<int>(nrb * ksplit);
  a.by_ksplit = FastDiv(static_cast<uint32_t>(ksplit));
  a.by_group = FastDiv(static_cast<uint32_t>(in.group));
  const bool g64 = in.group % 64 == 0;
  const void* k = g64 ? reinterpret_cast<const void*>(&quant_dot_mma_kernel<true>)
                      : reinterpret_cast<const void*>(&quant_dot_mma_kernel<false>);
  const int smem = static_cast<int>(sizeof(QdSmem));
  *st = QZ_ERR_CUDA;
  if (!set_dyn_smem(k, smem)) return true;
  if (ksplit > 1 && launch_zero_z(in.z, in.ld_z, in.n0, n1, s) != QZ_OK) return true;
  const int grid = grid_for(k, a.nitems, s, smem);
  if (g64) quant_dot_mma_kernel<true><<<grid, kThreads, smem, s>>>(a, n1, yvec);
  else quant_dot_mma_kernel<false><<<grid, kThreads, smem, s>>>(a, n1, yvec);
  *st = launch_status();
  return true;
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
  if (a.ksplit > 1 && launch_zero_z(a.z, a.ld_z, a.n0, N1, s) != QZ_OK) return QZ_ERR_CUDA;
  const int grid = grid_for(reinterpret_cast<const void*>(k),
                            (nblocks * a.ksplit + kWarps - 1) / kWarps, s);
  k<<<grid, kThreads, 0, s>>>(a, yvec);
  return launch_status();
}

// n1 <= 8 columns: the tensor-core (mma.sync) form or the FMA form
qz_status quant_dot_few(const uint32_t* w, const float* scales, const uint32_t* shifts, int64_t n0, int64_t mid,
                        int64_t group, const void* y, int64_t ld_y, int64_t n1, float* z, int64_t ld_z,
                        cudaStream_t s) {
  const QdArgs a{w, scales, shifts, static_cast<const uint16_t*>(y), z, n0, mid, group, ld_y, ld_z, 1, 0};
  const bool yvec = reinterpret_cast<uintptr_t>(y) % 16 == 0 && ld_y % 8 == 0;
  qz_status st = QZ_OK;
  if (group % 16 == 0 && mid % 64 == 0 && reinterpret_cast<uintptr_t>(w) % 16 == 0 &&
      run_mma(a, static_cast<int>(n1), yvec && n1 == 8, s, &st))
    return st;
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

}  // namespace

qz_status launch_zero_z(float* z, int64_t ld_z, int64_t n0, int64_t n1, cudaStream_t s) {
  const int64_t n = n0 * n1;
  if (n == 0) return QZ_OK;
  const int64_t ctas = std::min<int64_t>((n + kThreads - 1) / kThreads, static_cast<int64_t>(sm_count()) * 8);
  zero_z_kernel<<<static_cast<int>(ctas), kThreads, 0, s>>>(z, ld_z, n0, static_cast<int>(n1));
  return launch_status();
}

qz_status launch_quant_dot(const uint32_t* w, const float* scales, const uint32_t* shifts,
                           int64_t n0, int64_t mid, int64_t group, const void* y, int64_t ld_y,
                           int64_t n1, float* z, int64_t ld_z, cudaStream_t s) {
  if (n1 <= 8) return quant_dot_few(w, scales, shifts, n0, mid, group, y, ld_y, n1, z, ld_z, s);
  if (quant_dot_tc_applicable(w, n0, mid, group, y, ld_y, n1))
    return launch_quant_dot_tc(w, scales, shifts, n0, mid, group, y, ld_y, n1, z, ld_z, s);
  // shapes the tensor-memory kernel does not take (groups that are not a multiple of 16,
  // unaligned activations): blocks of 8 columns, each streaming the weights once more
  for (int64_t k = 0; k < n1; k += 8) {
    const qz_status st = quant_dot_few(w, scales, shifts, n0, mid, group, static_cast<const uint16_t*>(y) + k,
                                       ld_y, std::min<int64_t>(8, n1 - k), z + k, ld_z, s);
    if (st != QZ_OK) return st;
  }
  return QZ_OK;
}

}  // namespace qz
