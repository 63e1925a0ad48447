// qz_qdot_tc.cu -- the quantized matrix product of the blog's "Puzzles 12 Quantized Matrix
// Mult" (section of its "Triton" post) for many activation columns, on the sm_103a tensor
// cores (tcgen05.mma, accumulators in tensor memory):
//     z[j][k] = sum_l sc[j][l/g] (w[j][l] - sh[j][l/g]) y[l][k]
// with 4-bit weights w (8 per 32-bit word, low nibble first), one fp32 scale and one 4-bit
// shift per group of g weights along l, and bf16 activations y [mid, n1].
//
// With many columns (prefill-sized batches) the product does 2 n1 flops per weight and is
// a dense contraction.  The sum is regrouped as sum over groups of sc * P_g with
// P_g = sum_{l in g} (w - sh) y: w - sh is an integer in [-15, 15], exact in bf16, and every
// product with a bf16 y is exact in fp32, so P_g runs on the tensor cores (kind::f16, bf16
// operands, fp32 accumulation) and the scale is applied by one fp32 FMA per output and
// group, keeping the result within the bound include/qz.h states.
//
// One CTA per SM, persistent over work items (a tile of 128 weight rows x up to 256
// activation columns, times one slice of l when the tiles are too few to fill the GPU).
// Roles (warp-specialised, every wait bounded in time):
//   warp 0        lane 0 streams each 64-wide l-step of y into a ring of kYStages shared-
//                 memory stages by TMA: up to four 64 x 64 bf16 boxes (128-byte swizzle,
//                 activation columns contiguous: the MMA's "MN-major" B operand).  The warp
//                 also owns the tensor-memory allocation.
//   warp 1        lane 0 issues the MMAs: four 128 x N x 16 steps per stage into one of two
//                 tensor-memory buffers of 256 fp32 columns, a new buffer at every group
//                 boundary (and every 1024 values of a longer group), commits each stage's
//                 completion to the "empty" barriers of both rings (after the next stage's
//                 first MMA) and each finished group to "P full".
//   decoders      warps 2, 3, 4 and 6 (groups of 64 and more; one weight row per thread)
//                 or warps 2 and 3 (shorter groups; two rows per thread), never a warp on
//                 the MMA warp's scheduler (w % 4 == 1).  Each thread copies its rows'
//                 code words itself (cp.async, kRawAhead stages ahead), turns every word
//                 into eight bf16 values w - sh (nibbles split by mask, paired by a byte
//                 permute, OR-ed into bf16 128 + w, one bf16x2 add of -(128 + sh)) and
//                 stores them in a ring of kAStages stages in the MMA's K-major 128-byte
//                 swizzled layout, then signals "A full".  The decoders run ahead of the
//                 MMAs independently of the activation copies.
//   epilogue      the 16 warps after them (8-23, or 4-19): warp w reads tensor-memory lanes
//                 32 (w % 4) .. + 31 (its rows) and 64 of the 256 columns; for every
//                 finished group it adds sc * P into its 64 fp32 outputs (packed FMAs),
//                 frees the buffer, and at the end of the item stores z (16-byte stores, or
//                 reductions when the item is one slice of several).
#include <cuda.h>  // CUtensorMap and its enumerators (types only; the encoder is looked up)
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "qz_device.cuh"
#include "qz_internal.h"
#include "qz_pipe.cuh"

namespace qz {
namespace {

constexpr int kBM = 128;        // weight rows per tile (MMA M, tensor-memory lanes)
constexpr int kBN = 256;        // activation columns per tile (MMA N at most)
constexpr int kBK = 64;         // l per stage (one 128-byte swizzle row of bf16)
constexpr int kYStages = 5;     // activation boxes in flight (TMA ring)
constexpr int kAStages = 3;     // decoded weight stages (decoder ring)
constexpr int kRawAhead = 3;    // code-word stages a decoder copies ahead of its decoding
constexpr int kRawStages = kRawAhead + 1;
constexpr int kEpiWarps = 16;
constexpr int kFirstDec = 2;
// Warp layout for D decoder warps (two or four: see quant_dot_tc_kernel).  A warp runs on
// scheduler (SM sub-partition) warp % 4, and an MMA is slowed by every busy warp that
// shares the issuing warp's scheduler (measured: 128 cycles per 128 x 256 x 16 MMA alone,
// 210 with four warps of dependent FMAs beside it, 586 with four warps running a long
// unrolled body; the same warps on the other three schedulers, or warps polling a barrier,
// cost nothing).  So no decoder is a warp w with w % 4 == 1, the MMA warp's scheduler: the
// decoders are the first D warps of [2, kFirstEpi) outside it, and the others idle.  The
// epilogue warps must cover all four schedulers (a warp reads tensor-memory lanes
// 32 (w % 4) .. + 31 only), and their work is kept short.
template <int D>
struct TcShape {
  static constexpr int kDecWarps = D;
  static constexpr int kDecRows = kBM / (32 * D);  // weight rows per decoder thread
  static constexpr int kFirstEpi = D == 2 ? 4 : 8;
  static constexpr int kThreads = 32 * (kFirstEpi + kEpiWarps);
  // decoder index of warp w in [2, kFirstEpi), -1 for an idle warp
  static __device__ __forceinline__ int dec_of(int w) {
    if ((w & 3) == 1) return -1;
    const int d = (w - kFirstDec) - (w - kFirstDec) / 4;  // less the warps 5, 9, ... below w
    return d < D ? d : -1;
  }
};
static_assert(TcShape<2>::kFirstEpi % 4 == 0 && TcShape<4>::kFirstEpi % 4 == 0, "epilogue quarters by warp % 4");
constexpr uint32_t kSlabBytes = 64 * kBK * 2;    // one 64-column box of y: 8 KiB
constexpr uint32_t kYBytes = 4 * kSlabBytes;     // 32 KiB
constexpr uint32_t kABytes = kBM * kBK * 2;      // 16 KiB of decoded bf16 weights
constexpr uint32_t kRawBytes = kBM * kBK / 2;    // 4 KiB of code words
constexpr uint32_t kAOff = kYStages * kYBytes;   // multiples of 1 KiB
constexpr uint32_t kRawOff = kAOff + kAStages * kABytes;
constexpr uint32_t kSmemTc = kRawOff + kRawStages * kRawBytes + 1024;  // + alignment slack
constexpr int kPieceCap = 1024;  // values of one group accumulated per tensor-memory buffer
constexpr uint32_t kTmemCols = 512;  // two buffers of 256 fp32 columns
constexpr uint64_t kTcWaitNs = 1000000000ull;  // 1 s: far beyond any step's latency

struct TcParams {
  CUtensorMap tmap_y;  // bf16 y [mid rows][n1 columns], box 64 x 64, 128-byte swizzle
  const uint32_t* w;
  const float* scales;
  const uint32_t* shifts;
  float* z;
  int64_t ld_z;
  int n0, n1, mid, group, ng, sw;
  // items [0, n_full) are whole tiles 0 .. n_full - 1; every later tile is split along l
  // into ksplit slices of slice_stages stages (the last one shorter), one item each
  int tiles_n, n_full, ksplit, slice_stages, stages_total, items;
};

// ---- small PTX wrappers -----------------------------------------------------------------
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// D[tmem] (+)= A[smem] * B[smem] for one 128 x N x 16 step
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc ? 1u : 0u)
      : "memory");
}
// 16 consecutive fp32 columns of this thread's tensor-memory lane, as 8 fp32 pairs (the
// operands of the packed FMAs of the epilogue)
__device__ __forceinline__ void tmem_ld16_pairs(uint32_t taddr, uint64_t (&v)[8]) {
  asm volatile(
      "{\n\t.reg .b32 r<16>;\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {r0,r1,r2,r3,r4,r5,r6,r7,r8,r9,r10,r11,r12,r13,r14,r15}, [%8];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n\t"
      "mov.b64 %0, {r0, r1};\n\tmov.b64 %1, {r2, r3};\n\tmov.b64 %2, {r4, r5};\n\tmov.b64 %3, {r6, r7};\n\t"
      "mov.b64 %4, {r8, r9};\n\tmov.b64 %5, {r10, r11};\n\tmov.b64 %6, {r12, r13};\n\tmov.b64 %7, {r14, r15};\n\t}"
      : "=l"(v[0]), "=l"(v[1]), "=l"(v[2]), "=l"(v[3]), "=l"(v[4]), "=l"(v[5]), "=l"(v[6]), "=l"(v[7])
      : "r"(taddr)
      : "memory");
}
// 8 consecutive fp32 columns, as 4 fp32 pairs (keeps the four-decoder kernel's epilogue
// within the 80 registers a thread has there)
__device__ __forceinline__ void tmem_ld8_pairs(uint32_t taddr, uint64_t (&v)[4]) {
  asm volatile(
      "{\n\t.reg .b32 r<8>;\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {r0,r1,r2,r3,r4,r5,r6,r7}, [%4];\n\t"
      "tcgen05.wait::ld.sync.aligned;\n\t"
      "mov.b64 %0, {r0, r1};\n\tmov.b64 %1, {r2, r3};\n\tmov.b64 %2, {r4, r5};\n\tmov.b64 %3, {r6, r7};\n\t}"
      : "=l"(v[0]), "=l"(v[1]), "=l"(v[2]), "=l"(v[3])
      : "r"(taddr)
      : "memory");
}
// 16 bytes of z from two fp32 pairs: a store, or (a slice of several) a reduction
__device__ __forceinline__ void st_pairs(float* dst, uint64_t a, uint64_t b) {
  asm volatile("st.global.v2.b64 [%0], {%1, %2};" ::"l"(dst), "l"(a), "l"(b) : "memory");
}
__device__ __forceinline__ void red_pairs(float* dst, uint64_t a, uint64_t b) {
  asm volatile(
      "{\n\t.reg .f32 f<4>;\n\tmov.b64 {f0, f1}, %1;\n\tmov.b64 {f2, f3}, %2;\n\t"
      "red.global.add.v4.f32 [%0], {f0, f1, f2, f3};\n\t}" ::"l"(dst),
      "l"(a), "l"(b)
      : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ uint4 lds128_tc(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
  return v;
}

// Shared-memory matrix descriptor of tcgen05 (start address, leading and stride byte
// offsets in 16-byte units, descriptor version 1, 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(lbo >> 4) << 16) |
         (static_cast<uint64_t>(sbo >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, A K-major, B MN-major,
// N = n columns, M = 128.
__device__ __forceinline__ uint32_t idesc_bf16(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(kBM >> 4) << 24);
}

// Bounded wait on phase `parity` of a barrier; gives up (and raises the CTA's abort flag)
// after kTcWaitNs, or at once when another role has given up already.
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kTcWaitNs) {
      *abort = 1;
      return false;
    }
  }
  return true;
}

// The work item's tile and l range.
struct Item {
  int m0, nb, st0, nst;  // first weight row, first column, first stage, stages
  int nslab;             // 64-column boxes of y that hold columns < n1 (1 .. 4)
};
// Item `it` is one slice of several (its outputs are added into z).
__device__ __forceinline__ bool item_split(const TcParams& p, int it) { return it >= p.n_full && p.ksplit > 1; }
__device__ __forceinline__ Item item_of(const TcParams& p, int it) {
  Item r;
  int t = it, s = 0;
  if (it >= p.n_full) {
    const int j = it - p.n_full;
    t = p.n_full + j / p.ksplit;
    s = j % p.ksplit;
  }
  const bool split = item_split(p, it);
  r.m0 = (t / p.tiles_n) * kBM;
  r.nb = (t % p.tiles_n) * kBN;
  r.st0 = split ? s * p.slice_stages : 0;
  r.nst = split ? min(p.slice_stages, p.stages_total - r.st0) : p.stages_total;
  r.nslab = min(4, (p.n1 - r.nb + 63) / 64);
  return r;
}

__device__ __forceinline__ void cp_async16_tc(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Walks the (item, stage) sequence of one CTA.
// Walks the (item, stage) sequence of one CTA; the item's fields are computed once per item
// (item_of divides by run-time values).
struct Cursor {
  int it, st, nst, m0, st0;
  bool valid;
  __device__ __forceinline__ void load(const TcParams& p) {
    valid = it < p.items;
    if (valid) {
      const Item I = item_of(p, it);
      nst = I.nst;
      m0 = I.m0;
      st0 = I.st0;
    } else {
      nst = 0;
    }
  }
  __device__ __forceinline__ void start(const TcParams& p, int first) {
    it = first;
    st = 0;
    load(p);
  }
  __device__ __forceinline__ void next(const TcParams& p, int step) {
    if (++st < nst) return;
    it += step;
    st = 0;
    load(p);
  }
};

// DEC decoder warps: four for groups of 64 and more (4096^3: group 128 345 -> 296 us when
// introduced; group 64 282 -> 264 us once the decode was straight-line); with their 768
// threads (80 registers each) the epilogue's 64 accumulators spill a little, which costs
// more than the extra decoders gain when every 16 or 32 values end a group (group 32:
// 348 -> 445 us), so those run with two (640 threads, 96 registers).
//
// GW: code words per group when a stage's groups sit at fixed places in it -- 8 for every
// group that is a multiple of 64 values (a stage lies inside one group), 4 for groups of
// 32, 2 for groups of 16 (2 or 4 whole groups a stage) -- so the decode of a stage is
// straight-line code; 0 for the other groups (48, 80, ...), whose boundaries move from
// stage to stage.
template <int DEC, int GW>
__global__ void __launch_bounds__(TcShape<DEC>::kThreads, 1) quant_dot_tc_kernel(const __grid_constant__ TcParams p) {
  constexpr int kDecWarps = TcShape<DEC>::kDecWarps, kDecRows = TcShape<DEC>::kDecRows;
  constexpr int kFirstEpi = TcShape<DEC>::kFirstEpi;
  // tensor-memory columns per epilogue load: 16 with the 96 registers of the two-decoder
  // layout (half the load waits), 8 within the 80 of the four-decoder one
  constexpr int kLdCols = DEC == 2 ? 16 : 8;
  extern __shared__ uint8_t tc_smem_raw[];
  __shared__ __align__(8) uint64_t yfull_bar[kYStages], yempty_bar[kYStages];
  __shared__ __align__(8) uint64_t afull_bar[kAStages], aempty_bar[kAStages];
  __shared__ __align__(8) uint64_t pfull_bar[2], pempty_bar[2], drain_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t base = (smem_addr(tc_smem_raw) + 1023u) & ~1023u;  // 1 KiB-aligned stages
  const auto y_of = [&](int s) { return base + static_cast<uint32_t>(s) * kYBytes; };
  const auto a_of = [&](int s) { return base + kAOff + static_cast<uint32_t>(s) * kABytes; };
  const auto raw_of = [&](int s) { return base + kRawOff + static_cast<uint32_t>(s) * kRawBytes; };

  if (tid == 0) {
    for (int s = 0; s < kYStages; ++s) {
      mbar_init(smem_addr(&yfull_bar[s]), 1);
      mbar_init(smem_addr(&yempty_bar[s]), 1);
    }
    for (int s = 0; s < kAStages; ++s) {
      mbar_init(smem_addr(&afull_bar[s]), kDecWarps);
      mbar_init(smem_addr(&aempty_bar[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_addr(&pfull_bar[b]), 1);
      mbar_init(smem_addr(&pempty_bar[b]), kEpiWarps);
    }
    mbar_init(smem_addr(&drain_bar), 1);
    mbar_init_fence();
    s_abort = 0;
  }
  if (warp == 0) {  // the whole warp allocates the two accumulator buffers
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int first_item = blockIdx.x, item_step = gridDim.x;

  if (warp == 0) {
    // ---------------- TMA producer of the activation ring: lane 0 alone ----------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int inflight = 0;  // stages issued and not yet known to have landed (for the drain)
      for (int it = first_item; it < p.items && !s_abort; it += item_step) {
        const Item I = item_of(p, it);
        for (int st = 0; st < I.nst; ++st) {
          if (!tc_wait(smem_addr(&yempty_bar[stage]), phase ^ 1u, &s_abort)) break;
          const uint32_t fb = smem_addr(&yfull_bar[stage]);
          const int l0 = (I.st0 + st) * kBK;
          mbar_expect_tx(fb, kSlabBytes * static_cast<uint32_t>(I.nslab));
          for (int sl = 0; sl < I.nslab; ++sl)
            tma_load_2d(y_of(stage) + sl * kSlabBytes, &p.tmap_y, I.nb + 64 * sl, l0, fb);
          inflight = min(inflight + 1, kYStages);
          if (++stage == kYStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (s_abort) {
        // let the copies already issued land before the shared memory is released: the
        // last `inflight` stages before `stage` (bounded waits; a timeout just ends it)
        for (int k = 1; k <= inflight; ++k) {
          const int s = (stage - k + kYStages) % kYStages;
          const uint32_t ph = (stage - k < 0) ? (phase ^ 1u) : phase;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(smem_addr(&yfull_bar[s]), ph) && globaltimer_ns() - t0 < kTcWaitNs) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer: lane 0 alone, the rest of the warp waits at the end ----
    // An MMA is taken by the tensor core only when the one before it has started, so at
    // most about two MMAs are queued while this thread works, and everything between two
    // MMAs leaves the tensor core idle once those have run.  So the loop is software-
    // pipelined: the next stage's "full" barriers are waited for before the stage's last
    // MMA, and a stage's "empty" barriers are signalled after the next stage's first MMA
    // (a commit tracks every MMA before it, so this frees the stage slightly later, which
    // the ring depths absorb).  The piece boundaries come from a countdown of 16-wide
    // steps and a running group boundary.
    if (lane == 0) {
      int ys = 0, as = 0, buf = 0, pys = 0, pas = 0;
      uint32_t yph = 0, aph = 0, pe_bits = 3u;  // bit b: parity of the next wait on "P empty" b
      bool issued = false;
      bool ready = false;  // this stage's "full" barriers were waited for in the stage before
      bool pend = false;   // stage (pys, pas) is read and its "empty" barriers not yet signalled
      for (int it = first_item; it < p.items && !s_abort; it += item_step) {
        const Item I = item_of(p, it);
        const uint32_t idesc = idesc_bf16(64 * I.nslab);
        const int l_end = (I.st0 + I.nst) * kBK;
        int l = I.st0 * kBK;
        int gb = (l / p.group + 1) * p.group;  // the next group boundary after l
        int left = 0;  // 16-wide steps of the open piece still to come (0: a new piece starts)
        bool open = false, acc = false, ok = true;
        for (int st = 0; st < I.nst && ok; ++st) {
          if (!ready && (!tc_wait(smem_addr(&yfull_bar[ys]), yph, &s_abort) ||
                         !tc_wait(smem_addr(&afull_bar[as]), aph, &s_abort)))
            break;
          ready = false;
          tc_fence_after();
          // A: rows of 128 bytes, 8-row groups 1 KiB apart, +32 bytes per 16 values of l;
          // B: 64-column boxes 8 KiB apart, 8-row groups of l 1 KiB apart, +2 KiB per 16 l
          const uint64_t ad0 = smem_desc_sw128(a_of(as), 16u, 1024u);
          const uint64_t bd0 = smem_desc_sw128(y_of(ys), kSlabBytes, 1024u);
          const int ys1 = ys + 1 == kYStages ? 0 : ys + 1, as1 = as + 1 == kAStages ? 0 : as + 1;
          const uint32_t yph1 = ys1 == 0 ? yph ^ 1u : yph, aph1 = as1 == 0 ? aph ^ 1u : aph;
          const bool more = st + 1 < I.nst;  // the next stage belongs to this item
#pragma unroll
          for (int j = 0; j < kBK / 16; ++j, l += 16) {
            if (j == 1 && pend) {  // the stage before is read: free it in both rings
              tc_commit(smem_addr(&yempty_bar[pys]));
              tc_commit(smem_addr(&aempty_bar[pas]));
              pend = false;
            }
            if (j == kBK / 16 - 1 && more) {  // the next stage, while two MMAs are queued
              if (!tc_wait(smem_addr(&yfull_bar[ys1]), yph1, &s_abort) ||
                  !tc_wait(smem_addr(&afull_bar[as1]), aph1, &s_abort)) {
                ok = false;
                break;
              }
              ready = true;
            }
            // where a piece can start: groups that are multiples of 64 values begin at a
            // stage, groups of 32 at every other 16-wide step, groups of 16 at every step;
            // other groups anywhere.  Only those places carry the piece code.
            const bool may_start = GW == 0 || GW == 2 || (GW == 4 && (j & 1) == 0) || (GW == 8 && j == 0);
            if (may_start && left == 0) {  // a new piece: the end of its group (and of each 1024 values)
              if (open) {
                tc_commit(smem_addr(&pfull_bar[buf]));
                buf ^= 1;
              }
              if (!tc_wait(smem_addr(&pempty_bar[buf]), (pe_bits >> buf) & 1u, &s_abort)) {
                ok = false;
                break;
              }
              pe_bits ^= 1u << buf;
              tc_fence_after();
              int nxt = min(l_end, gb);
              if (p.group > kPieceCap) nxt = min(nxt, (l / kPieceCap + 1) * kPieceCap);
              if (nxt == gb) gb += p.group;
              left = (nxt - l) / 16;
              open = true;
              acc = false;
            }
            tc_mma(tmem + static_cast<uint32_t>(buf) * kBN, ad0 + 2u * j, bd0 + 128u * j, idesc, acc);
            acc = true;
            issued = true;
            --left;
          }
          if (!ok) break;
          pend = true;  // both slots are free once these MMAs have read them
          pys = ys;
          pas = as;
          ys = ys1;
          yph = yph1;
          as = as1;
          aph = aph1;
        }
        if (s_abort || !ok) break;
        if (open) {
          tc_commit(smem_addr(&pfull_bar[buf]));
          buf ^= 1;
        }
      }
      if (pend && !s_abort) {
        tc_commit(smem_addr(&yempty_bar[pys]));
        tc_commit(smem_addr(&aempty_bar[pas]));
      }
      if (issued) {  // every MMA issued has completed before tensor memory is released
        tc_commit(smem_addr(&drain_bar));
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_addr(&drain_bar), 0u) && globaltimer_ns() - t0 < kTcWaitNs) {
        }
      }
    }
    __syncwarp();
  } else if (warp < kFirstEpi && TcShape<DEC>::dec_of(warp) >= 0) {
    // ---------------- decoders: code words -> bf16 (w - sh), swizzled K-major ----------------
    // Each thread owns one row (two when there are two decoder warps) of every stage.  It
    // copies their code words itself (cp.async, kRawAhead stages ahead, into its own slots
    // of a small ring: no other thread touches them, so its own wait_group is the only
    // synchronisation), keeps the shift word of the current group and the one after it in
    // registers, and fills the decoded-weight ring, which the MMA warp frees stage by stage.
    const int dt = 32 * TcShape<DEC>::dec_of(warp) + lane;  // rows dt + 32 kDecWarps h, h < kDecRows
    const int wpr = p.mid / 8;
    const int wpg = p.group / 8;          // code words per group (group % 16 == 0)
    Cursor pre;                           // the stage whose code words are copied next
    pre.start(p, first_item);
    const auto issue_raw = [&](int slot) {
      if (pre.valid) {
#pragma unroll
        for (int h = 0; h < kDecRows; ++h) {
          const int r = dt + 32 * kDecWarps * h, row = pre.m0 + r;
          if (row < p.n0) {
            const uint32_t* src = p.w + static_cast<int64_t>(row) * wpr + (pre.st0 + pre.st) * (kBK / 8);
            // the first 16 bytes of every row, then the second 16: a warp's 16-byte loads
            // below are then consecutive (a row-major 32-byte stride is a 2-way conflict)
            cp_async16_tc(raw_of(slot) + 16u * r, src);
            cp_async16_tc(raw_of(slot) + 16u * (kBM + r), src + 4);
          }
        }
        pre.next(p, item_step);
      }
      asm volatile("cp.async.commit_group;" ::: "memory");  // empty groups keep the count uniform
    };
#pragma unroll
    for (int k = 0; k < kRawAhead; ++k) issue_raw(k);
    int f = 0, as = 0;
    uint32_t aph = 0;
    for (int it = first_item; it < p.items && !s_abort; it += item_step) {
      const Item I = item_of(p, it);
      int widx[kDecRows];
      uint32_t wcur[kDecRows], wnxt[kDecRows];
      const int gfirst = I.st0 * (kBK / 8) / wpg;
#pragma unroll
      for (int h = 0; h < kDecRows; ++h) {
        const int row = I.m0 + dt + 32 * kDecWarps * h;
        const uint32_t* sr = p.shifts + static_cast<int64_t>(row < p.n0 ? row : 0) * p.sw;
        widx[h] = gfirst >> 3;
        wcur[h] = row < p.n0 ? __ldg(sr + widx[h]) : 0u;
        wnxt[h] = (row < p.n0 && widx[h] + 1 < p.sw) ? __ldg(sr + widx[h] + 1) : 0u;
      }
      // group of the stage's first code word and the words left in that group, advanced
      // stage by stage
      int g0 = gfirst, left0 = (gfirst + 1) * wpg - I.st0 * (kBK / 8);
      bool ok = true;
      for (int st = 0; st < I.nst; ++st, ++f) {
        issue_raw((f + kRawAhead) % kRawStages);
        asm volatile("cp.async.wait_group %0;" ::"n"(kRawAhead) : "memory");  // stage f's words are in
        const uint32_t raw = raw_of(f % kRawStages);
        if (!__all_sync(kFull, tc_wait(smem_addr(&aempty_bar[as]), aph ^ 1u, &s_abort))) {
          ok = false;
          break;
        }
#pragma unroll
        for (int h = 0; h < kDecRows; ++h) {
          const int r = dt + 32 * kDecWarps * h;
          const int row = I.m0 + r;
          uint32_t cw[8];
          if (row < p.n0) {
            const uint4 c0 = lds128_tc(raw + 16u * r);
            const uint4 c1 = lds128_tc(raw + 16u * (kBM + r));
            cw[0] = c0.x; cw[1] = c0.y; cw[2] = c0.z; cw[3] = c0.w;
            cw[4] = c1.x; cw[5] = c1.y; cw[6] = c1.z; cw[7] = c1.w;
          } else {
#pragma unroll
            for (int c = 0; c < 8; ++c) cw[c] = 0u;
          }
          const uint32_t arow = a_of(as) + 128u * r;
          constexpr int NG = GW ? 8 / GW : 1;  // groups of the stage with fixed places
          uint32_t addcs[NG];  // their bf16 pairs (-(128 + sh), -(128 + sh))
          if constexpr (GW != 0) {
            // the stage's NG groups g0 .. g0 + NG - 1 share one shift word (g0 is a
            // multiple of NG), and the word advances by at most one a stage
            if ((g0 >> 3) != widx[h]) {
              widx[h] = g0 >> 3;
              wcur[h] = wnxt[h];
              wnxt[h] = (row < p.n0 && widx[h] + 1 < p.sw)
                            ? __ldg(p.shifts + static_cast<int64_t>(row) * p.sw + widx[h] + 1)
                            : 0u;
            }
#pragma unroll
            for (int k = 0; k < NG; ++k)
              addcs[k] = 0xC300C300u + 0x00010001u * ((wcur[h] >> (4 * ((g0 + k) & 7))) & 0xFu);
          }
          int g = g0, left = left0;  // GW = 0: group of word c, and its words still to come
          uint32_t addc = 0u;        // bf16 pair (-(128 + sh), -(128 + sh)) of group g
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            if constexpr (GW != 0) {
              addc = addcs[c / GW];
            } else if (c == 0 || left == 0) {
              if (c != 0) {
                ++g;
                left = wpg;
              }
              if ((g >> 3) != widx[h]) {  // groups advance one at a time: the next word
                widx[h] = g >> 3;
                wcur[h] = wnxt[h];
                wnxt[h] = (row < p.n0 && widx[h] + 1 < p.sw)
                              ? __ldg(p.shifts + static_cast<int64_t>(row) * p.sw + widx[h] + 1)
                              : 0u;
              }
              const uint32_t sh = (wcur[h] >> (4 * (g & 7))) & 0xFu;
              addc = 0xC300C300u + 0x00010001u * sh;  // bf16 -(128 + sh): ulp 1 at 128
            }
            if constexpr (GW == 0) --left;
            // even nibbles (elements 0, 2, 4, 6) in bytes 0..3 of t0, odd ones in t1; value
            // pair q is bytes q of t0 and t1 side by side, OR 0x4300 in each half is the
            // bf16 128 + nibble, and one bf16x2 add of -(128 + sh) leaves w - sh exactly.
            // (Leaving the two byte masks to the OR below is one instruction less a word but
            // made the four-decoder kernel spill more: 226 -> 249 us.)
            const uint32_t t0 = cw[c] & 0x0F0F0F0Fu, t1 = (cw[c] >> 4) & 0x0F0F0F0Fu;
            uint32_t v[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t d, x;
              asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(t0), "r"(t1), "r"(0x0400u * 0x11u + q * 0x0101u));
              asm("lop3.b32 %0, %1, 0x000F000F, 0x43004300, 0xEA;" : "=r"(x) : "r"(d));  // (a & b) | c
              asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(v[q]) : "r"(x), "r"(addc));
            }
            sts128(arow + static_cast<uint32_t>(((c ^ (r & 7)) << 4)), v[0], v[1], v[2], v[3]);
          }
        }
        fence_proxy_async();  // generic-proxy stores -> visible to the tensor cores
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&afull_bar[as]));
        if (++as == kAStages) {
          as = 0;
          aph ^= 1u;
        }
        if constexpr (GW == 2 || GW == 4) {
          g0 += 8 / GW;
        } else {
          for (left0 -= kBK / 8; left0 <= 0; left0 += wpg) ++g0;
        }
      }
      if (!ok) break;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // no copy of this thread is left in flight
  } else if (warp >= kFirstEpi) {
    // ---------------- epilogue ----------------
    const int q = warp & 3;                 // tensor-memory lane quarter of this warp
    const int cq = (warp - kFirstEpi) >> 2; // its 64-column quarter of the tile
    const int r = 32 * q + lane;            // tile row of this thread
    uint32_t pf_bits = 0u;  // bit b: parity of the next wait on "P full" b
    // rows of z 16-byte aligned: vector stores
    const bool zvec = (reinterpret_cast<uintptr_t>(p.z) & 15u) == 0 && (p.ld_z & 3) == 0;
    int buf = 0;
    for (int it = first_item; it < p.items && !s_abort; it += item_step) {
      const Item I = item_of(p, it);
      const int row = I.m0 + r;
      const bool row_ok = row < p.n0;
      uint64_t z2[32];  // the 64 outputs of this thread as fp32 pairs
#pragma unroll
      for (int i = 0; i < 32; ++i) z2[i] = pk(0.0f, 0.0f);
      const int l_begin = I.st0 * kBK, l_end = l_begin + I.nst * kBK;
      int g = l_begin / p.group, gb = (g + 1) * p.group;  // group of l, its end
      bool ok = true;
      for (int l = l_begin; l < l_end;) {
        int nxt = min(l_end, gb);
        if (p.group > kPieceCap) nxt = min(nxt, (l / kPieceCap + 1) * kPieceCap);
        const float sc = row_ok ? __ldg(p.scales + static_cast<int64_t>(row) * p.ng + g) : 0.0f;
        const uint64_t sc2 = pk(sc, sc);
        if (!__all_sync(kFull, tc_wait(smem_addr(&pfull_bar[buf]), (pf_bits >> buf) & 1u, &s_abort))) {
          ok = false;
          break;
        }
        pf_bits ^= 1u << buf;
        tc_fence_after();
        const uint32_t ta = tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(buf * kBN + 64 * cq);
#pragma unroll
        for (int c = 0; c < 64 / kLdCols; ++c) {  // z = fl32(sc * P + z) for each element, two per FMA
          uint64_t v[kLdCols / 2];
          if constexpr (kLdCols == 16) tmem_ld16_pairs(ta + 16u * c, v);
          else tmem_ld8_pairs(ta + 8u * c, v);
#pragma unroll
          for (int i = 0; i < kLdCols / 2; ++i) z2[(kLdCols / 2) * c + i] = fma2(v[i], sc2, z2[(kLdCols / 2) * c + i]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&pempty_bar[buf]));
        buf ^= 1;
        l = nxt;
        if (l == gb) {
          ++g;
          gb += p.group;
        }
      }
      if (!ok) break;
      if (row_ok) {
        const bool split = item_split(p, it);  // recomputed here: one register less in the loop
        const int c0 = I.nb + 64 * cq;
        float* zr = p.z + static_cast<int64_t>(row) * p.ld_z + c0;
        const int nv = min(64, p.n1 - c0);
        if (nv == 64 && zvec) {  // 16-byte stores (or reductions): 64 contiguous bytes a pair
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            if (split) red_pairs(zr + 2 * i, z2[i], z2[i + 1]);
            else st_pairs(zr + 2 * i, z2[i], z2[i + 1]);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float z0, z1;
            upk(z2[i], z0, z1);
            if (split) {
              if (2 * i < nv) atomicAdd(zr + 2 * i, z0);
              if (2 * i + 1 < nv) atomicAdd(zr + 2 * i + 1, z1);
            } else {
              if (2 * i < nv) zr[2 * i] = z0;
              if (2 * i + 1 < nv) zr[2 * i + 1] = z1;
            }
          }
        }
      }
    }
  }

  // every role is done (or has given up) and every MMA has completed: release the
  // tensor memory, and report a give-up as NaN in this CTA's outputs
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
  if (s_abort && warp >= kFirstEpi) {
    const int q = warp & 3, cq = (warp - kFirstEpi) >> 2, r = 32 * q + lane;
    for (int it = first_item; it < p.items; it += item_step) {
      const Item I = item_of(p, it);
      const int row = I.m0 + r, c0 = I.nb + 64 * cq;
      if (row >= p.n0) continue;
      for (int i = 0; i < 64 && c0 + i < p.n1; ++i)
        p.z[static_cast<int64_t>(row) * p.ld_z + c0 + i] = __uint_as_float(0x7fc00000u);
    }
  }
}

// ---- host side ----------------------------------------------------------------------------
std::mutex g_encode_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::lock_guard<std::mutex> lock(g_encode_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode;
}

}  // namespace

bool quant_dot_tc_applicable(const uint32_t* w, int64_t n0, int64_t mid, int64_t group, const void* y,
                             int64_t ld_y, int64_t n1) {
  return n1 > 8 && group % 16 == 0 && mid % kBK == 0 && mid < (int64_t{1} << 30) && n0 < (int64_t{1} << 30) &&
         n1 < (int64_t{1} << 30) && ld_y % 8 == 0 && reinterpret_cast<uintptr_t>(y) % 16 == 0 &&
         reinterpret_cast<uintptr_t>(w) % 16 == 0;
}

qz_status launch_quant_dot_tc(const uint32_t* w, const float* scales, const uint32_t* shifts, int64_t n0,
                              int64_t mid, int64_t group, const void* y, int64_t ld_y, int64_t n1, float* z,
                              int64_t ld_z, cudaStream_t s) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return QZ_ERR_CUDA;
  TcParams p{};
  {  // y: dimension 0 = columns (contiguous), dimension 1 = l
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(n1), static_cast<cuuint64_t>(mid)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld_y) * 2};
    const cuuint32_t box[2] = {64, kBK}, es[2] = {1, 1};
    if (enc(&p.tmap_y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(y), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return QZ_ERR_CUDA;
  }
  const int sms = sm_count();
  const int64_t tiles_m = (n0 + kBM - 1) / kBM, tiles_n = (n1 + kBN - 1) / kBN;
  const int64_t tiles = tiles_m * tiles_n, stages_total = mid / kBK;
  // The whole waves of tiles run as they are; the tiles of the last, partly filled wave (all
  // of them when there are fewer tiles than SMs) are split along l into as many slices as
  // keep one slice per SM (k = floor(sms / tail)), of at least 256 values each, so that
  // wave takes 1/k of a tile's time.  Measured against splitting only when there are fewer
  // tiles than SMs (then into ceil(sms / tiles) slices): 4096^3 at groups of 128 (512
  // tiles, 56 in the last wave, k = 2) 228 -> 215 us, groups of 32 342 -> 312 us,
  // 32768 x 8192 x 2048 1436 -> 1409 us, 4096 x 4096 x 512 (64 tiles, k = 2 instead of 3)
  // 57 -> 43 us.
  const int64_t tail = tiles % sms;
  int64_t ksplit = 1;
  if (tail > 0) ksplit = std::max<int64_t>(1, std::min<int64_t>(sms / tail, stages_total / 4));
  const int64_t slice_stages = (stages_total + ksplit - 1) / ksplit;
  ksplit = (stages_total + slice_stages - 1) / slice_stages;
  const int64_t n_full = ksplit > 1 ? tiles - tail : tiles;
  const int64_t items = n_full + (tiles - n_full) * ksplit;
  if (items >= (int64_t{1} << 31)) return QZ_ERR_UNSUPPORTED;
  p.w = w;
  p.scales = scales;
  p.shifts = shifts;
  p.z = z;
  p.ld_z = ld_z;
  p.n0 = static_cast<int>(n0);
  p.n1 = static_cast<int>(n1);
  p.mid = static_cast<int>(mid);
  p.group = static_cast<int>(group);
  p.ng = static_cast<int>(mid / group);
  p.sw = static_cast<int>((mid / group + 7) / 8);
  p.tiles_n = static_cast<int>(tiles_n);
  p.n_full = static_cast<int>(n_full);
  p.ksplit = static_cast<int>(ksplit);
  p.slice_stages = static_cast<int>(slice_stages);
  p.stages_total = static_cast<int>(stages_total);
  p.items = static_cast<int>(items);
  const bool four = group >= 64;
  const int gw = group % 64 == 0 ? 8 : group == 32 ? 4 : group == 16 ? 2 : 0;
  void (*kern)(TcParams);
  if (four) kern = gw == 8 ? &quant_dot_tc_kernel<4, 8> : &quant_dot_tc_kernel<4, 0>;
  else if (gw == 8) kern = &quant_dot_tc_kernel<2, 8>;
  else if (gw == 4) kern = &quant_dot_tc_kernel<2, 4>;
  else if (gw == 2) kern = &quant_dot_tc_kernel<2, 2>;
  else kern = &quant_dot_tc_kernel<2, 0>;
  if (!set_dyn_smem(reinterpret_cast<const void*>(kern), static_cast<int>(kSmemTc))) return QZ_ERR_CUDA;
  if (ksplit > 1) {  // the split tiles add into z: zero their rows (from the first split tile's)
    const int64_t row0 = (n_full / tiles_n) * kBM;
    if (launch_zero_z(z + row0 * ld_z, ld_z, n0 - row0, n1, s) != QZ_OK) return QZ_ERR_CUDA;
  }
  const int grid = static_cast<int>(std::min<int64_t>(items, sms));
  kern<<<grid, four ? TcShape<4>::kThreads : TcShape<2>::kThreads, kSmemTc, s>>>(p);
  return launch_status();
}

}  // namespace qz
