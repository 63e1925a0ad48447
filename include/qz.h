/*
 * qz.h -- C ABI of libqz: quantize a 2-D tensor on a GB300 (sm_103a) GPU to symmetric INT8,
 * FP8 E4M3 / E5M2, MXFP4, NVFP4 or grouped symmetric INT4, dequantize it again, and reduce
 * the quantization error; dequantize asymmetric 4-bit grouped weights.
 *
 * The operations are the ones defined in the blog post "浅谈低精度浮点数" ("A brief talk
 * on low-precision floats", july-h5kf3.github.io column blog):
 *   - section "FP8": symmetric INT8, x^ = s * round(x / s), q in [-127, 127],
 *     s = alpha / 127 with alpha the largest magnitude; FP8 E4M3 and E5M2;
 *   - section "FP4 / MXFP4 / NVFP4": the E2M1 element values {0, 0.5, 1, 1.5, 2, 3, 4, 6},
 *     MXFP4 (32 values share one power-of-two E8M0 scale, s = 2^round(log2(A/6)), rounded
 *     up in practice), NVFP4 (16 values share one E4M3 scale, times one fp32 per-tensor
 *     scale: s_global = global_amax / (6 * 448), s_block = (block_amax / 6) / s_global,
 *     x^ = s_global * s_block * Q_E2M1(x / (s_global * s_block)));
 *   - same section, closing paragraph: symmetric INT4, q in [-7, 7], s = A / 7, analysed
 *     like INT8 (here one fp32 scale per group of block_size values along cols);
 *   - the error measures discussed there: |x - x^| and |x - x^| / |x|.
 * The asymmetric 4-bit group dequantization sc * (w - sh) is the one of the "Puzzles 12
 * Quantized Matrix Mult" section of the same blog's "Triton" post.
 * Packing of two FP4 codes per byte follows the "Puzzles 12 Quantized Matrix Mult" section
 * of the same blog's "Triton" post: element j of a packed word sits in bits [4j, 4j+4), so
 * the first element of a pair is the low nibble.
 *
 * Exact semantics (every result is bit-exact, error statistics aside):
 *   element step   v = fl32(x / s)  (IEEE binary32 division), then round to the nearest
 *                  grid value, ties to the code with an even last bit; values at or beyond
 *                  the format maximum saturate (INT8 127, E4M3 448, E5M2 57344, E2M1 6);
 *                  FP formats keep the sign of zero, INT8 has one zero (-128 never occurs).
 *   INT8 / FP8     s = fl32(alpha / qmax) with qmax = 127, 448 or 57344; alpha is the
 *                  largest |x| of the tensor (TENSOR) or of the row (ROW); s = 1 when that
 *                  quotient is 0.  UNIT uses s = 1.
 *   MXFP4          per 32-element block with largest magnitude A: t = fl32(A / 6);
 *                  k = smallest integer with 2^k >= t (QZ_SCALE_UP) or k = round(log2 t)
 *                  (QZ_SCALE_NEAREST), clamped to [-127, 127], k = -127 when t = 0;
 *                  scale code (E8M0, bias 127) = k + 127; v = x * 2^-k (exact).
 *                  UNIT uses k = 0.
 *   NVFP4          s_g = fl32(alpha / 2688) (1 when 0); per 16-element block
 *                  t = fl32(fl32(A / 6) / s_g); block code = smallest E4M3 value >= t,
 *                  saturated at 448 (QZ_SCALE_UP) or RNE-saturating E4M3 (QZ_SCALE_NEAREST);
 *                  s = fl32(s_g * decode(block code)); s = 0 gives signed-zero codes.
 *                  UNIT uses s_g = 1 and block code 0x38 (1.0).
 *   INT4           per group of block_size values with largest magnitude A: s = fl32(A / 7)
 *                  (1 when 0), q = RNE(fl32(x / s)) clamped to [-7, 7], one zero; stored as
 *                  a 4-bit two's complement nibble (-8 never occurs).
 *   dequantize     x^ = fl32(decode(q) * s), then converted to the output dtype (bf16 by
 *                  round-to-nearest-even, or fp32 as is).
 *   stats          e = fl32(x - x^) with the fp32 x^; sum_sq_err = sum e^2; mse =
 *                  sum_sq_err / n; max_abs_err = max |e| (exact); max_rel_err = max over
 *                  x != 0 of fl32(|e| / |x|) (exact).  sum_sq_err / mse are accumulated
 *                  with compensated fp32 per thread and fp64 across threads: relative
 *                  error below 1e-5.
 *
 * Layouts.  The high-precision tensor (x for quantize / stats, y for dequantize) is
 * [rows, cols] row-major with leading dimension ld >= cols, in elements.  Everything else
 * is dense row-major:
 *   codes   INT8 / FP8: rows * cols bytes; MXFP4 / NVFP4 / INT4: rows * cols / 2 bytes.
 *   scales  ROW: rows fp32; MXFP4: rows * cols / 32 E8M0 bytes; NVFP4: rows * cols / 16
 *           E4M3 bytes; INT4: rows * cols / block_size fp32; otherwise unused (may be NULL).
 *   tensor_scale  one fp32: s for TENSOR, s_g for NVFP4 BLOCK, 1 for UNIT.
 * Blocks run along cols.  MXFP4 needs cols % 32 == 0, NVFP4 cols % 16 == 0, INT4
 * cols % block_size == 0.
 *
 * Ownership and concurrency.  The caller allocates every buffer (all device memory except
 * the host pointer of qz_get_device_status).  The library allocates nothing, except a host
 * round-trip plan (qz_host_plan_create, at the end of this header); its only other
 * host-side state is a per-device cache of launch parameters (SM count, resident CTAs per
 * SM, shared-memory opt-ins), guarded by a mutex.  Every call is asynchronous on `stream`
 * (NULL = the legacy default stream); argument errors are returned synchronously, before
 * anything is enqueued.
 * Calls that share one workspace must be ordered on one stream.
 *
 * Alignment.  Pointers need only the natural alignment of their element type.  Fast
 * vectorised kernels are used when x / y and ld allow 16-byte (INT8 / FP8) or 32-byte
 * (MXFP4 / NVFP4) row access and codes are 16-byte aligned; other shapes run element-wise
 * kernels with the same results.
 *
 * Non-finite inputs (NaN, +-Inf) are outside the contract: the codes are unspecified and
 * bit 0 of the workspace status word is set (read it with qz_get_device_status).
 */
#ifndef QZ_H
#define QZ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define QZ_API __attribute__((visibility("default")))
#else
#define QZ_API
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* qz_stream_t;

typedef enum {
  QZ_OK = 0,
  QZ_ERR_NULL = 1,        /* a required pointer is NULL                                */
  QZ_ERR_ENUM = 2,        /* a descriptor field holds an unknown enumerator            */
  QZ_ERR_SHAPE = 3,       /* rows / cols / ld out of range, or cols % block_size != 0  */
  QZ_ERR_ALIGN = 4,       /* a pointer lacks the natural alignment of its element type */
  QZ_ERR_UNSUPPORTED = 5, /* a valid but unsupported combination (format x granularity) */
  QZ_ERR_CUDA = 6,        /* a kernel launch failed                                    */
  QZ_ERR_WORKSPACE = 7    /* workspace missing or smaller than qz_workspace_size()     */
} qz_status;

typedef enum {
  QZ_INT8 = 1, QZ_FP8_E4M3 = 2, QZ_FP8_E5M2 = 3, QZ_MXFP4 = 4, QZ_NVFP4 = 5, QZ_INT4 = 6
} qz_format;
typedef enum { QZ_BF16 = 1, QZ_F32 = 2 } qz_dtype;
typedef enum {
  QZ_GRAN_TENSOR = 1, /* one scale for the tensor (INT8 / FP8)                     */
  QZ_GRAN_ROW = 2,    /* one scale per row: per output channel / per token (INT8/FP8) */
  QZ_GRAN_BLOCK = 3,  /* per block along cols (MXFP4 32, NVFP4 16, INT4 block_size) */
  QZ_GRAN_UNIT = 4    /* scale 1: the bare element cast (all formats)              */
} qz_granularity;
typedef enum { QZ_ROUND_RNE = 0 } qz_elem_round;
typedef enum { QZ_SCALE_UP = 0, QZ_SCALE_NEAREST = 1 } qz_scale_round;

/* Status-word bits (qz_get_device_status). */
#define QZ_FLAG_NONFINITE_INPUT 0x1u /* a NaN or Inf element was read                   */
#define QZ_FLAG_BAD_AMAX 0x2u        /* a caller-supplied tensor amax was < 0 or NaN     */
#define QZ_FLAG_PIPELINE_TIMEOUT 0x4u /* a kernel gave up waiting for its own staged copy   */
                                      /* (never expected; re-initialise the workspace)   */

typedef struct {
  int32_t format;      /* qz_format                                                  */
  int32_t in_dtype;    /* qz_dtype of x (quantize, stats, amax)                      */
  int32_t granularity; /* qz_granularity                                             */
  int32_t block_size;  /* 32 for MXFP4, 16 for NVFP4, 16/32/64/128 for INT4, else 0  */
  int32_t elem_round;  /* QZ_ROUND_RNE                                               */
  int32_t scale_round; /* qz_scale_round (MXFP4 / NVFP4 BLOCK)                       */
  int64_t rows;        /* >= 0                                                       */
  int64_t cols;        /* >= 0                                                       */
  int64_t ld;          /* leading dimension of x / y in elements, >= cols            */
} qz_desc;

/* Error statistics, written to device memory by qz_quantize / qz_error_stats. */
typedef struct {
  double sum_sq_err;
  double mse;
  float max_rel_err;
  float max_abs_err;
  uint64_t n;
} qz_stats;

/* Human-readable name of a status code (static storage). */
QZ_API const char* qz_status_string(qz_status status);

/* Bytes of device workspace the calls below need for this descriptor (the same for every
 * descriptor of this library version).  The workspace must be zeroed once before its first
 * use (qz_workspace_init); the calls leave it ready for the next call. */
QZ_API size_t qz_workspace_size(const qz_desc* desc);

/* Zero `bytes` of workspace on `stream`. */
QZ_API qz_status qz_workspace_init(void* ws, size_t bytes, qz_stream_t stream);

/* Largest |x| of the tensor into *amax_dev (device fp32).  Sets QZ_FLAG_NONFINITE_INPUT
 * when a NaN / Inf is read.  Needs the workspace. */
QZ_API qz_status qz_amax(const qz_desc* desc, const void* x, float* amax_dev, void* ws,
                  qz_stream_t stream);

/* Quantize x into codes (+ scales, + tensor_scale_dev).
 *   tensor_amax_dev  optional device fp32: the alpha of TENSOR / NVFP4 BLOCK (the post
 *                    leaves open where NVFP4's global amax comes from); NULL = computed
 *                    here with an extra read of x.  Must be finite and >= 0.
 *   tensor_scale_dev written (one fp32) when non-NULL; required for TENSOR and NVFP4 BLOCK.
 *   stats_dev        optional: the error statistics of this quantization, fused into the
 *                    same pass (no extra read of x).
 *   ws               workspace (qz_workspace_size bytes); required when the amax is
 *                    computed or stats_dev is non-NULL, may be NULL otherwise. */
QZ_API qz_status qz_quantize(const qz_desc* desc, const void* x, void* codes, void* scales,
                      float* tensor_scale_dev, const float* tensor_amax_dev,
                      qz_stats* stats_dev, void* ws, qz_stream_t stream);

/* Quantize with a per-tensor scale taken from a previous tensor ("delayed" scaling), and
 * return this tensor's own amax for the next call.  The post leaves open where NVFP4's
 * global amax comes from (section "FP4 / MXFP4 / NVFP4"): this is the reading in which it
 * comes from an earlier step, so the quantize needs no extra read of x.
 *   amax_in_dev   device fp32, required for TENSOR and NVFP4 BLOCK (else ignored, may be
 *                 NULL): the alpha of the scale, exactly as tensor_amax_dev of qz_quantize.
 *                 Elements beyond it saturate, as the formats define.
 *   amax_out_dev  device fp32, required: max |x| of this tensor, bit-identical to what
 *                 qz_amax writes (QZ_FLAG_NONFINITE_INPUT on NaN / Inf).  On dense, 16-byte
 *                 aligned TENSOR / UNIT / BLOCK tensors it is folded into the quantize
 *                 kernel; elsewhere (ROW, strided or unaligned) it takes a separate read.
 *                 May alias amax_in_dev: the scale is read before amax_out is written.
 *   ws            workspace, required.
 * Everything else as qz_quantize (codes, scales, tensor_scale_dev, stats_dev). */
QZ_API qz_status qz_quantize_delayed(const qz_desc* desc, const void* x, void* codes, void* scales,
                                     float* tensor_scale_dev, const float* amax_in_dev,
                                     float* amax_out_dev, qz_stats* stats_dev, void* ws,
                                     qz_stream_t stream);

/* Dequantize codes (+ scales, + tensor_scale_dev) into y ([rows, cols], leading dimension
 * desc->ld) of dtype out_dtype.  desc->in_dtype is ignored. */
QZ_API qz_status qz_dequantize(const qz_desc* desc, const void* codes, const void* scales,
                        const float* tensor_scale_dev, void* y, int32_t out_dtype,
                        qz_stream_t stream);

/* Error statistics of existing codes against x, without writing anything but stats_dev. */
QZ_API qz_status qz_error_stats(const qz_desc* desc, const void* x, const void* codes,
                         const void* scales, const float* tensor_scale_dev,
                         qz_stats* stats_dev, void* ws, qz_stream_t stream);

/* qz_error_stats without a workspace argument, for callers that cannot allocate device
 * memory (code running under another framework's memory pool, paths on which cudaMalloc /
 * cudaFree and their device synchronisation are not allowed, plugins handed only their
 * input and output buffers).  The post has no counterpart; this is an interface matter.
 * Same arguments, results and argument errors as qz_error_stats otherwise.
 *   Scratch: a fixed array of qz_workspace_size() bytes (82 176 in this version) in device
 *   memory, part of the library module: every GPU that loads the library holds it until
 *   the process exits.  The statistics need no more scratch for larger tensors; a
 *   descriptor whose workspace would exceed the array is rejected with QZ_ERR_WORKSPACE.
 *   Allocation: none -- no cudaMalloc, cudaFree or allocating library call.
 *   First call on a device: looks up the array's device address (cudaGetSymbolAddress,
 *   with that device current) and caches it for the life of the device's context; make
 *   that first call before any stream capture on the device, and do not use this entry
 *   (or qz_error_stats_noalloc_status) across a cudaDeviceReset.
 *   Status: a NaN / Inf element sets QZ_FLAG_NONFINITE_INPUT in the array's status word,
 *   which keeps collecting flags until qz_error_stats_noalloc_status reads and clears it.
 *   Sharing: every call on a device uses the same array, which keeps what the previous
 *   call left (its completion counters return to 0 at the end of each call's kernel).
 *   Calls that overlap on the GPU (different streams, no ordering between them) race on
 *   the array and give wrong statistics. */
QZ_API qz_status qz_error_stats_noalloc(const qz_desc* desc, const void* x, const void* codes,
                                        const void* scales, const float* tensor_scale_dev,
                                        qz_stats* stats_dev, qz_stream_t stream);

/* Status flags (QZ_FLAG_* bits) that qz_error_stats_noalloc calls on the current device have
 * raised since the last call of this function, read into *flags_host and cleared, both in
 * order on `stream` behind the calls already enqueued there; then synchronizes `stream`.
 * Allocates nothing.  The post has no counterpart; an interface matter. */
QZ_API qz_status qz_error_stats_noalloc_status(uint32_t* flags_host, qz_stream_t stream);

/* Statistics of one tensor from the statistics of its parts: `parts` holds `count` records
 * (device, 8-byte aligned) written by qz_quantize / qz_error_stats over disjoint parts of
 * the tensor (row ranges, say, quantized as they arrive).  *out (device) gets the sum of
 * their sum_sq_err and n, mse = sum_sq_err / n (0 when n = 0), and the maximum of their
 * max_abs_err and max_rel_err -- the statistics the definitions above give for the whole
 * tensor (blocks never straddle a part, so the codes are the same), the sum of squares
 * within the same 1e-5 relative bound.  The sums run in fp64 in a fixed order, so equal
 * inputs give equal results.  `out` may be one of the parts.  count = 0 writes an empty
 * record; count < 0 is QZ_ERR_SHAPE.  One small kernel on `stream`; no workspace. */
QZ_API qz_status qz_stats_merge(const qz_stats* parts, int64_t count, qz_stats* out,
                                qz_stream_t stream);

/* Asymmetric 4-bit group dequantization ("Puzzles 12 Quantized Matrix Mult", Triton post):
 *   y[r][c] = fl32(sc[r][c / group] * (w[r][c] - sh[r][c / group])), w - sh exact.
 *   w       device, [rows, cols / 8] 32-bit words: 8 unsigned 4-bit codes each, element c
 *           in bits [4 (c % 8), 4 (c % 8) + 4) of word c / 8 (the puzzle's extract order)
 *   scales  device, [rows, cols / group] fp32
 *   shifts  device, [rows, ceil((cols / group) / 8)] 32-bit words: 8 unsigned 4-bit shifts
 *           each, group j in nibble j % 8 of word j / 8
 *   y       device, [rows, ld] of out_dtype (bf16 by RNE, or fp32), ld >= cols
 * Requires cols % 8 == 0, group > 0, cols % group == 0 (QZ_ERR_SHAPE otherwise); words and
 * scales 4-byte aligned.  Asynchronous on `stream`; needs no workspace. */
QZ_API qz_status qz_dequantize_asym4(const uint32_t* w, const float* scales,
                                     const uint32_t* shifts, int64_t rows, int64_t cols,
                                     int64_t group, void* y, int64_t ld, int32_t out_dtype,
                                     qz_stream_t stream);

/* The quantized matrix product of "Puzzles 12 Quantized Matrix Mult" (Triton post):
 *   z[j][k] = sum_l sc[j][l / group] * (w[j][l] - sh[j][l / group]) * y[l][k]
 *   w, scales, shifts  device, the weights [n0, mid] exactly as qz_dequantize_asym4 (rows =
 *                      n0, cols = mid): each weight is fl32(sc * (w - sh)), as that call writes
 *   y                  device, bf16 activations [mid, ld_y], ld_y >= n1, 2-byte aligned
 *   z                  device, fp32 [n0, ld_z], ld_z >= n1, 4-byte aligned
 * The sum runs in fp32 in an unspecified order.  With group % 16 == 0 it runs on the tensor
 * cores as sum over groups of sc * sum (w - sh) y: the integer factors w - sh are exact in
 * bf16, every product (w - sh) y is exact in fp32, and the scale is applied by one fp32 FMA
 * per output and group (and per 1024 values of a longer group).  Every z[j][k] is within
 *     E * 2^-24 * sum_l |weight * y|,   E = 34 ceil(g' / 16) + ceil(mid / g') + ceil(mid / 32)
 *                                            + ceil(mid / 256) + 24,   g' = min(group, 1024)
 * of the exact sum.  The 34 per 16 terms covers one tensor-core step c + sum of 16 exact
 * products whose addends are aligned to the largest one and cut to 24 bits (truncation)
 * and whose result is normalised with at most one more ulp: 16 addends lose under one ulp
 * of the largest each, 2^-23 = 2 * 2^-24 relative, and the normalisation two more.  The
 * other terms count the remaining fp32 roundings of the order used: one per weight
 * rounding, one per group FMA, one per partial sum of split rows (FMA form: one per term a
 * lane accumulates, mid / 32 at most, five in the warp reduction).
 * Forms by the number of activation columns:
 *   n1 <= 8   (decode, small batches): the packed weights are streamed once; the product is
 *             bound by HBM.  Tensor-core form by mma.sync when group % 16 == 0, mid % 64 == 0
 *             and w is 16-byte aligned; an FMA form otherwise.
 *   n1 > 8    (prefill-sized batches): a dense contraction on tcgen05 tensor cores with the
 *             partial sums in tensor memory, when group % 16 == 0, mid % 64 == 0, w and y
 *             16-byte aligned and ld_y % 8 == 0; otherwise blocks of 8 columns by the n1 <= 8
 *             forms (correct, but the weights are read once per block).
 * mid % 8 == 0, group > 0, mid % group == 0 (QZ_ERR_SHAPE); n1 < 2^30 (QZ_ERR_UNSUPPORTED).
 * Asynchronous on `stream`; needs no workspace.  A tcgen05 kernel that gives up waiting for
 * its own copies (never expected: every wait is bounded) writes NaN to the outputs of its
 * tiles instead of hanging. */
QZ_API qz_status qz_quant_dot(const uint32_t* w, const float* scales, const uint32_t* shifts,
                              int64_t n0, int64_t mid, int64_t group, const void* y, int64_t ld_y,
                              int64_t n1, float* z, int64_t ld_z, qz_stream_t stream);

/* Self-test of the staged kernels' failure path (the post has no counterpart; an interface
 * matter).  Every wait of the staged kernels on their own bulk copies gives up after a
 * limit, sets QZ_FLAG_PIPELINE_TIMEOUT in the workspace status word and returns.  This call
 * runs that same bounded wait, with limit_ns in (0, 100 ms], on a barrier that nothing
 * completes, so the flag must come up while the context stays usable.  Nothing faults.
 * QZ_ERR_UNSUPPORTED for a limit outside the range; needs the workspace; asynchronous. */
QZ_API qz_status qz_selftest_pipeline_timeout(void* ws, uint64_t limit_ns, qz_stream_t stream);

/* Synchronize `stream`, then copy the workspace status word (QZ_FLAG_* bits, sticky until
 * qz_workspace_init) into *flags_host. */
QZ_API qz_status qz_get_device_status(const void* ws, uint32_t* flags_host, qz_stream_t stream);

/* ---- Host round trip ---------------------------------------------------------------------
 * The quantization of a tensor that sits in host memory: x goes to the device in chunks of
 * whole rows, each chunk is quantized (with the fused statistics when the plan asks for
 * them) and dequantized as soon as it has landed, and its codes and scales go back while
 * later chunks arrive -- three CUDA streams of the plan's own (host-to-device, kernels,
 * device-to-host), ordered by events.  Formats with a per-tensor scale (TENSOR, NVFP4
 * BLOCK) take the amax of every chunk as it lands and are quantized once the last chunk is
 * in, with the tensor's amax (the largest of the chunk amaxes) supplied.  The operations
 * are the ones of qz_quantize / qz_dequantize / qz_stats_merge above, which the plan calls:
 * codes, scales and tensor scales are bit-identical to one qz_quantize of the whole tensor
 * (blocks and rows never straddle a chunk), the statistics are the chunks' merged.  The
 * post has no counterpart: this is the runtime around the calls above.
 *
 * Unlike the other calls, a plan allocates, once, at qz_host_plan_create on the current
 * device: a device copy of x ([rows, cols]), a workspace, per-chunk statistics and amaxes,
 * three streams and their events; qz_host_plan_destroy frees them.  qz_host_run allocates
 * nothing.  A plan is used by one host thread at a time. */
#define QZ_HOST_MAX_RUNS 16

typedef struct qz_host_plan qz_host_plan;

/* Buffers of one run (one format / granularity) of a plan.  Device outputs as qz_quantize /
 * qz_dequantize write them for the whole tensor (caller-allocated, dense):
 *   codes, scales (NULL when the format has none), tensor_scale (one fp32, required),
 *   y     the dequantized tensor, [rows, cols] of the plan's out_dtype, or NULL for none,
 *   stats the merged statistics (required when the plan fuses them, else ignored).
 * Host copies, each NULL for "not copied": codes_host, scales_host (the same bytes as the
 * device buffers), tensor_scale_host (one fp32), stats_host (one qz_stats).  Host memory
 * that is page-locked (cudaHostAlloc / cudaHostRegister) lets the copies overlap the
 * kernels; pageable memory works, with copies that do not overlap. */
typedef struct {
  void* codes;
  void* scales;
  float* tensor_scale;
  void* y;
  qz_stats* stats;
  void* codes_host;
  void* scales_host;
  float* tensor_scale_host;
  qz_stats* stats_host;
} qz_host_io;

/* A plan for `n_runs` (1 .. QZ_HOST_MAX_RUNS) quantizations of one [rows, cols] tensor:
 * runs[j] is a descriptor as for qz_quantize; every run has the same in_dtype, rows and cols,
 * and ld == cols (the host tensor is dense).  chunk_rows >= 1 rows go over per copy (a
 * chunk larger than the tensor is the whole tensor).  out_dtype (QZ_BF16 / QZ_F32) is the
 * dtype of the dequantized tensors; fuse_stats != 0 fuses the error statistics.
 * Errors: QZ_ERR_NULL (runs or plan NULL), QZ_ERR_SHAPE (n_runs or chunk_rows out of range,
 * runs of different shapes, ld != cols), QZ_ERR_ENUM (out_dtype, mixed in_dtype), every
 * descriptor error of qz_quantize, QZ_ERR_CUDA (an allocation failed; nothing is kept).
 * *plan is NULL on every error. */
QZ_API qz_status qz_host_plan_create(const qz_desc* runs, int32_t n_runs, int64_t chunk_rows,
                                     int32_t out_dtype, int32_t fuse_stats, qz_host_plan** plan);

/* One round trip of x_host (host, [rows, cols] dense, the plan's in_dtype; may be NULL for
 * an empty tensor): io[j] holds the buffers of run j (n_runs entries).  Returns when every
 * device output and host copy is complete (the plan's streams are synchronised; the
 * caller's streams are not touched).  Errors: QZ_ERR_NULL (plan, io, x_host, or a required
 * buffer of io NULL -- checked before anything is enqueued), a status of one of the calls
 * above (enqueueing stops there; what was enqueued is waited for), QZ_ERR_CUDA (a copy or
 * event failed). */
QZ_API qz_status qz_host_run(qz_host_plan* plan, const void* x_host, const qz_host_io* io);

/* Status word of the plan's workspace (QZ_FLAG_* bits raised by its calls, sticky), into
 * *flags_host; synchronous. */
QZ_API qz_status qz_host_plan_status(const qz_host_plan* plan, uint32_t* flags_host);

/* Wait for the plan's streams and free everything it allocated.  NULL is ignored. */
QZ_API void qz_host_plan_destroy(qz_host_plan* plan);

#ifdef __cplusplus
}
#endif
#endif /* QZ_H */
