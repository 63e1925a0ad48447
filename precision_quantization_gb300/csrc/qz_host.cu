// qz_host.cu -- the host round trip of include/qz.h (qz_host_plan_create / qz_host_run /
// qz_host_plan_status / qz_host_plan_destroy): a tensor in host memory is copied to the
// device in row chunks on one stream, each chunk is quantized (with the fused error
// statistics) and dequantized on a second stream as soon as it has landed, and its codes
// and scales go back on a third while later chunks arrive.  Only host code: every step on
// the GPU is one of the library's own calls (qz_quantize, qz_dequantize, qz_amax,
// qz_stats_merge) on the plan's kernel stream.
//
// Why the chunked results equal the whole-tensor call: blocks and rows never straddle a
// chunk (chunks are whole rows), a row scale is its row's own, and the formats with a
// per-tensor scale (TENSOR, NVFP4 BLOCK) are quantized only after the amax of every chunk
// has been folded into the tensor's amax (the largest of non-negative values is their
// amax), which each chunk's call then takes as its supplied alpha.  The statistics of the
// chunks are folded by qz_stats_merge.
#include <cstdint>
#include <new>
#include <utility>
#include <vector>

#include "qz.h"
#include "qz_internal.h"

struct qz_host_plan {
  int dev = 0;
  int64_t rows = 0, cols = 0;
  int32_t in_dtype = QZ_BF16, out_dtype = QZ_BF16;
  bool stats = true;
  bool need_alpha = false;
  std::vector<qz_desc> runs;                        // whole-tensor descriptors
  std::vector<std::pair<int64_t, int64_t>> chunks;  // [r0, r1) row ranges
  void* x = nullptr;                                // device copy of x, [rows, cols] dense
  void* ws = nullptr;                               // workspace of the plan's calls
  qz_stats* parts = nullptr;                        // [runs][chunks] chunk statistics
  float* amax_parts = nullptr;                      // [chunks] chunk amaxes
  float* alpha = nullptr;                           // the folded tensor amax
  cudaStream_t s_in = nullptr, s_k = nullptr, s_out = nullptr;
  std::vector<cudaEvent_t> ev_in;   // chunk i landed
  std::vector<cudaEvent_t> ev_run;  // run j, chunk i quantized: index j * chunks + i
  cudaEvent_t ev_end = nullptr;
};

namespace {

bool is_fp4(int f) { return f == QZ_MXFP4 || f == QZ_NVFP4; }

bool needs_tensor_amax(const qz_desc& d) {
  return d.granularity == QZ_GRAN_TENSOR || (d.format == QZ_NVFP4 && d.granularity == QZ_GRAN_BLOCK);
}

// Bytes per row of the codes and of the scales (dense layouts of include/qz.h).
int64_t code_row_bytes(const qz_desc& d) { return (is_fp4(d.format) || d.format == QZ_INT4) ? d.cols / 2 : d.cols; }
int64_t scale_row_bytes(const qz_desc& d) {
  if (d.format == QZ_MXFP4) return d.cols / 32;
  if (d.format == QZ_NVFP4) return d.cols / 16;
  if (d.format == QZ_INT4) return d.cols / d.block_size * 4;
  if (d.granularity == QZ_GRAN_ROW) return 4;
  return 0;
}
int elem_bytes(int32_t dt) { return dt == QZ_BF16 ? 2 : 4; }

qz_desc chunk_desc(const qz_desc& d, int64_t rows) {
  qz_desc c = d;
  c.rows = rows;
  c.ld = d.cols;
  return c;
}

template <typename T>
T* at(void* base, int64_t bytes) {
  return base ? reinterpret_cast<T*>(static_cast<char*>(base) + bytes) : nullptr;
}

// Makes the plan's device current for the scope and restores the caller's.
struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

void release(qz_host_plan* p) {
  if (!p) return;
  cudaFree(p->x);
  cudaFree(p->ws);
  cudaFree(p->parts);
  cudaFree(p->amax_parts);
  cudaFree(p->alpha);
  for (cudaEvent_t e : p->ev_in) cudaEventDestroy(e);
  for (cudaEvent_t e : p->ev_run) cudaEventDestroy(e);
  if (p->ev_end) cudaEventDestroy(p->ev_end);
  if (p->s_in) cudaStreamDestroy(p->s_in);
  if (p->s_k) cudaStreamDestroy(p->s_k);
  if (p->s_out) cudaStreamDestroy(p->s_out);
  delete p;
}

// Everything enqueued so far has finished (streams synchronised); the first error wins.
qz_status finish(qz_host_plan* p, qz_status st) {
  const cudaError_t a = cudaStreamSynchronize(p->s_in);
  const cudaError_t b = cudaStreamSynchronize(p->s_k);
  const cudaError_t c = cudaStreamSynchronize(p->s_out);
  if (st == QZ_OK && (a != cudaSuccess || b != cudaSuccess || c != cudaSuccess)) return QZ_ERR_CUDA;
  return st;
}

qz_status copy(void* dst, const void* src, int64_t bytes, cudaMemcpyKind kind, cudaStream_t s) {
  if (!dst || bytes == 0) return QZ_OK;
  return cudaMemcpyAsync(dst, src, static_cast<size_t>(bytes), kind, s) == cudaSuccess ? QZ_OK : QZ_ERR_CUDA;
}

// Quantize (+ statistics) and dequantize chunk i of run j on the kernel stream, then send
// its codes and scales back on the out stream.
qz_status run_chunk(qz_host_plan* p, int j, int i, const float* alpha, const qz_host_io& io) {
  const qz_desc& d = p->runs[j];
  const int64_t r0 = p->chunks[i].first, r1 = p->chunks[i].second;
  const qz_desc c = chunk_desc(d, r1 - r0);
  const int64_t cb = code_row_bytes(d), sb = scale_row_bytes(d);
  void* codes = at<char>(io.codes, r0 * cb);
  void* scales = sb ? at<char>(io.scales, r0 * sb) : nullptr;
  const void* x = at<char>(p->x, r0 * p->cols * elem_bytes(p->in_dtype));
  qz_stats* part = p->stats ? p->parts + static_cast<int64_t>(j) * p->chunks.size() + i : nullptr;
  const qz_stream_t sk = reinterpret_cast<qz_stream_t>(p->s_k);
  qz_status st = qz_quantize(&c, x, codes, scales, io.tensor_scale, alpha, part, p->ws, sk);
  if (st != QZ_OK) return st;
  if (io.y) {
    void* y = at<char>(io.y, r0 * p->cols * elem_bytes(p->out_dtype));
    if ((st = qz_dequantize(&c, codes, scales, io.tensor_scale, y, p->out_dtype, sk)) != QZ_OK) return st;
  }
  cudaEvent_t ev = p->ev_run[static_cast<size_t>(j) * p->chunks.size() + i];
  if (cudaEventRecord(ev, p->s_k) != cudaSuccess || cudaStreamWaitEvent(p->s_out, ev, 0) != cudaSuccess)
    return QZ_ERR_CUDA;
  if ((st = copy(at<char>(io.codes_host, r0 * cb), codes, (r1 - r0) * cb, cudaMemcpyDeviceToHost, p->s_out)) != QZ_OK)
    return st;
  if (sb)
    st = copy(at<char>(io.scales_host, r0 * sb), scales, (r1 - r0) * sb, cudaMemcpyDeviceToHost, p->s_out);
  return st;
}

qz_status enqueue(qz_host_plan* p, const void* x_host, const qz_host_io* io) {
  const int nr = static_cast<int>(p->runs.size());
  const qz_stream_t sk = reinterpret_cast<qz_stream_t>(p->s_k);
  qz_status st = QZ_OK;
  if (p->chunks.empty()) {  // empty tensor: each run's call writes its tensor scale and statistics
    for (int j = 0; j < nr && st == QZ_OK; ++j)
      st = qz_quantize(&p->runs[j], p->x, io[j].codes, io[j].scales, io[j].tensor_scale, nullptr,
                       p->stats ? io[j].stats : nullptr, p->ws, sk);
  } else {
    const int64_t xrow = p->cols * elem_bytes(p->in_dtype);
    for (size_t i = 0; i < p->chunks.size() && st == QZ_OK; ++i) {
      const int64_t r0 = p->chunks[i].first, r1 = p->chunks[i].second;
      st = copy(at<char>(p->x, r0 * xrow), static_cast<const char*>(x_host) + r0 * xrow, (r1 - r0) * xrow,
                cudaMemcpyHostToDevice, p->s_in);
      if (st == QZ_OK && cudaEventRecord(p->ev_in[i], p->s_in) != cudaSuccess) st = QZ_ERR_CUDA;
    }
    // formats whose scales are local to a row or a block: as each chunk lands; the chunk's
    // amax for the formats with a per-tensor scale
    for (size_t i = 0; i < p->chunks.size() && st == QZ_OK; ++i) {
      if (cudaStreamWaitEvent(p->s_k, p->ev_in[i], 0) != cudaSuccess) return QZ_ERR_CUDA;
      for (int j = 0; j < nr && st == QZ_OK; ++j)
        if (!needs_tensor_amax(p->runs[j])) st = run_chunk(p, j, static_cast<int>(i), nullptr, io[j]);
      if (st == QZ_OK && p->need_alpha) {
        const int64_t r0 = p->chunks[i].first, r1 = p->chunks[i].second;
        qz_desc a = chunk_desc(p->runs[0], r1 - r0);
        a.format = QZ_INT8;
        a.granularity = QZ_GRAN_TENSOR;
        a.block_size = 0;
        st = qz_amax(&a, at<char>(p->x, r0 * p->cols * elem_bytes(p->in_dtype)), p->amax_parts + i, p->ws, sk);
      }
    }
    // the tensor's amax, then the formats with a per-tensor scale, chunk by chunk
    if (st == QZ_OK && p->need_alpha) {
      qz_desc fold{};
      fold.format = QZ_INT8;
      fold.in_dtype = QZ_F32;
      fold.granularity = QZ_GRAN_TENSOR;
      fold.rows = 1;
      fold.cols = static_cast<int64_t>(p->chunks.size());
      fold.ld = fold.cols;
      st = qz_amax(&fold, p->amax_parts, p->alpha, p->ws, sk);
      for (size_t i = 0; i < p->chunks.size() && st == QZ_OK; ++i)
        for (int j = 0; j < nr && st == QZ_OK; ++j)
          if (needs_tensor_amax(p->runs[j])) st = run_chunk(p, j, static_cast<int>(i), p->alpha, io[j]);
    }
    if (st == QZ_OK && p->stats)
      for (int j = 0; j < nr && st == QZ_OK; ++j)
        st = qz_stats_merge(p->parts + static_cast<int64_t>(j) * p->chunks.size(),
                            static_cast<int64_t>(p->chunks.size()), io[j].stats, sk);
  }
  if (st != QZ_OK) return st;
  // tensor scales and statistics once the kernel stream is through
  if (cudaEventRecord(p->ev_end, p->s_k) != cudaSuccess || cudaStreamWaitEvent(p->s_out, p->ev_end, 0) != cudaSuccess)
    return QZ_ERR_CUDA;
  for (int j = 0; j < nr && st == QZ_OK; ++j) {
    st = copy(io[j].tensor_scale_host, io[j].tensor_scale, sizeof(float), cudaMemcpyDeviceToHost, p->s_out);
    if (st == QZ_OK && p->stats)
      st = copy(io[j].stats_host, io[j].stats, sizeof(qz_stats), cudaMemcpyDeviceToHost, p->s_out);
  }
  return st;
}

}  // namespace

extern "C" qz_status qz_host_plan_create(const qz_desc* runs, int32_t n_runs, int64_t chunk_rows,
                                         int32_t out_dtype, int32_t fuse_stats, qz_host_plan** plan) {
  if (!runs || !plan) return QZ_ERR_NULL;
  *plan = nullptr;
  if (n_runs < 1 || n_runs > QZ_HOST_MAX_RUNS || chunk_rows < 1) return QZ_ERR_SHAPE;
  if (out_dtype != QZ_BF16 && out_dtype != QZ_F32) return QZ_ERR_ENUM;
  if (runs[0].in_dtype != QZ_BF16 && runs[0].in_dtype != QZ_F32) return QZ_ERR_ENUM;
  for (int j = 0; j < n_runs; ++j) {
    const qz_desc& d = runs[j];
    if (d.in_dtype != runs[0].in_dtype) return QZ_ERR_ENUM;
    if (d.rows != runs[0].rows || d.cols != runs[0].cols || d.ld != d.cols) return QZ_ERR_SHAPE;
    const qz_status st = qz::validate_desc(&d);
    if (st != QZ_OK) return st;
  }
  qz_host_plan* p = new (std::nothrow) qz_host_plan;
  if (!p) return QZ_ERR_CUDA;
  if (cudaGetDevice(&p->dev) != cudaSuccess) {
    delete p;
    return QZ_ERR_CUDA;
  }
  p->rows = runs[0].rows;
  p->cols = runs[0].cols;
  p->in_dtype = runs[0].in_dtype;
  p->out_dtype = out_dtype;
  p->stats = fuse_stats != 0;
  p->runs.assign(runs, runs + n_runs);
  for (int j = 0; j < n_runs; ++j) p->need_alpha = p->need_alpha || needs_tensor_amax(runs[j]);
  if (p->rows > 0 && p->cols > 0)
    for (int64_t r0 = 0; r0 < p->rows; r0 += chunk_rows)
      p->chunks.emplace_back(r0, r0 + chunk_rows < p->rows ? r0 + chunk_rows : p->rows);
  const size_t nc = p->chunks.size() ? p->chunks.size() : 1;
  const size_t ws_bytes = qz_workspace_size(&runs[0]);
  bool ok = cudaMalloc(&p->ws, ws_bytes) == cudaSuccess &&
            cudaMalloc(&p->parts, sizeof(qz_stats) * nc * n_runs) == cudaSuccess &&
            cudaMalloc(&p->amax_parts, sizeof(float) * nc) == cudaSuccess &&
            cudaMalloc(&p->alpha, sizeof(float)) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p->s_in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p->s_k, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p->s_out, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&p->ev_end, cudaEventDisableTiming) == cudaSuccess;
  if (ok && p->rows * p->cols > 0)
    ok = cudaMalloc(&p->x, static_cast<size_t>(p->rows * p->cols * elem_bytes(p->in_dtype))) == cudaSuccess;
  for (size_t i = 0; ok && i < p->chunks.size(); ++i) {
    cudaEvent_t e = nullptr;
    ok = cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess;
    if (ok) p->ev_in.push_back(e);
  }
  for (size_t i = 0; ok && i < p->chunks.size() * n_runs; ++i) {
    cudaEvent_t e = nullptr;
    ok = cudaEventCreateWithFlags(&e, cudaEventDisableTiming) == cudaSuccess;
    if (ok) p->ev_run.push_back(e);
  }
  ok = ok && qz_workspace_init(p->ws, ws_bytes, reinterpret_cast<qz_stream_t>(p->s_k)) == QZ_OK &&
       cudaStreamSynchronize(p->s_k) == cudaSuccess;
  if (!ok) {
    release(p);
    return QZ_ERR_CUDA;
  }
  *plan = p;
  return QZ_OK;
}

extern "C" qz_status qz_host_run(qz_host_plan* plan, const void* x_host, const qz_host_io* io) {
  if (!plan || !io) return QZ_ERR_NULL;
  if (!plan->chunks.empty() && !x_host) return QZ_ERR_NULL;
  for (size_t j = 0; j < plan->runs.size(); ++j) {
    const qz_host_io& o = io[j];
    if (!o.tensor_scale || (plan->stats && !o.stats)) return QZ_ERR_NULL;
    if (!plan->chunks.empty() && !o.codes) return QZ_ERR_NULL;
    if (!plan->chunks.empty() && scale_row_bytes(plan->runs[j]) && !o.scales) return QZ_ERR_NULL;
  }
  DeviceGuard guard(plan->dev);
  return finish(plan, enqueue(plan, x_host, io));
}

extern "C" qz_status qz_host_plan_status(const qz_host_plan* plan, uint32_t* flags_host) {
  if (!plan || !flags_host) return QZ_ERR_NULL;
  DeviceGuard guard(plan->dev);
  return qz_get_device_status(plan->ws, flags_host, reinterpret_cast<qz_stream_t>(plan->s_k));
}

extern "C" void qz_host_plan_destroy(qz_host_plan* plan) {
  if (!plan) return;
  DeviceGuard guard(plan->dev);
  cudaStreamSynchronize(plan->s_in);
  cudaStreamSynchronize(plan->s_k);
  cudaStreamSynchronize(plan->s_out);
  release(plan);
}
