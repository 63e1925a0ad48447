// qz_api.cu -- the C ABI of libqz (declared and documented in include/qz.h): argument
// validation on the host, then the kernel launches on the caller's stream.
#include <climits>
#include <cstdint>
#include <mutex>

#include "qz_device.cuh"
#include "qz_internal.h"

namespace qz {

Geom make_geom(const qz_desc& d, const void* hp, int eb, int align) {
  Geom g;
  g.rows = d.rows;
  g.cols = d.cols;
  g.ld = d.ld;
  const int epc = 32 / eb;
  g.cpr = (d.cols + epc - 1) / epc;
  g.n_chunks = g.rows * g.cpr;
  const bool full = d.cols % epc == 0;
  const bool aligned = reinterpret_cast<uintptr_t>(hp) % align == 0 &&
                       (d.rows <= 1 || (d.ld * eb) % align == 0);
  g.vec = full && aligned;
  g.dense = g.vec && (d.ld == d.cols || d.rows <= 1);
  return g;
}

// Launch parameters that depend only on the kernel and the device (SM count, resident CTAs
// per SM, the dynamic shared-memory opt-in), looked up once and reused: a call then costs
// the launch alone, not a round of driver queries.
namespace {
constexpr int kCacheDevices = 64;
constexpr int kCacheSlots = 1024;
struct LaunchEntry {
  const void* kernel;
  size_t smem;
  int dev;
  int occ;
};
std::mutex g_launch_mu;
LaunchEntry g_launch[kCacheSlots];
int g_launch_n = 0;
int g_sms[kCacheDevices];
}  // namespace

int sm_count() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(g_launch_mu);
    if (dev >= 0 && dev < kCacheDevices && g_sms[dev] > 0) return g_sms[dev];
  }
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms < 1) sms = 1;
  std::lock_guard<std::mutex> lock(g_launch_mu);
  if (dev >= 0 && dev < kCacheDevices) g_sms[dev] = sms;
  return sms;
}

int grid_for(const void* kernel, int64_t work_ctas, cudaStream_t, size_t dyn_smem) {
  int dev = 0, sms = 1, occ = 1;
  cudaGetDevice(&dev);
  bool cached = false;
  {
    std::lock_guard<std::mutex> lock(g_launch_mu);
    if (dev >= 0 && dev < kCacheDevices && g_sms[dev] > 0) {
      sms = g_sms[dev];
      for (int i = 0; i < g_launch_n; ++i)
        if (g_launch[i].kernel == kernel && g_launch[i].smem == dyn_smem && g_launch[i].dev == dev) {
          occ = g_launch[i].occ;
          cached = true;
          break;
        }
    }
  }
  if (!cached) {
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kThreads, dyn_smem);
    std::lock_guard<std::mutex> lock(g_launch_mu);
    if (dev >= 0 && dev < kCacheDevices) {
      g_sms[dev] = sms;
      if (g_launch_n < kCacheSlots && occ > 0) g_launch[g_launch_n++] = LaunchEntry{kernel, dyn_smem, dev, occ};
    }
  }
  if (occ < 1) occ = 1;
  int64_t g = static_cast<int64_t>(sms) * occ;
  if (work_ctas < g) g = work_ctas;
  if (g < 1) g = 1;
  if (g > kMaxCtas) g = kMaxCtas;
  return static_cast<int>(g);
}

namespace {
struct AttrEntry {
  const void* kernel;
  int dev;
  int bytes;
};
std::mutex g_attr_mu;
AttrEntry g_attr[kCacheSlots];
int g_attr_n = 0;
}  // namespace

bool set_dyn_smem(const void* kernel, int bytes) {
  int dev = 0;
  cudaGetDevice(&dev);
  {
    std::lock_guard<std::mutex> lock(g_attr_mu);
    for (int i = 0; i < g_attr_n; ++i)
      if (g_attr[i].kernel == kernel && g_attr[i].dev == dev && g_attr[i].bytes >= bytes) return true;
  }
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return false;
  std::lock_guard<std::mutex> lock(g_attr_mu);
  if (g_attr_n < kCacheSlots) g_attr[g_attr_n++] = AttrEntry{kernel, dev, bytes};
  return true;
}

namespace {

__global__ void fill_kernel(float* a, float va, qz_stats* st, float* zero_out = nullptr) {
  if (a) *a = va;
  if (zero_out) *zero_out = 0.0f;
  if (st) {
    st->sum_sq_err = 0.0;
    st->mse = 0.0;
    st->max_rel_err = 0.0f;
    st->max_abs_err = 0.0f;
    st->n = 0;
  }
}

bool is8(int f) { return f == QZ_INT8 || f == QZ_FP8_E4M3 || f == QZ_FP8_E5M2; }
bool is4(int f) { return f == QZ_MXFP4 || f == QZ_NVFP4; }
bool isint4(int f) { return f == QZ_INT4; }
bool aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

qz_status check_shape(const qz_desc* d) {
  if (d->rows < 0 || d->cols < 0 || d->ld < d->cols) return QZ_ERR_SHAPE;
  if (d->rows > 0 && d->ld > 0 && d->rows > (INT64_MAX / 8) / d->ld) return QZ_ERR_SHAPE;
  return QZ_OK;
}

qz_status check_dtype(int dt) { return (dt == QZ_BF16 || dt == QZ_F32) ? QZ_OK : QZ_ERR_ENUM; }

// Format / granularity / block size / rounding fields.
qz_status check_desc(const qz_desc* d) {
  if (!d) return QZ_ERR_NULL;
  if (!is8(d->format) && !is4(d->format) && !isint4(d->format)) return QZ_ERR_ENUM;
  if (d->granularity < QZ_GRAN_TENSOR || d->granularity > QZ_GRAN_UNIT) return QZ_ERR_ENUM;
  if (d->elem_round != QZ_ROUND_RNE) return QZ_ERR_ENUM;
  if (d->scale_round != QZ_SCALE_UP && d->scale_round != QZ_SCALE_NEAREST) return QZ_ERR_ENUM;
  const qz_status st = check_shape(d);
  if (st != QZ_OK) return st;
  if (is8(d->format)) {
    if (d->granularity == QZ_GRAN_BLOCK || d->block_size != 0) return QZ_ERR_UNSUPPORTED;
  } else if (isint4(d->format)) {
    const int bs = d->block_size;
    if (bs != 16 && bs != 32 && bs != 64 && bs != 128) return QZ_ERR_UNSUPPORTED;
    if (d->granularity != QZ_GRAN_BLOCK) return QZ_ERR_UNSUPPORTED;
    if (d->cols % bs != 0) return QZ_ERR_SHAPE;
  } else {
    const int bs = d->format == QZ_MXFP4 ? 32 : 16;
    if (d->block_size != bs) return QZ_ERR_UNSUPPORTED;
    if (d->granularity != QZ_GRAN_BLOCK && d->granularity != QZ_GRAN_UNIT) return QZ_ERR_UNSUPPORTED;
    if (d->cols % bs != 0) return QZ_ERR_SHAPE;
  }
  return QZ_OK;
}

bool needs_scales(const qz_desc* d) {
  return d->granularity == QZ_GRAN_ROW || is4(d->format) || isint4(d->format);
}
bool needs_tscale(const qz_desc* d) {
  return (is8(d->format) && d->granularity == QZ_GRAN_TENSOR) ||
         (d->format == QZ_NVFP4 && d->granularity == QZ_GRAN_BLOCK);
}

qz_status check_ws(const void* ws) {
  if (!ws) return QZ_ERR_WORKSPACE;
  return aligned(ws, 16) ? QZ_OK : QZ_ERR_ALIGN;
}

}  // namespace

qz_status validate_desc(const qz_desc* d) {
  const qz_status st = check_desc(d);
  return st != QZ_OK ? st : check_dtype(d->in_dtype);
}

}  // namespace qz

using namespace qz;

extern "C" const char* qz_status_string(qz_status s) {
  switch (s) {
    case QZ_OK: return "ok";
    case QZ_ERR_NULL: return "a required pointer is NULL";
    case QZ_ERR_ENUM: return "unknown enumerator in a descriptor field";
    case QZ_ERR_SHAPE: return "rows / cols / ld out of range or cols not a multiple of the block size";
    case QZ_ERR_ALIGN: return "pointer not aligned to its element type";
    case QZ_ERR_UNSUPPORTED: return "unsupported format / granularity / block size combination";
    case QZ_ERR_CUDA: return "CUDA launch failed";
    case QZ_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

extern "C" size_t qz_workspace_size(const qz_desc*) { return kWsBytes; }

extern "C" qz_status qz_workspace_init(void* ws, size_t bytes, qz_stream_t stream) {
  if (!ws) return QZ_ERR_NULL;
  if (bytes < kWsBytes) return QZ_ERR_WORKSPACE;
  if (!aligned(ws, 16)) return QZ_ERR_ALIGN;
  return cudaMemsetAsync(ws, 0, bytes, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? QZ_OK
             : QZ_ERR_CUDA;
}

extern "C" qz_status qz_amax(const qz_desc* d, const void* x, float* amax_dev, void* ws,
                             qz_stream_t stream) {
  if (!d) return QZ_ERR_NULL;
  qz_status st = check_dtype(d->in_dtype);
  if (st != QZ_OK) return st;
  if ((st = check_shape(d)) != QZ_OK) return st;
  if (!amax_dev) return QZ_ERR_NULL;
  if ((st = check_ws(ws)) != QZ_OK) return st;
  const int eb = d->in_dtype == QZ_BF16 ? 2 : 4;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (d->rows * d->cols == 0) {
    fill_kernel<<<1, 1, 0, s>>>(amax_dev, 0.0f, nullptr);
    return launch_status();
  }
  if (!x) return QZ_ERR_NULL;
  if (!aligned(x, eb) || !aligned(amax_dev, 4)) return QZ_ERR_ALIGN;
  return launch_amax(*d, x, amax_dev, ws, s);
}

extern "C" qz_status qz_quantize(const qz_desc* d, const void* x, void* codes, void* scales,
                                 float* tensor_scale_dev, const float* tensor_amax_dev,
                                 qz_stats* stats_dev, void* ws, qz_stream_t stream) {
  qz_status st = check_desc(d);
  if (st != QZ_OK) return st;
  if ((st = check_dtype(d->in_dtype)) != QZ_OK) return st;
  const int64_t n = d->rows * d->cols;
  const bool tensor_alpha = needs_tscale(d);
  const bool compute_amax = tensor_alpha && tensor_amax_dev == nullptr;
  if (tensor_alpha && !tensor_scale_dev) return QZ_ERR_NULL;
  if (compute_amax || stats_dev) {
    if ((st = check_ws(ws)) != QZ_OK) return st;
  }
  if (tensor_scale_dev && !aligned(tensor_scale_dev, 4)) return QZ_ERR_ALIGN;
  if (tensor_amax_dev && !aligned(tensor_amax_dev, 4)) return QZ_ERR_ALIGN;
  if (stats_dev && !aligned(stats_dev, 8)) return QZ_ERR_ALIGN;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (n == 0) {
    if (tensor_scale_dev || stats_dev) {
      fill_kernel<<<1, 1, 0, s>>>(tensor_scale_dev, 1.0f, stats_dev);
      return launch_status();
    }
    return QZ_OK;
  }
  if (!x || !codes) return QZ_ERR_NULL;
  if (needs_scales(d) && !scales) return QZ_ERR_NULL;
  const int eb = d->in_dtype == QZ_BF16 ? 2 : 4;
  if (!aligned(x, eb)) return QZ_ERR_ALIGN;
  if ((d->granularity == QZ_GRAN_ROW || isint4(d->format)) && !aligned(scales, 4)) return QZ_ERR_ALIGN;
  if (isint4(d->format)) return launch_quant_int4(*d, x, codes, scales, tensor_scale_dev, stats_dev, ws, s);
  const float* amax = tensor_amax_dev;
  if (compute_amax) {
    if ((st = launch_amax(*d, x, nullptr, ws, s)) != QZ_OK) return st;
    amax = &static_cast<WsHeader*>(ws)->amax;
  }
  if (is8(d->format))
    return launch_quant8(*d, x, codes, scales, tensor_scale_dev, amax, !compute_amax, stats_dev, ws, s);
  return launch_quant4(*d, x, codes, scales, tensor_scale_dev, amax, !compute_amax, stats_dev, ws, s);
}

extern "C" qz_status qz_quantize_delayed(const qz_desc* d, const void* x, void* codes, void* scales,
                                         float* tensor_scale_dev, const float* amax_in_dev,
                                         float* amax_out_dev, qz_stats* stats_dev, void* ws,
                                         qz_stream_t stream) {
  qz_status st = check_desc(d);
  if (st != QZ_OK) return st;
  if ((st = check_dtype(d->in_dtype)) != QZ_OK) return st;
  const bool tensor_alpha = needs_tscale(d);
  if (!amax_out_dev || (tensor_alpha && (!amax_in_dev || !tensor_scale_dev))) return QZ_ERR_NULL;
  if ((st = check_ws(ws)) != QZ_OK) return st;
  if (!aligned(amax_out_dev, 4) || (amax_in_dev && !aligned(amax_in_dev, 4))) return QZ_ERR_ALIGN;
  if (tensor_scale_dev && !aligned(tensor_scale_dev, 4)) return QZ_ERR_ALIGN;
  if (stats_dev && !aligned(stats_dev, 8)) return QZ_ERR_ALIGN;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (d->rows * d->cols == 0) {
    // an empty tensor's amax is 0, as qz_amax would write
    fill_kernel<<<1, 1, 0, s>>>(tensor_scale_dev, 1.0f, stats_dev, amax_out_dev);
    return launch_status();
  }
  if (!x || !codes) return QZ_ERR_NULL;
  if (needs_scales(d) && !scales) return QZ_ERR_NULL;
  const int eb = d->in_dtype == QZ_BF16 ? 2 : 4;
  if (!aligned(x, eb)) return QZ_ERR_ALIGN;
  if ((d->granularity == QZ_GRAN_ROW || isint4(d->format)) && !aligned(scales, 4)) return QZ_ERR_ALIGN;
  if (isint4(d->format)) {
    st = launch_quant_int4(*d, x, codes, scales, tensor_scale_dev, stats_dev, ws, s);
    return st == QZ_OK ? launch_amax(*d, x, amax_out_dev, ws, s) : st;
  }
  const float* amax = tensor_alpha ? amax_in_dev : nullptr;
  if (is8(d->format))
    return launch_quant8(*d, x, codes, scales, tensor_scale_dev, amax, true, stats_dev, ws, s, amax_out_dev);
  return launch_quant4(*d, x, codes, scales, tensor_scale_dev, amax, true, stats_dev, ws, s, amax_out_dev);
}

extern "C" qz_status qz_dequantize(const qz_desc* d, const void* codes, const void* scales,
                                   const float* tensor_scale_dev, void* y, int32_t out_dtype,
                                   qz_stream_t stream) {
  qz_status st = check_desc(d);
  if (st != QZ_OK) return st;
  if ((st = check_dtype(out_dtype)) != QZ_OK) return st;
  if (d->rows * d->cols == 0) return QZ_OK;
  if (!codes || !y) return QZ_ERR_NULL;
  if (needs_scales(d) && !scales) return QZ_ERR_NULL;
  if (needs_tscale(d) && !tensor_scale_dev) return QZ_ERR_NULL;
  if (!aligned(y, out_dtype == QZ_BF16 ? 2 : 4)) return QZ_ERR_ALIGN;
  if ((d->granularity == QZ_GRAN_ROW || isint4(d->format)) && !aligned(scales, 4)) return QZ_ERR_ALIGN;
  if (tensor_scale_dev && !aligned(tensor_scale_dev, 4)) return QZ_ERR_ALIGN;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (isint4(d->format)) return launch_dequant_int4(*d, codes, scales, y, out_dtype, s);
  if (is8(d->format)) return launch_dequant8(*d, codes, scales, tensor_scale_dev, y, out_dtype, s);
  return launch_dequant4(*d, codes, scales, tensor_scale_dev, y, out_dtype, s);
}

extern "C" qz_status qz_error_stats(const qz_desc* d, const void* x, const void* codes,
                                    const void* scales, const float* tensor_scale_dev,
                                    qz_stats* stats_dev, void* ws, qz_stream_t stream) {
  qz_status st = check_desc(d);
  if (st != QZ_OK) return st;
  if ((st = check_dtype(d->in_dtype)) != QZ_OK) return st;
  if (!stats_dev) return QZ_ERR_NULL;
  if ((st = check_ws(ws)) != QZ_OK) return st;
  if (!aligned(stats_dev, 8)) return QZ_ERR_ALIGN;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (d->rows * d->cols == 0) {
    fill_kernel<<<1, 1, 0, s>>>(nullptr, 0.0f, stats_dev);
    return launch_status();
  }
  if (!x || !codes) return QZ_ERR_NULL;
  if (needs_scales(d) && !scales) return QZ_ERR_NULL;
  if (needs_tscale(d) && !tensor_scale_dev) return QZ_ERR_NULL;
  if (!aligned(x, d->in_dtype == QZ_BF16 ? 2 : 4)) return QZ_ERR_ALIGN;
  if (d->granularity == QZ_GRAN_ROW && !aligned(scales, 4)) return QZ_ERR_ALIGN;
  if (tensor_scale_dev && !aligned(tensor_scale_dev, 4)) return QZ_ERR_ALIGN;
  if (isint4(d->format)) return launch_stats_int4(*d, x, codes, scales, stats_dev, ws, s);
  if (is8(d->format)) return launch_stats8(*d, x, codes, scales, tensor_scale_dev, stats_dev, ws, s);
  return launch_stats4(*d, x, codes, scales, tensor_scale_dev, stats_dev, ws, s);
}

extern "C" qz_status qz_stats_merge(const qz_stats* parts, int64_t count, qz_stats* out,
                                    qz_stream_t stream) {
  if (!out || (count > 0 && !parts)) return QZ_ERR_NULL;
  if (count < 0) return QZ_ERR_SHAPE;
  if (!aligned(out, 8) || (count > 0 && !aligned(parts, 8))) return QZ_ERR_ALIGN;
  return launch_stats_merge(parts, count, out, reinterpret_cast<cudaStream_t>(stream));
}

extern "C" qz_status qz_dequantize_asym4(const uint32_t* w, const float* scales,
                                         const uint32_t* shifts, int64_t rows, int64_t cols,
                                         int64_t group, void* y, int64_t ld, int32_t out_dtype,
                                         qz_stream_t stream) {
  qz_status st = check_dtype(out_dtype);
  if (st != QZ_OK) return st;
  if (rows < 0 || cols < 0 || ld < cols || group <= 0 || cols % 8 != 0 || cols % group != 0)
    return QZ_ERR_SHAPE;
  if (rows > 0 && ld > 0 && rows > (INT64_MAX / 8) / ld) return QZ_ERR_SHAPE;
  if (rows * cols == 0) return QZ_OK;
  if (!w || !scales || !shifts || !y) return QZ_ERR_NULL;
  if (!aligned(w, 4) || !aligned(scales, 4) || !aligned(shifts, 4) ||
      !aligned(y, out_dtype == QZ_BF16 ? 2 : 4))
    return QZ_ERR_ALIGN;
  return launch_dequant_asym4(w, scales, shifts, rows, cols, group, y, ld, out_dtype,
                              reinterpret_cast<cudaStream_t>(stream));
}

extern "C" qz_status qz_quant_dot(const uint32_t* w, const float* scales, const uint32_t* shifts,
                                  int64_t n0, int64_t mid, int64_t group, const void* y,
                                  int64_t ld_y, int64_t n1, float* z, int64_t ld_z,
                                  qz_stream_t stream) {
  if (n0 < 0 || mid < 0 || n1 < 0 || group <= 0 || mid % 8 != 0 || mid % group != 0 || ld_y < n1 ||
      ld_z < n1)
    return QZ_ERR_SHAPE;
  if (n1 >= (int64_t{1} << 30) || n0 >= (int64_t{1} << 40)) return QZ_ERR_UNSUPPORTED;
  if ((mid > 0 && ld_y > 0 && mid > (INT64_MAX / 8) / ld_y) || (n0 > 0 && ld_z > 0 && n0 > (INT64_MAX / 8) / ld_z))
    return QZ_ERR_SHAPE;
  if (n0 * n1 == 0) return QZ_OK;
  if (!w || !scales || !shifts || !y || !z) return QZ_ERR_NULL;
  if (!aligned(w, 4) || !aligned(scales, 4) || !aligned(shifts, 4) || !aligned(y, 2) || !aligned(z, 4))
    return QZ_ERR_ALIGN;
  if (mid == 0) {  // empty sums
    return launch_zero_z(z, ld_z, n0, n1, reinterpret_cast<cudaStream_t>(stream));
  }
  return launch_quant_dot(w, scales, shifts, n0, mid, group, y, ld_y, n1, z, ld_z,
                          reinterpret_cast<cudaStream_t>(stream));
}

extern "C" qz_status qz_get_device_status(const void* ws, uint32_t* flags_host, qz_stream_t stream) {
  if (!ws || !flags_host) return QZ_ERR_NULL;
  if (!aligned(ws, 16)) return QZ_ERR_ALIGN;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(flags_host, ws, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return QZ_ERR_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? QZ_OK : QZ_ERR_CUDA;
}
