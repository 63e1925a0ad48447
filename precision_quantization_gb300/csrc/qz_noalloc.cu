// qz_noalloc.cu -- qz_error_stats_noalloc: the error statistics for callers that cannot
// allocate device memory themselves, and qz_error_stats_noalloc_status, which reads the
// status flags those calls raise.
//
// Some callers are not in a position to provide the workspace that qz_error_stats needs:
// code that runs inside another framework's memory pool and may not call cudaMalloc
// behind its back, code on a latency-critical path where cudaMalloc / cudaFree (which can
// synchronise the device) are not allowed, or a plugin that is handed only its input and
// output buffers.  This entry point takes no workspace: its scratch is a fixed array in
// device memory that belongs to the library module.  The entry point itself allocates
// nothing (no cudaMalloc, cudaFree, or allocating library call).
#include <mutex>

#include "qz_device.cuh"
#include "qz_internal.h"

namespace {

// The scratch of qz_error_stats_noalloc: one workspace (qz_workspace_size() bytes) in
// device memory.  It is part of the module, so every GPU that loads the library holds it
// until the process exits.  The scratch the statistics need does not grow with the tensor
// (one partial per CTA of a grid capped at the workspace's slot count).  Like a caller's
// workspace it starts zeroed: its completion counters wrap back to 0 at the end of every
// statistics kernel, and its status word collects QZ_FLAG_* bits until
// qz_error_stats_noalloc_status reads and clears them.
static __device__ __align__(256) unsigned char g_stats_scratch[qz::kWsBytes];

// In host code g_stats_scratch names a host-side stand-in, not device memory: the device
// address is looked up once per device (with that device current) and cached here.  The
// cache lives as long as the device's primary context: after cudaDeviceReset the module is
// loaded anew, possibly at another address, so these entry points must not be used across
// a device reset.
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

qz_status scratch_of_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return QZ_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return QZ_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_stats_scratch) != cudaSuccess || p == nullptr) return QZ_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return QZ_OK;
}

}  // namespace

extern "C" qz_status qz_error_stats_noalloc(const qz_desc* desc, const void* x, const void* codes,
                                            const void* scales, const float* tensor_scale_dev,
                                            qz_stats* stats_dev, qz_stream_t stream) {
  if (!desc) return QZ_ERR_NULL;
  if (qz_workspace_size(desc) > sizeof(g_stats_scratch)) return QZ_ERR_WORKSPACE;
  void* ws = nullptr;
  const qz_status st = scratch_of_current_device(&ws);
  if (st != QZ_OK) return st;
  // The statistics kernels leave the completion counters at 0 and only ever set status
  // bits, so the array is ready for the next call without any clearing here.
  return qz_error_stats(desc, x, codes, scales, tensor_scale_dev, stats_dev, ws, stream);
}

extern "C" qz_status qz_error_stats_noalloc_status(uint32_t* flags_host, qz_stream_t stream) {
  if (!flags_host) return QZ_ERR_NULL;
  void* ws = nullptr;
  const qz_status st = scratch_of_current_device(&ws);
  if (st != QZ_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint32_t* status = &static_cast<qz::WsHeader*>(ws)->status;
  // read, then clear, in stream order behind the calls already enqueued on `stream`
  if (cudaMemcpyAsync(flags_host, status, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return QZ_ERR_CUDA;
  if (cudaMemsetAsync(status, 0, sizeof(uint32_t), s) != cudaSuccess) return QZ_ERR_CUDA;
  return cudaStreamSynchronize(s) == cudaSuccess ? QZ_OK : QZ_ERR_CUDA;
}
