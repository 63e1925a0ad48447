// qz_selftest.cu -- exercises the failure path of the staged kernels without a fault.
//
// Every wait of the staged kernels (a thread waiting for its tile's bulk copy to land on an
// mbarrier) is bounded: past the limit the kernel sets QZ_FLAG_PIPELINE_TIMEOUT in the
// workspace status word and returns, so the context stays usable and the host reads the
// status.  No real copy ever takes that long, so this entry point runs the same bounded
// wait (mbar_wait) on a barrier that nothing completes -- it expects one arrival and gets
// none -- with a short limit, and reports the timeout the same way.  No copy is in flight,
// so nothing has to be drained.
#include "qz_device.cuh"
#include "qz_internal.h"
#include "qz_pipe.cuh"

namespace qz {
namespace {

__global__ void pipeline_timeout_kernel(void* ws, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    mbar_init_fence();
  }
  __syncthreads();
  // phase 0 never completes: no thread arrives and no copy is issued
  const bool ok = mbar_wait(smem_addr(&bar), 0u, limit_ns);
  if (__syncthreads_or(!ok) && threadIdx.x == 0) flag_status(ws, QZ_FLAG_PIPELINE_TIMEOUT);
}

}  // namespace
}  // namespace qz

extern "C" qz_status qz_selftest_pipeline_timeout(void* ws, uint64_t limit_ns, qz_stream_t stream) {
  if (!ws) return QZ_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) % 16 != 0) return QZ_ERR_ALIGN;
  if (limit_ns == 0 || limit_ns > 100000000ull) return QZ_ERR_UNSUPPORTED;  // (0, 100 ms]
  qz::pipeline_timeout_kernel<<<1, qz::kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(ws, limit_ns);
  return qz::launch_status();
}
