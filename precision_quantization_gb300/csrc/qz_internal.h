// qz_internal.h -- host-side plumbing shared by the translation units of libqz.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "qz.h"

namespace qz {

// Geometry of one launch over a [rows, cols] high-precision tensor cut into 32-byte
// chunks along each row.
struct Geom {
  int64_t rows = 0, cols = 0, ld = 0;
  int64_t cpr = 0;       // chunks per row (ceil(cols / elements-per-chunk))
  int64_t n_chunks = 0;  // rows * cpr
  bool dense = false;    // ld == cols: a chunk's address is base + 32 * index
  bool vec = false;      // 32-byte vector access is legal (alignment + full chunks)
};

Geom make_geom(const qz_desc& d, const void* hp, int elem_bytes, int align_bytes);

// Persistent-grid size: resident CTAs of `kernel` on every SM, capped by the work and by
// the partial-result slots of the workspace.
int grid_for(const void* kernel, int64_t work_ctas, cudaStream_t stream, size_t dyn_smem = 0);

// SM count of the current device (cached).
int sm_count();

// Opt `kernel` in to `bytes` of dynamic shared memory on the current device (once).
bool set_dyn_smem(const void* kernel, int bytes);

qz_status launch_amax(const qz_desc& d, const void* x, float* out, void* ws, cudaStream_t s);

// amax_out (may be null): also write this tensor's max |x|, bit-identical to launch_amax --
// folded into the staged kernels, a separate amax pass elsewhere.
qz_status launch_quant8(const qz_desc& d, const void* x, void* codes, void* scales,
                        float* tscale_out, const float* amax, bool amax_supplied,
                        qz_stats* stats, void* ws, cudaStream_t s, float* amax_out = nullptr);
qz_status launch_quant4(const qz_desc& d, const void* x, void* codes, void* scales,
                        float* tscale_out, const float* amax, bool amax_supplied,
                        qz_stats* stats, void* ws, cudaStream_t s, float* amax_out = nullptr);
qz_status launch_dequant8(const qz_desc& d, const void* codes, const void* scales,
                          const float* tscale, void* y, int out_dtype, cudaStream_t s);
qz_status launch_dequant4(const qz_desc& d, const void* codes, const void* scales,
                          const float* tscale, void* y, int out_dtype, cudaStream_t s);
qz_status launch_stats8(const qz_desc& d, const void* x, const void* codes,
                        const void* scales, const float* tscale, qz_stats* stats, void* ws,
                        cudaStream_t s);
qz_status launch_stats4(const qz_desc& d, const void* x, const void* codes,
                        const void* scales, const float* tscale, qz_stats* stats, void* ws,
                        cudaStream_t s);
// fold `count` statistics records of disjoint parts of one tensor into *out
qz_status launch_stats_merge(const qz_stats* parts, int64_t count, qz_stats* out, cudaStream_t s);
qz_status launch_empty(float* tscale_out, qz_stats* stats, cudaStream_t s);

// grouped symmetric INT4 (block_size = group) and the asymmetric 4-bit group dequantize
qz_status launch_quant_int4(const qz_desc& d, const void* x, void* codes, void* scales,
                            float* tscale_out, qz_stats* stats, void* ws, cudaStream_t s);
qz_status launch_stats_int4(const qz_desc& d, const void* x, const void* codes, const void* scales,
                            qz_stats* stats, void* ws, cudaStream_t s);
qz_status launch_dequant_int4(const qz_desc& d, const void* codes, const void* scales, void* y,
                              int out_dtype, cudaStream_t s);
qz_status launch_dequant_asym4(const uint32_t* w, const float* scales, const uint32_t* shifts,
                               int64_t rows, int64_t cols, int64_t group, void* y, int64_t ld,
                               int out_dtype, cudaStream_t s);
// z[j][0 .. n1) = 0 for j < n0 (rows ld_z floats apart)
qz_status launch_zero_z(float* z, int64_t ld_z, int64_t n0, int64_t n1, cudaStream_t s);
// the tensor-core (tcgen05) product for many activation columns: applicable when n1 > 8,
// group % 16 == 0, mid % 64 == 0, w and y 16-byte aligned and ld_y % 8 == 0
bool quant_dot_tc_applicable(const uint32_t* w, int64_t n0, int64_t mid, int64_t group, const void* y,
                             int64_t ld_y, int64_t n1);
qz_status launch_quant_dot_tc(const uint32_t* w, const float* scales, const uint32_t* shifts, int64_t n0,
                              int64_t mid, int64_t group, const void* y, int64_t ld_y, int64_t n1, float* z,
                              int64_t ld_z, cudaStream_t s);
qz_status launch_quant_dot(const uint32_t* w, const float* scales, const uint32_t* shifts,
                           int64_t n0, int64_t mid, int64_t group, const void* y, int64_t ld_y,
                           int64_t n1, float* z, int64_t ld_z, cudaStream_t s);

inline qz_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? QZ_OK : QZ_ERR_CUDA;
}

// The descriptor checks of qz_quantize (fields, shape, input dtype), without a launch.
qz_status validate_desc(const qz_desc* d);

}  // namespace qz
