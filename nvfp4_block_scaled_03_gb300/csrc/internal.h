// internal.h -- host-side declarations shared by the library's translation
// units (not part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/nvfp4.h"

namespace nvfp4 {

// Launches kern with programmatic stream serialization: the grid may be
// scheduled before the previous kernel on the stream has finished, and each
// kernel launched this way calls griddep_wait() before its first access to
// global memory.  Within a captured CUDA graph the same dependency becomes a
// programmatic edge.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

struct DeviceInfo {
  int device;
  int sm_count;
  int major, minor;
};

// Cached attributes of the current device; NVFP4_ERR_ARCH if it is not sm_103.
nvfp4_status current_device(DeviceInfo* info);

// Partial maxima slots in a quantiser workspace (one float per amax CTA).
constexpr int kMaxPartials = 1024;
constexpr size_t kQuantWorkspaceBytes = kMaxPartials * sizeof(float);

size_t swizzled_scale_bytes(int64_t rows, int64_t cols);

nvfp4_status quantize_impl(const void* x, int32_t in_dtype, int64_t rows, int64_t cols,
                           int64_t ld, int32_t mode, uint32_t flags, uint64_t seed,
                           uint64_t offset, nvfp4_tensor* out, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream);

nvfp4_status quantize_rowcol_impl(const void* x, int32_t in_dtype, int64_t rows, int64_t cols,
                                  int64_t ld, uint32_t row_flags, uint32_t col_flags,
                                  uint64_t seed, uint64_t row_offset, uint64_t col_offset,
                                  nvfp4_tensor* row_out, nvfp4_tensor* col_out,
                                  cudaStream_t stream);

nvfp4_status gemm_impl(const nvfp4_tensor* A, int32_t a_view, const nvfp4_tensor* B,
                       int32_t b_view, void* D, int32_t d_mode, const void* C, int64_t M,
                       int64_t N, int64_t K, int32_t tile, cudaStream_t stream);

// Reads and clears the GEMM kernels' device error word (after a sync).
nvfp4_status gemm_read_error(unsigned int* code);

// SwiGLU forward / backward on bf16 [rows, cols] tensors (rows % 16 == 0,
// cols % 8 == 0), also writing the tensor amaxes of each bf16 output for its
// row-wise (amax_*_row: max |x|) and column-wise (amax_*_col: max |RHT(x)|
// over 16-row column blocks with the seed's signs when rht, else max |x|)
// NVFP4 quantisations.  partials: 16-byte aligned device scratch of at least
// kSwigluPartialsBytes.
constexpr size_t kSwigluPartialsBytes = 4 * kMaxPartials * sizeof(float);
nvfp4_status swiglu_fwd_impl(const void* G, const void* U, void* H, int64_t rows, int64_t cols,
                             uint64_t seed, bool rht, float* amax_row, float* amax_col,
                             void* partials, size_t partials_bytes, cudaStream_t stream);
nvfp4_status swiglu_bwd_impl(const void* dH, const void* G, const void* U, void* dG, void* dU,
                             int64_t rows, int64_t cols, uint64_t seed, bool rht,
                             float* amax_dg_row, float* amax_dg_col, float* amax_du_row,
                             float* amax_du_col, void* partials, size_t partials_bytes,
                             cudaStream_t stream);

// cuTensorMapEncodeTiled, reached through the runtime's driver entry-point
// query (null if the driver does not provide it).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();

nvfp4_status amax_impl(const void* x, int32_t in_dtype, int64_t rows, int64_t cols, int64_t ld,
                       uint64_t seed, float* amax_plain, float* amax_rht, void* workspace,
                       size_t workspace_bytes, cudaStream_t stream);

// Reads and clears the quantisers' device error word (after a sync).
nvfp4_status quant_read_error(unsigned int* code);

// Failure injection of nvfp4_debug_inject: stall flag and pipeline wait limit.
nvfp4_status quant_set_injection(unsigned int stall, unsigned long long wait_ns);
nvfp4_status gemm_set_injection(unsigned int stall, unsigned long long wait_ns);

nvfp4_status gemm_mx_impl(const void* a_codes, const void* a_sf, const void* b_codes,
                          const void* b_sf, int32_t fmt, void* D, int64_t M, int64_t N,
                          int64_t K, cudaStream_t stream);

nvfp4_status mx_sizes_impl(int64_t rows, int64_t cols, int32_t mode, int32_t fmt,
                           size_t* codes_bytes, size_t* scales_bytes, size_t* scales_sw_bytes);
nvfp4_status mx_quantize_impl(const void* x, int32_t in_dtype, int64_t rows, int64_t cols,
                              int64_t ld, int32_t mode, int32_t fmt, void* codes, void* scales,
                              void* scales_sw, cudaStream_t stream);

inline nvfp4_status cuda_status(cudaError_t e) {
  return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // namespace nvfp4
