// api.cu -- the extern "C" entry points of libnvfp4.so (declared and
// documented in include/nvfp4.h): argument checks, device checks and
// dispatch to the kernels' host launchers.
#include <mutex>

#include "internal.h"

namespace nvfp4 {

nvfp4_status current_device(DeviceInfo* info) {
  static std::mutex mu;
  static DeviceInfo cache[64];
  static bool have[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return NVFP4_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 64) return NVFP4_ERR_CUDA;
  if (!have[dev]) {
    DeviceInfo d;
    d.device = dev;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return NVFP4_ERR_CUDA;
    cache[dev] = d;
    have[dev] = true;
  }
  *info = cache[dev];
  if (info->major != 10 || info->minor != 3) return NVFP4_ERR_ARCH;
  return NVFP4_OK;
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

const char* nvfp4_status_string(nvfp4_status s) {
  switch (s) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_INVALID_ARG: return "invalid argument";
    case NVFP4_ERR_SHAPE: return "unsupported shape";
    case NVFP4_ERR_ALIGN: return "misaligned pointer or leading dimension";
    case NVFP4_ERR_ARCH: return "device is not sm_103 (GB300)";
    case NVFP4_ERR_WORKSPACE: return "workspace missing or too small";
    case NVFP4_ERR_CUDA: return "CUDA error";
    case NVFP4_ERR_DEVICE_TIMEOUT: return "a kernel's bounded wait expired";
  }
  return "unknown status";
}

int nvfp4_version(void) { return 100; }

nvfp4_status nvfp4_device_check(int device) {
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  return (major == 10 && minor == 3) ? NVFP4_OK : NVFP4_ERR_ARCH;
}

nvfp4_status nvfp4_check_device_errors(nvfp4_stream stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  unsigned int gcode = 0, qcode = 0;
  nvfp4_status st = gemm_read_error(&gcode);
  if (st != NVFP4_OK) return st;
  st = quant_read_error(&qcode);
  if (st != NVFP4_OK) return st;
  return (gcode || qcode) ? NVFP4_ERR_DEVICE_TIMEOUT : NVFP4_OK;
}

nvfp4_status nvfp4_debug_inject(uint32_t stall_mask, uint64_t wait_limit_ns) {
  if (stall_mask & ~(uint32_t)(NVFP4_STALL_QUANTIZE | NVFP4_STALL_GEMM))
    return NVFP4_ERR_INVALID_ARG;
  const unsigned long long ns = wait_limit_ns ? wait_limit_ns : 2000000000ull;
  if (cudaDeviceSynchronize() != cudaSuccess) return NVFP4_ERR_CUDA;
  nvfp4_status st = quant_set_injection((stall_mask & NVFP4_STALL_QUANTIZE) ? 1u : 0u, ns);
  if (st != NVFP4_OK) return st;
  return gemm_set_injection((stall_mask & NVFP4_STALL_GEMM) ? 1u : 0u, ns);
}

nvfp4_status nvfp4_quantize_sizes(int64_t rows, int64_t cols, int32_t mode, uint32_t flags,
                                  size_t* codes_bytes, size_t* scales_bytes,
                                  size_t* scales_t_bytes, size_t* workspace_bytes) {
  if (mode < NVFP4_ROW_1X16 || mode > NVFP4_BLOCK_16X16) return NVFP4_ERR_INVALID_ARG;
  if (rows <= 0 || cols <= 0) return NVFP4_ERR_SHAPE;
  const int64_t orows = mode == NVFP4_COL_1X16 ? cols : rows;
  const int64_t ocols = mode == NVFP4_COL_1X16 ? rows : cols;
  if (ocols % 16) return NVFP4_ERR_SHAPE;
  if (codes_bytes) *codes_bytes = (size_t)(orows * (ocols / 2));
  if (scales_bytes) *scales_bytes = swizzled_scale_bytes(orows, ocols);
  if (scales_t_bytes)
    *scales_t_bytes = (flags & NVFP4_EMIT_T) && orows % 16 == 0
                          ? swizzled_scale_bytes(ocols, orows) : 0;
  if (workspace_bytes) *workspace_bytes = (flags & NVFP4_AMAX_GIVEN) ? 0 : kQuantWorkspaceBytes;
  return NVFP4_OK;
}

nvfp4_status nvfp4_quantize(const void* x, int32_t in_dtype, int64_t rows, int64_t cols,
                            int64_t ld, int32_t mode, uint32_t flags, uint64_t seed,
                            uint64_t offset, nvfp4_tensor* out, void* workspace,
                            size_t workspace_bytes, nvfp4_stream stream) {
  return quantize_impl(x, in_dtype, rows, cols, ld, mode, flags, seed, offset, out, workspace,
                       workspace_bytes, static_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_quantize_rowcol(const void* x, int32_t in_dtype, int64_t rows, int64_t cols,
                                   int64_t ld, uint32_t row_flags, uint32_t col_flags,
                                   uint64_t seed, uint64_t row_offset, uint64_t col_offset,
                                   nvfp4_tensor* row_out, nvfp4_tensor* col_out,
                                   nvfp4_stream stream) {
  return quantize_rowcol_impl(x, in_dtype, rows, cols, ld, row_flags, col_flags, seed, row_offset,
                              col_offset, row_out, col_out, static_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_amax(const void* x, int32_t in_dtype, int64_t rows, int64_t cols, int64_t ld,
                        uint64_t seed, float* amax_plain, float* amax_rht, void* workspace,
                        size_t workspace_bytes, nvfp4_stream stream) {
  return amax_impl(x, in_dtype, rows, cols, ld, seed, amax_plain, amax_rht, workspace,
                   workspace_bytes, static_cast<cudaStream_t>(stream));
}

size_t nvfp4_swiglu_workspace_bytes(void) { return kSwigluPartialsBytes; }

nvfp4_status nvfp4_swiglu_fwd(const void* G, const void* U, void* H, int64_t rows, int64_t cols,
                              uint32_t flags, uint64_t seed, float* amax_h_row,
                              float* amax_h_col, void* workspace, size_t workspace_bytes,
                              nvfp4_stream stream) {
  if (flags & ~(uint32_t)NVFP4_RHT) return NVFP4_ERR_INVALID_ARG;
  return swiglu_fwd_impl(G, U, H, rows, cols, seed, flags & NVFP4_RHT, amax_h_row, amax_h_col,
                         workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_swiglu_bwd(const void* dH, const void* G, const void* U, void* dG, void* dU,
                              int64_t rows, int64_t cols, uint32_t flags, uint64_t seed,
                              float* amax_dg_row, float* amax_dg_col, float* amax_du_row,
                              float* amax_du_col, void* workspace, size_t workspace_bytes,
                              nvfp4_stream stream) {
  if (flags & ~(uint32_t)NVFP4_RHT) return NVFP4_ERR_INVALID_ARG;
  return swiglu_bwd_impl(dH, G, U, dG, dU, rows, cols, seed, flags & NVFP4_RHT, amax_dg_row,
                         amax_dg_col, amax_du_row, amax_du_col, workspace, workspace_bytes,
                         static_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_mx_sizes(int64_t rows, int64_t cols, int32_t mode, int32_t fmt,
                            size_t* codes_bytes, size_t* scales_bytes, size_t* scales_sw_bytes) {
  return mx_sizes_impl(rows, cols, mode, fmt, codes_bytes, scales_bytes, scales_sw_bytes);
}

nvfp4_status nvfp4_mx_quantize(const void* x, int32_t in_dtype, int64_t rows, int64_t cols,
                               int64_t ld, int32_t mode, int32_t fmt, void* codes, void* scales,
                               void* scales_sw, nvfp4_stream stream) {
  return mx_quantize_impl(x, in_dtype, rows, cols, ld, mode, fmt, codes, scales, scales_sw,
                          static_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_mx_gemm(const void* a_codes, const void* a_scales_sw, const void* b_codes,
                           const void* b_scales_sw, int32_t fmt, void* D, int64_t M, int64_t N,
                           int64_t K, nvfp4_stream stream) {
  return gemm_mx_impl(a_codes, a_scales_sw, b_codes, b_scales_sw, fmt, D, M, N, K,
                      static_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_gemm(const nvfp4_tensor* A, int32_t a_view, const nvfp4_tensor* B,
                        int32_t b_view, void* D, int32_t d_mode, const void* C, int64_t M,
                        int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                        nvfp4_stream stream) {
  (void)workspace;
  (void)workspace_bytes;
  return gemm_impl(A, a_view, B, b_view, D, d_mode, C, M, N, K, 0,
                   static_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_gemm_ex(const nvfp4_tensor* A, int32_t a_view, const nvfp4_tensor* B,
                           int32_t b_view, void* D, int32_t d_mode, const void* C, int64_t M,
                           int64_t N, int64_t K, int32_t tile, nvfp4_stream stream) {
  return gemm_impl(A, a_view, B, b_view, D, d_mode, C, M, N, K, tile,
                   static_cast<cudaStream_t>(stream));
}

}  // extern "C"
