// mx.cu -- MXFP4 / MXFP8 quantisers: the comparison formats of the "NVFP4
// pretraining recipe" page ("NVFP4 format and advantages": MXFP4 takes
// 32-element blocks with power-of-two E8M0 scales; MXFP8 the same blocks with
// E4M3 elements).  The conversion is the OCP Microscaling specification's,
// which the page links: a block's shared exponent is floor(log2(amax)) minus
// the element format's largest normal exponent (2 for E2M1, 8 for E4M3),
// clamped to [-127, 127]; each element is v / 2^shared rounded to
// nearest-even and saturated.  No per-tensor scale, no RHT, no stochastic
// rounding.  Readings: an all-zero block takes scale byte 0; a block holding
// a value that is not finite takes 0xFF (the E8M0 NaN) and zero codes;
// negative values that round to zero keep their sign.
#include "common.cuh"
#include "internal.h"

namespace nvfp4 {
namespace {

constexpr int kMxThreads = 256;
constexpr int kMxColTile = 256;  // input columns per CTA in the column mode

template <int FMT>
struct MxElem {
  static constexpr int kEmax = FMT == NVFP4_MXFP8 ? 8 : 2;
};

// floor(log2(a)) of a positive finite float from its bits (subnormals too).
NVFP4_DEV int floor_log2_bits(uint32_t bits) {
  const int e = (int)(bits >> 23);
  return e ? e - 127 : -118 - __clz((int)bits);
}

// E8M0 byte of a block and the element multiplier 2^-shared.
template <int FMT>
NVFP4_DEV uint32_t mx_scale(float amax, bool bad, float* mult) {
  int shared = -127;
  if (amax != 0.0f) shared = floor_log2_bits(__float_as_uint(amax)) - MxElem<FMT>::kEmax;
  shared = max(-127, min(127, shared));
  const int e = -shared;  // in [-127, 127]; 2^-127 is a subnormal float
  *mult = e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);
  return bad ? 0xFFu : (uint32_t)(shared + 127);
}

NVFP4_DEV uint32_t e4m3x2_rn_signed(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;  // lo in the low byte
}

// 8 consecutive elements of a row as floats.
NVFP4_DEV void load8(const uint16_t* p, float (&v)[8]) {
  const uint4 w = *reinterpret_cast<const uint4*>(p);
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(u[i] << 16);
    v[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}
NVFP4_DEV void load8(const float* p, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Blocks of 32 along the columns: four lanes per block, eight elements each.
template <typename T, int FMT>
__global__ void __launch_bounds__(kMxThreads) mx_row_kernel(const T* __restrict__ x, int64_t rows,
                                                            int64_t cols, int64_t ld,
                                                            uint8_t* __restrict__ codes,
                                                            uint8_t* __restrict__ scales,
                                                            uint8_t* __restrict__ scales_sw) {
  const int64_t per_row = cols / 8, total = rows * per_row;
  const int lane = threadIdx.x & 31;
  const int64_t warp0 = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  for (int64_t base = warp0 * 32; base < total; base += nwarps * 32) {
    const int64_t t = base + lane;
    const bool active = t < total;  // total is a multiple of 4: a block's lanes agree
    const int64_t r = active ? t / per_row : 0, q = active ? t % per_row : 0;
    float v[8];
    if (active) {
      load8(x + r * ld + q * 8, v);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.0f;
    }
    float a = 0.0f;
    int bad = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      bad |= !isfinite(v[i]);
      a = fmaxf(a, fabsf(v[i]));
    }
    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2));
    bad |= __shfl_xor_sync(0xFFFFFFFFu, bad, 1);
    bad |= __shfl_xor_sync(0xFFFFFFFFu, bad, 2);
    float m;
    const uint32_t sb = mx_scale<FMT>(a, bad != 0, &m);
    if (!active) continue;
    if (FMT == NVFP4_MXFP4) {
      uint32_t packed = 0;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        packed |= e2m1x2_rn(__fmul_rn(v[2 * i], m), __fmul_rn(v[2 * i + 1], m)) << (8 * i);
      if (bad) packed = 0;
      *reinterpret_cast<uint32_t*>(codes + r * (cols / 2) + q * 4) = packed;
    } else {
      uint32_t w[2];
#pragma unroll
      for (int i = 0; i < 2; ++i)
        w[i] = e4m3x2_rn_signed(__fmul_rn(v[4 * i], m), __fmul_rn(v[4 * i + 1], m)) |
               (e4m3x2_rn_signed(__fmul_rn(v[4 * i + 2], m), __fmul_rn(v[4 * i + 3], m)) << 16);
      if (bad) w[0] = w[1] = 0;
      *reinterpret_cast<uint2*>(codes + r * cols + q * 8) = make_uint2(w[0], w[1]);
    }
    if ((q & 3) == 0) {
      scales[r * (cols / 32) + q / 4] = (uint8_t)sb;
      if (scales_sw) scales_sw[sf_offset(r, q / 4, (cols / 32 + 3) / 4 * 4)] = (uint8_t)sb;
    }
  }
}

// Blocks of 32 along the rows, output transposed ([cols][rows]): a CTA reads
// a tile of 32 rows x kMxColTile columns into shared memory with 16-byte
// loads; thread j then owns the tile's column j (one output block).
template <typename T, int FMT>
__global__ void __launch_bounds__(kMxThreads) mx_col_kernel(const T* __restrict__ x, int64_t rows,
                                                            int64_t cols, int64_t ld,
                                                            uint8_t* __restrict__ codes,
                                                            uint8_t* __restrict__ scales,
                                                            uint8_t* __restrict__ scales_sw) {
  __shared__ float tile[32][kMxColTile + 1];
  const int64_t ctiles = (cols + kMxColTile - 1) / kMxColTile, rblocks = rows / 32;
  for (int64_t tix = blockIdx.x; tix < ctiles * rblocks; tix += gridDim.x) {
    const int64_t rb = tix / ctiles, c0 = (tix % ctiles) * kMxColTile;
    __syncthreads();  // the previous tile's reads are done
    // 32 rows x 256 columns = 1024 pieces of 8 elements, 4 per thread
    for (int p = threadIdx.x; p < 32 * (kMxColTile / 8); p += blockDim.x) {
      const int i = p / (kMxColTile / 8), j8 = (p % (kMxColTile / 8)) * 8;
      float v[8];
      if (c0 + j8 < cols) {  // cols is a multiple of 8
        load8(x + (rb * 32 + i) * ld + c0 + j8, v);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = 0.0f;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) tile[i][j8 + k] = v[k];
    }
    __syncthreads();
    for (int j = threadIdx.x; j < kMxColTile; j += blockDim.x) {
      const int64_t c = c0 + j;
      if (c >= cols) continue;
      float a = 0.0f;
      bool bad = false;
#pragma unroll 8
      for (int i = 0; i < 32; ++i) {
        bad |= !isfinite(tile[i][j]);
        a = fmaxf(a, fabsf(tile[i][j]));
      }
      float m;
      const uint32_t sb = mx_scale<FMT>(a, bad, &m);
      if (FMT == NVFP4_MXFP4) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t word = 0;
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const int i = 8 * k + 2 * b;
            word |= e2m1x2_rn(__fmul_rn(tile[i][j], m), __fmul_rn(tile[i + 1][j], m)) << (8 * b);
          }
          w[k] = bad ? 0u : word;
        }
        *reinterpret_cast<uint4*>(codes + c * (rows / 2) + rb * 16) =
            make_uint4(w[0], w[1], w[2], w[3]);
      } else {
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int i = 4 * k;
          const uint32_t word =
              e4m3x2_rn_signed(__fmul_rn(tile[i][j], m), __fmul_rn(tile[i + 1][j], m)) |
              (e4m3x2_rn_signed(__fmul_rn(tile[i + 2][j], m), __fmul_rn(tile[i + 3][j], m))
               << 16);
          w[k] = bad ? 0u : word;
        }
        uint4* dst = reinterpret_cast<uint4*>(codes + c * rows + rb * 32);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      }
      scales[c * (rows / 32) + rb] = (uint8_t)sb;
      if (scales_sw) scales_sw[sf_offset(c, rb, (rows / 32 + 3) / 4 * 4)] = (uint8_t)sb;
    }
  }
}

template <typename T, int FMT>
nvfp4_status launch_mx(const void* x, int64_t rows, int64_t cols, int64_t ld, int32_t mode,
                       uint8_t* codes, uint8_t* scales, uint8_t* scales_sw, int sms,
                       cudaStream_t stream) {
  const T* xt = static_cast<const T*>(x);
  if (mode == NVFP4_MX_ROW) {
    const int64_t warps = (rows * (cols / 8) + 31) / 32;
    const int64_t grid = std::min<int64_t>((warps * 32 + kMxThreads - 1) / kMxThreads,
                                           (int64_t)sms * 16);
    mx_row_kernel<T, FMT><<<(unsigned)grid, kMxThreads, 0, stream>>>(xt, rows, cols, ld, codes,
                                                                      scales, scales_sw);
  } else {
    const int64_t tiles = ((cols + kMxColTile - 1) / kMxColTile) * (rows / 32);
    const int64_t grid = std::min<int64_t>(tiles, (int64_t)sms * 8);
    mx_col_kernel<T, FMT><<<(unsigned)grid, kMxThreads, 0, stream>>>(xt, rows, cols, ld, codes,
                                                                      scales, scales_sw);
  }
  return cuda_status(cudaGetLastError());
}

}  // namespace

nvfp4_status mx_sizes_impl(int64_t rows, int64_t cols, int32_t mode, int32_t fmt,
                           size_t* codes_bytes, size_t* scales_bytes, size_t* scales_sw_bytes) {
  if ((mode != NVFP4_MX_ROW && mode != NVFP4_MX_COL) || (fmt != NVFP4_MXFP4 && fmt != NVFP4_MXFP8))
    return NVFP4_ERR_INVALID_ARG;
  if (rows <= 0 || cols <= 0) return NVFP4_ERR_SHAPE;
  const int64_t orows = mode == NVFP4_MX_COL ? cols : rows;
  const int64_t ocols = mode == NVFP4_MX_COL ? rows : cols;
  if (ocols % 32 || (mode == NVFP4_MX_COL && cols % 8)) return NVFP4_ERR_SHAPE;
  if (codes_bytes) *codes_bytes = (size_t)(orows * (fmt == NVFP4_MXFP4 ? ocols / 2 : ocols));
  if (scales_bytes) *scales_bytes = (size_t)(orows * (ocols / 32));
  // the MMA layout: 512-byte atoms of 128 rows x 4 scale columns, padded
  if (scales_sw_bytes)
    *scales_sw_bytes = (size_t)(((orows + 127) / 128) * ((ocols / 32 + 3) / 4) * 512);
  return NVFP4_OK;
}

nvfp4_status mx_quantize_impl(const void* x, int32_t in_dtype, int64_t rows, int64_t cols,
                              int64_t ld, int32_t mode, int32_t fmt, void* codes, void* scales,
                              void* scales_sw, cudaStream_t stream) {
  if (!x || !codes || !scales) return NVFP4_ERR_INVALID_ARG;
  if (in_dtype != NVFP4_IN_BF16 && in_dtype != NVFP4_IN_FP32) return NVFP4_ERR_INVALID_ARG;
  size_t sw_bytes = 0;
  nvfp4_status st = mx_sizes_impl(rows, cols, mode, fmt, nullptr, nullptr, &sw_bytes);
  if (st != NVFP4_OK) return st;
  if (ld < cols || rows > INT32_MAX || cols > INT32_MAX) return NVFP4_ERR_SHAPE;
  const int64_t esize = in_dtype == NVFP4_IN_BF16 ? 2 : 4;
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (ld * esize) % 16 ||
      (reinterpret_cast<uintptr_t>(codes) & 15))
    return NVFP4_ERR_ALIGN;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  uint8_t* c = static_cast<uint8_t*>(codes);
  uint8_t* s = static_cast<uint8_t*>(scales);
  uint8_t* sw = static_cast<uint8_t*>(scales_sw);
  const int64_t orows = mode == NVFP4_MX_COL ? cols : rows;
  const int64_t ocols = mode == NVFP4_MX_COL ? rows : cols;
  // padding entries of the MMA layout (rows to 128, scale columns to 4) read
  // as zero
  if (sw && (orows % 128 || (ocols / 32) % 4) &&
      cudaMemsetAsync(sw, 0, sw_bytes, stream) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  const bool bf = in_dtype == NVFP4_IN_BF16;
  const int n = dev.sm_count;
  if (fmt == NVFP4_MXFP4)
    return bf ? launch_mx<uint16_t, NVFP4_MXFP4>(x, rows, cols, ld, mode, c, s, sw, n, stream)
              : launch_mx<float, NVFP4_MXFP4>(x, rows, cols, ld, mode, c, s, sw, n, stream);
  return bf ? launch_mx<uint16_t, NVFP4_MXFP8>(x, rows, cols, ld, mode, c, s, sw, n, stream)
            : launch_mx<float, NVFP4_MXFP8>(x, rows, cols, ld, mode, c, s, sw, n, stream);
}

}  // namespace nvfp4
