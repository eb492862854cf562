// swiglu.cu -- SwiGLU between the MLP's NVFP4 GEMMs (bandwidth kernels, 8
// bf16 per thread per 16-byte access, persistent grid):
//   forward  h = silu(g) * u,  silu(g) = g * sigmoid(g)
//   backward dU = dH * silu(g),  dG = dH * u * sigmoid(g) * (1 + g (1 - sigmoid(g)))
// evaluated in FP32 with the CUDA expf, rounded once to bf16.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;

NVFP4_DEV void unpack8(const uint4 u, float (&v)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
NVFP4_DEV uint4 pack8(const float (&v)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}
NVFP4_DEV float sigmoidf_(float g) { return __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-g))); }

__global__ void __launch_bounds__(kThreads) swiglu_fwd_kernel(const uint4* G, const uint4* U,
                                                               uint4* H, int64_t n8) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8;
       i += (int64_t)gridDim.x * blockDim.x) {
    float g[8], u[8], h[8];
    unpack8(__ldg(G + i), g);
    unpack8(__ldg(U + i), u);
#pragma unroll
    for (int e = 0; e < 8; ++e) h[e] = __fmul_rn(__fmul_rn(g[e], sigmoidf_(g[e])), u[e]);
    H[i] = pack8(h);
  }
}

__global__ void __launch_bounds__(kThreads) swiglu_bwd_kernel(const uint4* dH, const uint4* G,
                                                               const uint4* U, uint4* dG,
                                                               uint4* dU, int64_t n8) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n8;
       i += (int64_t)gridDim.x * blockDim.x) {
    float d[8], g[8], u[8], og[8], ou[8];
    unpack8(__ldg(dH + i), d);
    unpack8(__ldg(G + i), g);
    unpack8(__ldg(U + i), u);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float s = sigmoidf_(g[e]);
      ou[e] = __fmul_rn(d[e], __fmul_rn(g[e], s));
      const float ds = __fmul_rn(s, __fadd_rn(1.0f, __fmul_rn(g[e], __fsub_rn(1.0f, s))));
      og[e] = __fmul_rn(__fmul_rn(d[e], u[e]), ds);
    }
    dG[i] = pack8(og);
    dU[i] = pack8(ou);
  }
}

int grid_for(int64_t n8, int sms) {
  return (int)std::max<int64_t>(1, std::min<int64_t>((n8 + kThreads - 1) / kThreads,
                                                     (int64_t)sms * 8));
}

bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

nvfp4_status swiglu_fwd_impl(const void* G, const void* U, void* H, int64_t n,
                             cudaStream_t stream) {
  if (!G || !U || !H) return NVFP4_ERR_INVALID_ARG;
  if (n <= 0 || n % 8) return NVFP4_ERR_SHAPE;
  if (!a16(G) || !a16(U) || !a16(H)) return NVFP4_ERR_ALIGN;
  DeviceInfo dev;
  nvfp4_status st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  swiglu_fwd_kernel<<<grid_for(n / 8, dev.sm_count), kThreads, 0, stream>>>(
      static_cast<const uint4*>(G), static_cast<const uint4*>(U), static_cast<uint4*>(H), n / 8);
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

nvfp4_status swiglu_bwd_impl(const void* dH, const void* G, const void* U, void* dG, void* dU,
                             int64_t n, cudaStream_t stream) {
  if (!dH || !G || !U || !dG || !dU) return NVFP4_ERR_INVALID_ARG;
  if (n <= 0 || n % 8) return NVFP4_ERR_SHAPE;
  if (!a16(dH) || !a16(G) || !a16(U) || !a16(dG) || !a16(dU)) return NVFP4_ERR_ALIGN;
  DeviceInfo dev;
  nvfp4_status st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  swiglu_bwd_kernel<<<grid_for(n / 8, dev.sm_count), kThreads, 0, stream>>>(
      static_cast<const uint4*>(dH), static_cast<const uint4*>(G), static_cast<const uint4*>(U),
      static_cast<uint4*>(dG), static_cast<uint4*>(dU), n / 8);
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // namespace nvfp4
