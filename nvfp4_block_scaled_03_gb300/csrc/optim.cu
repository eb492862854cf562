// optim.cu -- the optimizer step of an FP32 master weight, fused with the
// amax its next NVFP4 quantisation needs.
//
// "NVFP4 pretraining recipe" page, Figure 1 text: the MLP GEMMs' BF16
// outputs end up folded into FP32 master weights on the optimizer step, and
// each step quantises the weights 16x16 under a per-tensor FP32 scale, which
// is computed from the tensor's amax.  Taking that amax while the update
// writes the weight removes the quantiser's own amax pass (one full read of
// the FP32 weight per step).  The pages name no optimizer; the update is
// plain SGD, elementwise in binary32 with the product rounded first:
//   W[i] <- W[i] - lr * G[i]
//   G[i] <- 0                  (NVFP4_ZERO_GRAD: ready for the next fold)
//   amax  = max_i |W[i]|       over the values written
// Work: persistent grid-stride over 16-byte chunks, four chunks of W and of
// G in flight per thread; one partial maximum per CTA, reduced by a second
// one-CTA launch (deterministic: a maximum does not depend on the order).
#include <algorithm>
#include <atomic>
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

NVFP4_DEV float sgd1(float w, float g, float lr) { return __fsub_rn(w, __fmul_rn(lr, g)); }

template <bool ZERO, bool AMAX>
__global__ void __launch_bounds__(kThreads) sgd_amax_kernel(float* __restrict__ W,
                                                            float* __restrict__ G, int64_t n4,
                                                            float lr, float* partials) {
  __shared__ float red[kThreads / 32];
  float4* w4 = reinterpret_cast<float4*>(W);
  float4* g4 = reinterpret_cast<float4*>(G);
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  float m = 0.0f;
  for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < n4; i += kUnroll * stride) {
    float4 w[kUnroll], g[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t q = i + u * stride;
      if (q < n4) {
        w[u] = w4[q];
        g[u] = g4[q];
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t q = i + u * stride;
      if (q < n4) {
        const float4 r = make_float4(sgd1(w[u].x, g[u].x, lr), sgd1(w[u].y, g[u].y, lr),
                                     sgd1(w[u].z, g[u].z, lr), sgd1(w[u].w, g[u].w, lr));
        w4[q] = r;
        if (ZERO) g4[q] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (AMAX)
          m = fmaxf(m, fmaxf(fmaxf(fabsf(r.x), fabsf(r.y)), fmaxf(fabsf(r.z), fabsf(r.w))));
      }
    }
  }
  if (AMAX) {
    m = block_max(m, red);
    if (threadIdx.x == 0) partials[blockIdx.x] = m;
  }
}

__global__ void __launch_bounds__(kThreads) sgd_amax_finalize_kernel(const float* partials, int n,
                                                                     float* amax) {
  __shared__ float red[kThreads / 32];
  float m = 0.0f;
  for (int i = threadIdx.x; i < n; i += kThreads) m = fmaxf(m, partials[i]);
  m = block_max(m, red);
  if (threadIdx.x == 0) *amax = m;
}

// CTAs of a persistent launch: as many as are resident at once (looked up
// once per kernel and device), at most one partial slot each, at most one
// per kThreads chunks.
template <auto KERN>
int sgd_grid(int64_t n4, int sms) {
  static std::atomic<int> fit[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) dev = 0;
  int per_sm = fit[dev].load(std::memory_order_relaxed);
  if (per_sm == 0) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, KERN, kThreads, 0) !=
            cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    fit[dev].store(per_sm, std::memory_order_relaxed);
  }
  const int64_t want = std::max<int64_t>(1, (n4 + kThreads - 1) / kThreads);
  return (int)std::min<int64_t>(std::min<int64_t>(want, (int64_t)sms * per_sm), kMaxPartials);
}

template <bool ZERO, bool AMAX>
nvfp4_status launch_sgd(float* W, float* G, int64_t n4, float lr, float* partials, int sms,
                        int* grid, cudaStream_t s) {
  auto kern = sgd_amax_kernel<ZERO, AMAX>;
  *grid = sgd_grid<sgd_amax_kernel<ZERO, AMAX>>(n4, sms);
  kern<<<*grid, kThreads, 0, s>>>(W, G, n4, lr, partials);
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" nvfp4_status nvfp4_sgd_step(float* W, float* G, int64_t n, float lr, uint32_t flags,
                                       float* amax, void* workspace, size_t workspace_bytes,
                                       nvfp4_stream stream) {
  if (!W || !G || (flags & ~(uint32_t)NVFP4_ZERO_GRAD) || !std::isfinite(lr))
    return NVFP4_ERR_INVALID_ARG;
  if (n <= 0 || n % 4) return NVFP4_ERR_SHAPE;
  const uintptr_t wb = reinterpret_cast<uintptr_t>(W), gb = reinterpret_cast<uintptr_t>(G);
  const uintptr_t bytes = (uintptr_t)n * sizeof(float);
  if (wb < gb + bytes && gb < wb + bytes) return NVFP4_ERR_INVALID_ARG;  // overlap
  if (!a16(W) || !a16(G) || (reinterpret_cast<uintptr_t>(amax) & 3u)) return NVFP4_ERR_ALIGN;
  if (amax && (!workspace || workspace_bytes < kQuantWorkspaceBytes || !a16(workspace)))
    return NVFP4_ERR_WORKSPACE;
  DeviceInfo dev;
  nvfp4_status st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float* partials = static_cast<float*>(workspace);
  const int64_t n4 = n / 4;
  const bool zero = flags & NVFP4_ZERO_GRAD;
  int grid = 0;
  if (amax) {
    st = zero ? launch_sgd<true, true>(W, G, n4, lr, partials, dev.sm_count, &grid, s)
              : launch_sgd<false, true>(W, G, n4, lr, partials, dev.sm_count, &grid, s);
    if (st != NVFP4_OK) return st;
    sgd_amax_finalize_kernel<<<1, kThreads, 0, s>>>(partials, grid, amax);
    return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
  }
  return zero ? launch_sgd<true, false>(W, G, n4, lr, nullptr, dev.sm_count, &grid, s)
              : launch_sgd<false, false>(W, G, n4, lr, nullptr, dev.sm_count, &grid, s);
}
