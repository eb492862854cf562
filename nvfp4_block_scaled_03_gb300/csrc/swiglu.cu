// swiglu.cu -- SwiGLU between the MLP's NVFP4 GEMMs:
//   forward  h = silu(g) * u,  silu(g) = g * sigmoid(g)
//   backward dU = dH * silu(g),  dG = dH * u * sigmoid(g) * (1 + g (1 - sigmoid(g)))
// evaluated in FP32 with the CUDA expf and __fdividef, rounded once to bf16.
//
// Each output feeds two NVFP4 quantisations (row-wise for FPROP / DGRAD,
// column-wise for WGRAD, "NVFP4 pretraining recipe" page, bullets 3-5), whose
// per-tensor scales need the output's amax -- and, with the random Hadamard
// transform on the WGRAD operand, max |RHT(column block)|.  The kernels take
// both from the bf16 values they store, so nothing re-reads H, dG or dU
// before quantising them.
//
// Work unit: a warp tile of 16 rows x 64 columns.  Lane l covers columns
// 8 (l % 8) .. +7 of rows l / 8 + 4 j, j = 0..3: each warp access reads or
// writes 128 contiguous bytes of each of 4 rows (the 8 warps of a CTA take
// adjacent tiles: 1 KB of each row).  With the transform the warp leaves its
// bf16 results in a shared-memory tile; then lane l reads columns 2 l and
// 2 l + 1 of it -- two whole 16-row column blocks -- and takes their
// transforms in registers, the quantiser's own arithmetic.

#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace nvfp4 {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSetStride = kMaxPartials;  // partial maxima of one amax set

NVFP4_DEV void unpack8(const uint4 u, float (&v)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
// Rounds to bf16; v keeps the rounded values (what the amaxes are taken of).
NVFP4_DEV uint4 pack8(float (&v)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// sigmoid(g) = 1 / (1 + e^-g) for g >= 0 and e^g / (1 + e^g) below: the same
// function, with e^-|g| <= 1 so nothing overflows (1 / (1 + e^-g) alone
// would give 0 once e^-g passes FLT_MAX, at g < -88.7, where silu(g) * u is
// still a normal bf16 value).  The denominator lies in [1, 2], where the fast
// quotient __fdividef is within 2 ulp.
NVFP4_DEV float sigmoidf_(float g) {
  const float t = expf(-fabsf(g));
  return __fdividef(g >= 0.0f ? 1.0f : t, __fadd_rn(1.0f, t));
}

// Shared-memory tile of one warp: 16 rows of 64 bf16, rows 144 bytes apart
// (a warp's 16-byte stores -- 8 lanes per row, 4 rows -- and its 32-bit
// column-pair reads -- 32 lanes, one row -- are free of bank conflicts).
constexpr int kRowU16 = 72;
constexpr int kTileU16 = 16 * kRowU16;

struct Tile {
  int64_t at;  // element offset of this lane's row l / 8, first column
  bool live;   // its 8 columns inside the tensor
};
NVFP4_DEV Tile lane_tile(int64_t w, int64_t tpr, int64_t cols, int lane) {
  const int64_t jb = w / tpr, tc = w - jb * tpr;
  const int64_t c = tc * 64 + (lane & 7) * 8;
  return {(jb * 16 + (lane >> 3)) * cols + c, c < cols};
}

NVFP4_DEV void tile_put(uint16_t* tile, int lane, int j, uint4 v) {
  *reinterpret_cast<uint4*>(tile + ((lane >> 3) + 4 * j) * kRowU16 + (lane & 7) * 8) = v;
}

// Columns 2 lane and 2 lane + 1 of the warp's tile: max |x| into mp and the
// 16-point transform of each into mr as max |sum| before the final x 1/4.
NVFP4_DEV void column_amax(const uint16_t* tile, int lane, uint32_t sign_bits, float& mp,
                           float& mr) {
  float a[16], b[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(tile + e * kRowU16 + 2 * lane);
    a[e] = __uint_as_float(w << 16);
    b[e] = __uint_as_float(w & 0xFFFF0000u);
    mp = fmaxf(mp, fmaxf(fabsf(a[e]), fabsf(b[e])));
  }
  mr = fmaxf(mr, fmaxf(rht16_absmax_unscaled(a, sign_bits), rht16_absmax_unscaled(b, sign_bits)));
}

// The transform's x 1/4 on the maximum instead of on every sum: rounding is
// monotone, so the maximum is the same bit for bit.
NVFP4_DEV float rht_scale(float mr) { return __fmul_rn(mr, 0.25f); }

NVFP4_DEV void load8(const uint16_t* p, bool live, float (&v)[8]) {
  if (live) {
    unpack8(__ldg(reinterpret_cast<const uint4*>(p)), v);
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = 0.0f;
  }
}

NVFP4_DEV float abs_max8(const float (&v)[8]) {
  float m = 0.0f;
#pragma unroll
  for (int k = 0; k < 8; ++k) m = fmaxf(m, fabsf(v[k]));
  return m;
}

template <bool RHT>
__global__ void __launch_bounds__(kThreads) swiglu_fwd_kernel(const uint16_t* G, const uint16_t* U,
                                                               uint16_t* H, int64_t rows,
                                                               int64_t cols, uint64_t seed,
                                                               float* partials) {
  __shared__ float red[kWarps];
  __shared__ __align__(16) uint16_t tiles[RHT ? kWarps * kTileU16 : 8];
  const uint32_t sign_bits = RHT ? rht_sign_bits(seed) : 0u;
  const int lane = threadIdx.x & 31;
  uint16_t* tile = tiles + (RHT ? (threadIdx.x >> 5) * kTileU16 : 0);
  const int64_t tpr = (cols + 63) / 64, n = (rows / 16) * tpr, step = 4 * cols;
  float mp = 0.0f, mr = 0.0f;
  for (int64_t w = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); w < n;
       w += (int64_t)gridDim.x * kWarps) {
    const Tile t = lane_tile(w, tpr, cols, lane);
    if (RHT) __syncwarp();  // the previous tile's column reads are done
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float g[8], u[8], h[8];
      load8(G + t.at + j * step, t.live, g);
      load8(U + t.at + j * step, t.live, u);
#pragma unroll
      for (int k = 0; k < 8; ++k) h[k] = __fmul_rn(__fmul_rn(g[k], sigmoidf_(g[k])), u[k]);
      const uint4 o = pack8(h);
      if (t.live) *reinterpret_cast<uint4*>(H + t.at + j * step) = o;
      if (RHT)
        tile_put(tile, lane, j, o);
      else
        mp = fmaxf(mp, abs_max8(h));
    }
    if (RHT) {
      __syncwarp();
      column_amax(tile, lane, sign_bits, mp, mr);
    }
  }
  mp = block_max(mp, red);
  if (threadIdx.x == 0) partials[blockIdx.x] = mp;
  if (RHT) {
    mr = block_max(rht_scale(mr), red);
    if (threadIdx.x == 0) partials[kSetStride + blockIdx.x] = mr;
  }
}

template <bool RHT>
__global__ void __launch_bounds__(kThreads) swiglu_bwd_kernel(const uint16_t* dH,
                                                               const uint16_t* G,
                                                               const uint16_t* U, uint16_t* dG,
                                                               uint16_t* dU, int64_t rows,
                                                               int64_t cols, uint64_t seed,
                                                               float* partials) {
  __shared__ float red[kWarps];
  __shared__ __align__(16) uint16_t tiles[RHT ? 2 * kWarps * kTileU16 : 8];
  const uint32_t sign_bits = RHT ? rht_sign_bits(seed) : 0u;
  const int lane = threadIdx.x & 31;
  uint16_t* tile_g = tiles + (RHT ? (threadIdx.x >> 5) * 2 * kTileU16 : 0);
  uint16_t* tile_u = tile_g + (RHT ? kTileU16 : 0);
  const int64_t tpr = (cols + 63) / 64, n = (rows / 16) * tpr, step = 4 * cols;
  float mpg = 0.0f, mrg = 0.0f, mpu = 0.0f, mru = 0.0f;
  for (int64_t w = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5); w < n;
       w += (int64_t)gridDim.x * kWarps) {
    const Tile t = lane_tile(w, tpr, cols, lane);
    if (RHT) __syncwarp();  // the previous tile's column reads are done
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t at = t.at + j * step;
      float d[8], g[8], u[8], rg[8], ru[8];
      load8(dH + at, t.live, d);
      load8(G + at, t.live, g);
      load8(U + at, t.live, u);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float s = sigmoidf_(g[k]);
        ru[k] = __fmul_rn(d[k], __fmul_rn(g[k], s));
        const float ds = __fmul_rn(s, __fadd_rn(1.0f, __fmul_rn(g[k], __fsub_rn(1.0f, s))));
        rg[k] = __fmul_rn(__fmul_rn(d[k], u[k]), ds);
      }
      const uint4 og = pack8(rg), ou = pack8(ru);
      if (t.live) {
        *reinterpret_cast<uint4*>(dG + at) = og;
        *reinterpret_cast<uint4*>(dU + at) = ou;
      }
      if (RHT) {
        tile_put(tile_g, lane, j, og);
        tile_put(tile_u, lane, j, ou);
      } else {
        mpg = fmaxf(mpg, abs_max8(rg));
        mpu = fmaxf(mpu, abs_max8(ru));
      }
    }
    if (RHT) {
      __syncwarp();
      column_amax(tile_g, lane, sign_bits, mpg, mrg);
      column_amax(tile_u, lane, sign_bits, mpu, mru);
    }
  }
  // sets: 0 = dG plain, 1 = dU plain, 2 = dG RHT, 3 = dU RHT
  mpg = block_max(mpg, red);
  if (threadIdx.x == 0) partials[blockIdx.x] = mpg;
  mpu = block_max(mpu, red);
  if (threadIdx.x == 0) partials[kSetStride + blockIdx.x] = mpu;
  if (RHT) {
    mrg = block_max(rht_scale(mrg), red);
    if (threadIdx.x == 0) partials[2 * kSetStride + blockIdx.x] = mrg;
    mru = block_max(rht_scale(mru), red);
    if (threadIdx.x == 0) partials[3 * kSetStride + blockIdx.x] = mru;
  }
}

// Where each set's maximum goes: dst[k][0] and, when set, dst[k][1].
struct AmaxDst {
  float* dst[4][2];
};

// CTA k reduces the n partial maxima of set k.
__global__ void __launch_bounds__(kThreads) swiglu_amax_finalize_kernel(const float* partials,
                                                                        int n, AmaxDst out) {
  __shared__ float red[kThreads / 32];
  const float* p = partials + (int64_t)blockIdx.x * kSetStride;
  float m = 0.0f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) m = fmaxf(m, p[i]);
  m = block_max(m, red);
  if (threadIdx.x == 0) {
    *out.dst[blockIdx.x][0] = m;
    if (out.dst[blockIdx.x][1]) *out.dst[blockIdx.x][1] = m;
  }
}

// Persistent grid: a multiple of the SM count (as many CTAs per SM as fit,
// within one set's partial slots), no more CTAs than warp tiles need.  The
// CTAs that fit per SM are looked up once per kernel and device.
template <auto KERN>
int grid_for(int64_t tiles, int sms) {
  static std::atomic<int> fit[64];  // one cache per kernel
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
  per_sm = std::max(1, std::min(per_sm, kSetStride / std::max(sms, 1)));
  const int64_t want = std::max<int64_t>(1, (tiles + kWarps - 1) / kWarps);
  return (int)std::min<int64_t>(std::min<int64_t>(want, (int64_t)sms * per_sm), kSetStride);
}

bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool a4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

nvfp4_status check_shape(int64_t rows, int64_t cols, void* partials, size_t partials_bytes) {
  if (rows <= 0 || cols <= 0 || rows % 16 || cols % 8) return NVFP4_ERR_SHAPE;
  if (!partials || partials_bytes < kSwigluPartialsBytes || !a16(partials))
    return NVFP4_ERR_WORKSPACE;
  return NVFP4_OK;
}

}  // namespace

nvfp4_status swiglu_fwd_impl(const void* G, const void* U, void* H, int64_t rows, int64_t cols,
                             uint64_t seed, bool rht, float* amax_row, float* amax_col,
                             void* partials, size_t partials_bytes, cudaStream_t stream) {
  if (!G || !U || !H || !amax_row || !amax_col) return NVFP4_ERR_INVALID_ARG;
  nvfp4_status st = check_shape(rows, cols, partials, partials_bytes);
  if (st != NVFP4_OK) return st;
  if (!a16(G) || !a16(U) || !a16(H) || !a4(amax_row) || !a4(amax_col)) return NVFP4_ERR_ALIGN;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  const int64_t tiles = (rows / 16) * ((cols + 63) / 64);
  float* pp = static_cast<float*>(partials);
  const auto* g = static_cast<const uint16_t*>(G);
  const auto* u = static_cast<const uint16_t*>(U);
  auto* h = static_cast<uint16_t*>(H);
  int grid;
  AmaxDst out{};
  if (rht) {
    grid = grid_for<swiglu_fwd_kernel<true>>(tiles, dev.sm_count);
    swiglu_fwd_kernel<true><<<grid, kThreads, 0, stream>>>(g, u, h, rows, cols,
                                                           seed, pp);
    out.dst[0][0] = amax_row;
    out.dst[1][0] = amax_col;
  } else {
    grid = grid_for<swiglu_fwd_kernel<false>>(tiles, dev.sm_count);
    swiglu_fwd_kernel<false><<<grid, kThreads, 0, stream>>>(g, u, h, rows, cols, 0, pp);
    out.dst[0][0] = amax_row;
    out.dst[0][1] = amax_col;
  }
  swiglu_amax_finalize_kernel<<<rht ? 2 : 1, kThreads, 0, stream>>>(pp, grid, out);
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

nvfp4_status swiglu_bwd_impl(const void* dH, const void* G, const void* U, void* dG, void* dU,
                             int64_t rows, int64_t cols, uint64_t seed, bool rht,
                             float* amax_dg_row, float* amax_dg_col, float* amax_du_row,
                             float* amax_du_col, void* partials, size_t partials_bytes,
                             cudaStream_t stream) {
  if (!dH || !G || !U || !dG || !dU || !amax_dg_row || !amax_dg_col || !amax_du_row ||
      !amax_du_col)
    return NVFP4_ERR_INVALID_ARG;
  nvfp4_status st = check_shape(rows, cols, partials, partials_bytes);
  if (st != NVFP4_OK) return st;
  if (!a16(dH) || !a16(G) || !a16(U) || !a16(dG) || !a16(dU) || !a4(amax_dg_row) ||
      !a4(amax_dg_col) || !a4(amax_du_row) || !a4(amax_du_col))
    return NVFP4_ERR_ALIGN;
  DeviceInfo dev;
  st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  const int64_t tiles = (rows / 16) * ((cols + 63) / 64);
  float* pp = static_cast<float*>(partials);
  const auto* d = static_cast<const uint16_t*>(dH);
  const auto* g = static_cast<const uint16_t*>(G);
  const auto* u = static_cast<const uint16_t*>(U);
  auto* og = static_cast<uint16_t*>(dG);
  auto* ou = static_cast<uint16_t*>(dU);
  int grid;
  AmaxDst out{};
  out.dst[0][0] = amax_dg_row;
  out.dst[1][0] = amax_du_row;
  if (rht) {
    grid = grid_for<swiglu_bwd_kernel<true>>(tiles, dev.sm_count);
    swiglu_bwd_kernel<true><<<grid, kThreads, 0, stream>>>(d, g, u, og, ou, rows, cols,
                                                           seed, pp);
    out.dst[2][0] = amax_dg_col;
    out.dst[3][0] = amax_du_col;
  } else {
    grid = grid_for<swiglu_bwd_kernel<false>>(tiles, dev.sm_count);
    swiglu_bwd_kernel<false><<<grid, kThreads, 0, stream>>>(d, g, u, og, ou, rows, cols, 0, pp);
    out.dst[0][1] = amax_dg_col;
    out.dst[1][1] = amax_du_col;
  }
  swiglu_amax_finalize_kernel<<<rht ? 4 : 2, kThreads, 0, stream>>>(pp, grid, out);
  return cudaGetLastError() == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

}  // namespace nvfp4
