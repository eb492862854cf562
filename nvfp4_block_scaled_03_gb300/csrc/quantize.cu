// quantize.cu -- NVFP4 quantisers for sm_103a ("NVFP4 pretraining recipe"
// page, bullets 1-5): per-tensor amax pre-pass, then one pass that computes
// the E4M3 block scales, encodes E2M1 codes (RNE via cvt.rn.satfinite, or
// stochastic rounding from Philox4x32-10) and writes the scales directly in
// the MMA's 128x4 atom layout.
//
// All three modes are bandwidth kernels: 16-byte coalesced loads (8 elements
// per thread), the 1x16 block amax with one warp shuffle (two threads per
// block) or a register-resident block (column mode), and outputs staged in
// shared memory so every global store is a coalesced 4- or 16-byte store.
// Kernels are persistent (grid-stride over tiles).
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;

struct QParams {
  const void* x;
  int64_t rows, cols, ld;  // input [rows, cols], leading dim in elements
  uint32_t flags;
  uint64_t seed, offset;
  uint8_t* codes;
  uint8_t* scales;
  uint8_t* codes_t;
  uint8_t* scales_t;
  float* amax_out;
  float* s_dec_out;
  const float* amax_in;  // NVFP4_AMAX_GIVEN
  float* partials;       // amax pass: written; quantise pass: read
  int num_partials;
};

// ---- loads -----------------------------------------------------------------
NVFP4_DEV void load8(const uint16_t* p, float (&v)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
NVFP4_DEV void load8(const float* p, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// ---- block-wide reductions ---------------------------------------------------
NVFP4_DEV float warp_max(float m) {
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
  return m;
}

// Max over all threads of the CTA (every thread gets the result).
NVFP4_DEV float block_max(float m, float* red) {
  m = warp_max(m);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = m;
  __syncthreads();
  if (warp == 0) {
    float t = lane < (int)(blockDim.x >> 5) ? red[lane] : 0.0f;
    t = warp_max(t);
    if (lane == 0) red[0] = t;
  }
  __syncthreads();
  return red[0];
}

// Per-tensor encode scale at the start of a quantise pass: reduce the amax
// pass's partial maxima (or read the caller's amax); CTA 0 publishes amax and
// s_dec.
NVFP4_DEV float tensor_s_enc(const QParams& p, float* red) {
  float amax;
  if (p.flags & NVFP4_AMAX_GIVEN) {
    amax = *p.amax_in;
  } else {
    float m = 0.0f;
    for (int i = threadIdx.x; i < p.num_partials; i += blockDim.x) m = fmaxf(m, p.partials[i]);
    amax = block_max(m, red);
  }
  const float s_enc = per_tensor_s_enc(amax);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (!(p.flags & NVFP4_AMAX_GIVEN)) *p.amax_out = amax;
    *p.s_dec_out = __fdiv_rn(1.0f, s_enc);
  }
  return s_enc;
}

// ---- random Hadamard transform -----------------------------------------------
// Butterfly stages h < width inside one thread's contiguous elements.
template <int N>
NVFP4_DEV void butterfly_local(float (&v)[N]) {
#pragma unroll
  for (int h = 1; h < N; h <<= 1) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = __fadd_rn(a, b);
        v[i + h] = __fsub_rn(a, b);
      }
    }
  }
}

// Full 16-point transform of one register-resident block: signs, stages
// h = 1, 2, 4, 8, then x 1/4.
NVFP4_DEV void rht16_block(float (&v)[16], uint32_t sign_bits) {
#pragma unroll
  for (int i = 0; i < 16; ++i)
    if ((sign_bits >> i) & 1u) v[i] = -v[i];
  butterfly_local<16>(v);
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __fmul_rn(v[i], 0.25f);
}

// Transform of a block split over a lane pair (lane^1): this thread holds
// elements half*8 .. half*8+7.  Stages h = 1, 2, 4 are local; h = 8 pairs
// element i of the two halves through one shuffle.
NVFP4_DEV void rht16_pair(float (&v)[8], uint32_t sign_bits, int half) {
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if ((sign_bits >> (half * 8 + i)) & 1u) v[i] = -v[i];
  butterfly_local<8>(v);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float o = __shfl_xor_sync(0xFFFFFFFFu, v[i], 1);
    v[i] = half == 0 ? __fadd_rn(v[i], o) : __fsub_rn(o, v[i]);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(v[i], 0.25f);
}

// ---- encode ------------------------------------------------------------------
NVFP4_DEV uint32_t block_scale_code(float a_b, float s_enc) {
  return e4m3_rn_satfinite(__fmul_rn(__fdiv_rn(a_b, 6.0f), s_enc));
}
NVFP4_DEV float encode_factor(uint32_t sc, float s_enc) {
  const float S = e4m3_value(sc);
  return S == 0.0f ? 0.0f : __fdiv_rn(s_enc, S);
}

// 8 elements -> 32 bits of packed codes (element 0 in the lowest nibble).
template <bool SR>
NVFP4_DEV uint32_t encode8(const float (&v)[8], float enc, uint4 w0, uint4 w1) {
  float y[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) y[i] = __fmul_rn(v[i], enc);
  uint32_t out = 0;
  if (SR) {
    const uint32_t r[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) out |= e2m1_sr(y[i], r[i]) << (4 * i);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) out |= e2m1x2_rn(y[2 * i], y[2 * i + 1]) << (8 * i);
  }
  return out;
}

// =============================================================================
// ROW_1X16: tile = 128 rows x 64 columns (one scale atom).  Thread t owns the
// 8-element chunk (row t/8 + 32 i, columns 8 (t%8) ..) for i = 0..3; lanes
// t and t^1 form a 16-element block.
// =============================================================================
template <typename T, bool RHT, bool SR, bool AMAX_ONLY>
__global__ void __launch_bounds__(kThreads) quant_row_kernel(QParams p) {
  __shared__ float red[kThreads / 32];
  __shared__ __align__(16) uint8_t atom[512];
  const int tid = threadIdx.x;
  const int c8 = tid & 7, rsub = tid >> 3, half = c8 & 1;
  const int64_t R = p.rows, C = p.cols;
  const int64_t ntc = (C + 63) / 64, ntiles = ((R + 127) / 128) * ntc;
  const int64_t atoms_per_row = ((C / 16) + 3) / 4;
  const T* x = static_cast<const T*>(p.x);
  const uint32_t sign_bits = RHT ? rht_sign_bits(p.seed) : 0u;
  float s_enc = 0.0f, my_max = 0.0f;
  if (!AMAX_ONLY) s_enc = tensor_s_enc(p, red);

  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t tr = tile / ntc, tc = tile % ntc;
    const int64_t c0 = tc * 64 + c8 * 8;
    float v[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t r = tr * 128 + i * 32 + rsub;
      if (r < R && c0 < C) {
        load8(x + r * p.ld + c0, v[i]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[i][e] = 0.0f;
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t r = tr * 128 + i * 32 + rsub;
      const bool ok = r < R && c0 < C;
      if (RHT) rht16_pair(v[i], sign_bits, half);
      float m = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(v[i][e]));
      m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
      if (AMAX_ONLY) {
        my_max = fmaxf(my_max, m);
        continue;
      }
      const uint32_t sc = ok ? block_scale_code(m, s_enc) : 0u;
      const float enc = encode_factor(sc, s_enc);
      uint4 w0 = make_uint4(0, 0, 0, 0), w1 = w0;
      if (SR && ok) {
        const uint64_t idx = (uint64_t)(r * C + c0);
        w0 = sr_words(p.seed, p.offset, idx);
        w1 = sr_words(p.seed, p.offset, idx + 4);
      }
      const uint32_t packed = encode8<SR>(v[i], enc, w0, w1);
      if (ok) *reinterpret_cast<uint32_t*>(p.codes + r * (C / 2) + c0 / 2) = packed;
      if (half == 0) atom[rsub * 16 + i * 4 + (c8 >> 1)] = (uint8_t)sc;
    }
    if (!AMAX_ONLY) {
      __syncthreads();
      if (tid < 32)
        reinterpret_cast<uint4*>(p.scales + (tr * atoms_per_row + tc) * 512)[tid] =
            reinterpret_cast<const uint4*>(atom)[tid];
      __syncthreads();
    }
  }
  if (AMAX_ONLY) {
    const float m = block_max(my_max, red);
    if (tid == 0) p.partials[blockIdx.x] = m;
  }
}

// =============================================================================
// COL_1X16 (transposing): tile = 64 input rows x 128 input columns, i.e. an
// output tile of 128 rows x 64 columns -- one scale atom.  Loaded coalesced
// into shared memory, then each thread quantises one 16-element column block
// (output row c, 16 consecutive input rows) from registers: RHT butterfly,
// block amax, scale, codes.  Codes and the atom are staged and written out
// as coalesced rows.
// =============================================================================
constexpr int kColTileR = 64, kColTileC = 128, kColPad = 132;

template <typename T, bool RHT, bool SR, bool AMAX_ONLY>
__global__ void __launch_bounds__(kThreads) quant_col_kernel(QParams p) {
  __shared__ __align__(16) float tile_s[kColTileR][kColPad];
  __shared__ __align__(16) uint32_t out_s[kColTileC][9];  // 32 code bytes per row, padded
  __shared__ __align__(16) uint8_t atom[512];
  __shared__ float red[kThreads / 32];
  const int tid = threadIdx.x;
  const int64_t R = p.rows, C = p.cols;  // output is [C, R]
  const int64_t ntc = (C + kColTileC - 1) / kColTileC;
  const int64_t ntiles = ((R + kColTileR - 1) / kColTileR) * ntc;
  const int64_t atoms_per_row = ((R / 16) + 3) / 4;
  const T* x = static_cast<const T*>(p.x);
  const uint32_t sign_bits = RHT ? rht_sign_bits(p.seed) : 0u;
  float s_enc = 0.0f, my_max = 0.0f;
  if (!AMAX_ONLY) s_enc = tensor_s_enc(p, red);

  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t tr = tile / ntc, tc = tile % ntc;
    const int64_t r0 = tr * kColTileR, c0 = tc * kColTileC;
    // load phase: thread -> (row tid/16 + 16 i, chunk tid%16)
    {
      const int ch = tid & 15;
      float v[4][8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int rl = (tid >> 4) + 16 * i;
        const int64_t r = r0 + rl, c = c0 + ch * 8;
        if (r < R && c < C) {
          load8(x + r * p.ld + c, v[i]);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) v[i][e] = 0.0f;
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int rl = (tid >> 4) + 16 * i;
        float4* dst = reinterpret_cast<float4*>(&tile_s[rl][ch * 8]);
        dst[0] = make_float4(v[i][0], v[i][1], v[i][2], v[i][3]);
        dst[1] = make_float4(v[i][4], v[i][5], v[i][6], v[i][7]);
      }
    }
    __syncthreads();
    // compute phase: thread -> (output row c = tid % 128, block j)
#pragma unroll
    for (int it = 0; it < 2; ++it) {
      const int cl = tid & 127, j = (tid >> 7) + 2 * it;
      const bool ok = (c0 + cl < C) && (r0 + 16 * j < R);
      float v[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] = tile_s[16 * j + e][cl];
      if (RHT) rht16_block(v, sign_bits);
      float m = 0.0f;
#pragma unroll
      for (int e = 0; e < 16; ++e) m = fmaxf(m, fabsf(v[e]));
      if (AMAX_ONLY) {
        my_max = fmaxf(my_max, m);
        continue;
      }
      const uint32_t sc = ok ? block_scale_code(m, s_enc) : 0u;
      const float enc = encode_factor(sc, s_enc);
      uint4 w[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                    make_uint4(0, 0, 0, 0)};
      if (SR && ok) {
        const uint64_t idx = (uint64_t)((c0 + cl) * R + r0 + 16 * j);
#pragma unroll
        for (int q = 0; q < 4; ++q) w[q] = sr_words(p.seed, p.offset, idx + 4 * q);
      }
      float lo[8], hi[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        lo[e] = v[e];
        hi[e] = v[8 + e];
      }
      out_s[cl][2 * j] = encode8<SR>(lo, enc, w[0], w[1]);
      out_s[cl][2 * j + 1] = encode8<SR>(hi, enc, w[2], w[3]);
      atom[(cl & 31) * 16 + ((cl >> 5) & 3) * 4 + j] = (uint8_t)sc;
    }
    if (!AMAX_ONLY) {
      __syncthreads();
      // codes: 128 output rows x 8 words
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int wi = tid + kThreads * k;
        const int rl = wi >> 3, word = wi & 7;
        const int64_t orow = c0 + rl;
        if (orow < C && r0 + word * 8 < R)
          *reinterpret_cast<uint32_t*>(p.codes + orow * (R / 2) + r0 / 2 + word * 4) =
              out_s[rl][word];
      }
      if (tid < 32)
        reinterpret_cast<uint4*>(p.scales + (tc * atoms_per_row + tr) * 512)[tid] =
            reinterpret_cast<const uint4*>(atom)[tid];
    }
    __syncthreads();
  }
  if (AMAX_ONLY) {
    const float m = block_max(my_max, red);
    if (tid == 0) p.partials[blockIdx.x] = m;
  }
}

// =============================================================================
// BLOCK_16X16 (weights): tile = 128 x 128 elements = 8 x 8 scale tiles.  Warp
// w owns rows 16w..16w+15; lane -> (row lane/2, half lane%2), 8 elements per
// 16x16 tile.  One warp reduction gives the tile amax.  Writes the K-major
// codes and, with EMIT_T, the nibble-transposed codes built from the same
// codes (the partner row's codes arrive by one shuffle), plus both scale
// layouts.
// =============================================================================
template <typename T, bool SR, bool EMIT_T>
__global__ void __launch_bounds__(kThreads) quant_16x16_kernel(QParams p) {
  __shared__ __align__(16) uint32_t outk_s[128][17];  // 64 code bytes per row, padded
  __shared__ __align__(16) uint8_t outt_s[128][68];
  __shared__ __align__(16) uint8_t atoms_k[2][512];
  __shared__ __align__(16) uint8_t atoms_t[2][512];
  __shared__ float red[kThreads / 32];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nl = lane >> 1, half = lane & 1;
  const int64_t R = p.rows, C = p.cols;
  const int64_t ntc = (C + 127) / 128, ntiles = ((R + 127) / 128) * ntc;
  const int64_t apr_k = ((C / 16) + 3) / 4;  // atoms per 128-row block, K-major view
  const int64_t apr_t = ((R / 16) + 3) / 4;  // transposed view
  const T* x = static_cast<const T*>(p.x);
  const float s_enc = tensor_s_enc(p, red);

  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t tr = tile / ntc, tc = tile % ntc;
    const int64_t r0 = tr * 128, c0 = tc * 128;
    const int rl = warp * 16 + nl;
    const int64_t r = r0 + rl;
    const bool row_ok = r0 + warp * 16 < R;  // rows come in whole 16-row strips
    float v[8][8];
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int64_t c = c0 + t * 16 + half * 8;
      if (row_ok && c < C) {
        load8(x + r * p.ld + c, v[t]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[t][e] = 0.0f;
      }
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      const int64_t c = c0 + t * 16 + half * 8;
      const bool ok = row_ok && (c0 + t * 16 < C);
      float m = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(v[t][e]));
      m = warp_max(m);
      const uint32_t sc = ok ? block_scale_code(m, s_enc) : 0u;
      const float enc = encode_factor(sc, s_enc);
      uint4 w0 = make_uint4(0, 0, 0, 0), w1 = w0;
      if (SR && ok) {
        const uint64_t idx = (uint64_t)(r * C + c);
        w0 = sr_words(p.seed, p.offset, idx);
        w1 = sr_words(p.seed, p.offset, idx + 4);
      }
      const uint32_t packed = encode8<SR>(v[t], enc, w0, w1);
      outk_s[rl][t * 2 + half] = packed;
      if (EMIT_T) {
        const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, packed, 2);  // row rl ^ 1
        if ((nl & 1) == 0) {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const uint32_t b = ((packed >> (4 * e)) & 0xFu) | (((other >> (4 * e)) & 0xFu) << 4);
            outt_s[t * 16 + half * 8 + e][rl >> 1] = (uint8_t)b;
          }
        }
      }
      // scale bytes: K-major rows rl (scale column t), transposed rows t*16+e
      if (half == 0)
        atoms_k[t >> 2][(rl & 31) * 16 + ((rl >> 5) & 3) * 4 + (t & 3)] = (uint8_t)sc;
      if (EMIT_T && lane < 16) {
        const int kr = t * 16 + lane;
        atoms_t[warp >> 2][(kr & 31) * 16 + ((kr >> 5) & 3) * 4 + (warp & 3)] = (uint8_t)sc;
      }
    }
    __syncthreads();
    // K-major codes: 128 rows x 16 words
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int wi = tid + kThreads * k;
      const int row = wi >> 4, word = wi & 15;
      if (r0 + row < R && c0 + word * 8 < C)
        *reinterpret_cast<uint32_t*>(p.codes + (r0 + row) * (C / 2) + c0 / 2 + word * 4) =
            outk_s[row][word];
    }
    if (EMIT_T) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int wi = tid + kThreads * k;
        const int row = wi >> 4, word = wi & 15;
        if (c0 + row < C && r0 + word * 8 < R)
          *reinterpret_cast<uint32_t*>(p.codes_t + (c0 + row) * (R / 2) + r0 / 2 + word * 4) =
              *reinterpret_cast<const uint32_t*>(&outt_s[row][word * 4]);
      }
    }
    if (tid < 64) {
      const int a = tid >> 5, l = tid & 31;
      const int64_t g = tc * 2 + a;  // scale-column group of the K-major view
      if (g < apr_k)
        reinterpret_cast<uint4*>(p.scales + (tr * apr_k + g) * 512)[l] =
            reinterpret_cast<const uint4*>(atoms_k[a])[l];
    } else if (EMIT_T && tid < 128) {
      const int a = (tid - 64) >> 5, l = tid & 31;
      const int64_t g = tr * 2 + a;  // scale-column group of the transposed view
      if (g < apr_t)
        reinterpret_cast<uint4*>(p.scales_t + (tc * apr_t + g) * 512)[l] =
            reinterpret_cast<const uint4*>(atoms_t[a])[l];
    }
    __syncthreads();
  }
}

// ---- host dispatch -------------------------------------------------------------
template <typename T>
void launch_amax(const QParams& p, int mode, int grid, cudaStream_t s) {
  const bool rht = p.flags & NVFP4_RHT;
  if (mode == NVFP4_COL_1X16 && rht)
    quant_col_kernel<T, true, false, true><<<grid, kThreads, 0, s>>>(p);
  else if (mode == NVFP4_ROW_1X16 && rht)
    quant_row_kernel<T, true, false, true><<<grid, kThreads, 0, s>>>(p);
  else  // plain max |x| (row, untransformed column, 16x16)
    quant_row_kernel<T, false, false, true><<<grid, kThreads, 0, s>>>(p);
}

template <typename T>
void launch_quant(const QParams& p, int mode, int grid, cudaStream_t s) {
  const bool rht = p.flags & NVFP4_RHT, sr = p.flags & NVFP4_SR, et = p.flags & NVFP4_EMIT_T;
  if (mode == NVFP4_ROW_1X16) {
    if (rht && sr) quant_row_kernel<T, true, true, false><<<grid, kThreads, 0, s>>>(p);
    else if (rht) quant_row_kernel<T, true, false, false><<<grid, kThreads, 0, s>>>(p);
    else if (sr) quant_row_kernel<T, false, true, false><<<grid, kThreads, 0, s>>>(p);
    else quant_row_kernel<T, false, false, false><<<grid, kThreads, 0, s>>>(p);
  } else if (mode == NVFP4_COL_1X16) {
    if (rht && sr) quant_col_kernel<T, true, true, false><<<grid, kThreads, 0, s>>>(p);
    else if (rht) quant_col_kernel<T, true, false, false><<<grid, kThreads, 0, s>>>(p);
    else if (sr) quant_col_kernel<T, false, true, false><<<grid, kThreads, 0, s>>>(p);
    else quant_col_kernel<T, false, false, false><<<grid, kThreads, 0, s>>>(p);
  } else {
    if (sr && et) quant_16x16_kernel<T, true, true><<<grid, kThreads, 0, s>>>(p);
    else if (sr) quant_16x16_kernel<T, true, false><<<grid, kThreads, 0, s>>>(p);
    else if (et) quant_16x16_kernel<T, false, true><<<grid, kThreads, 0, s>>>(p);
    else quant_16x16_kernel<T, false, false><<<grid, kThreads, 0, s>>>(p);
  }
}

int64_t num_tiles(int mode, int64_t R, int64_t C) {
  if (mode == NVFP4_ROW_1X16) return ((R + 127) / 128) * ((C + 63) / 64);
  if (mode == NVFP4_COL_1X16) return ((R + 63) / 64) * ((C + 127) / 128);
  return ((R + 127) / 128) * ((C + 127) / 128);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// ---- entry point that allocates nothing ---------------------------------------
// Some callers cannot hand the library a workspace: code that runs while a
// CUDA graph is being captured (where cudaMalloc is not permitted), plugins
// that receive only input and output pointers from a host framework, or
// applications whose allocator owns all device memory.  For them the amax
// partial maxima live in a fixed array inside the library instead.
namespace {

constexpr int kNoAllocPartials = kMaxPartials;  // 1024 floats: 4 KB per device
// Lives on every device that loads the library, until the process exits.
// In host code this name is only a stand-in: kernels receive the device
// address obtained with cudaGetSymbolAddress below.
static __device__ __align__(256) float g_noalloc_partials[kNoAllocPartials];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[64] = {};

// Device address of the array on the current device, looked up once per
// device (the first call on a device does this; make that first call before
// any stream capture).
nvfp4_status noalloc_scratch(void** addr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return NVFP4_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_partials) != cudaSuccess || !p) return NVFP4_ERR_CUDA;
    g_noalloc_addr[dev] = p;
  }
  *addr = g_noalloc_addr[dev];
  return NVFP4_OK;
}

}  // namespace
}  // namespace nvfp4

extern "C" nvfp4_status nvfp4_quantize_noalloc(const void* x, int32_t in_dtype, int64_t rows,
                                               int64_t cols, int64_t ld, int32_t mode,
                                               uint32_t flags, uint64_t seed, uint64_t offset,
                                               nvfp4_tensor* out, nvfp4_stream stream) {
  using namespace nvfp4;
  if (mode < NVFP4_ROW_1X16 || mode > NVFP4_BLOCK_16X16 || rows <= 0 || cols <= 0)
    return nvfp4_quantize(x, in_dtype, rows, cols, ld, mode, flags, seed, offset, out, nullptr, 0,
                          stream);  // argument errors are reported as by nvfp4_quantize
  if (flags & NVFP4_AMAX_GIVEN)      // no partial maxima needed
    return quantize_impl(x, in_dtype, rows, cols, ld, mode, flags, seed, offset, out, nullptr, 0,
                         static_cast<cudaStream_t>(stream));
  DeviceInfo dev;
  nvfp4_status st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  // the amax pass writes one partial per CTA: reject what the array cannot hold
  if ((int64_t)dev.sm_count * 4 > kNoAllocPartials) return NVFP4_ERR_WORKSPACE;
  void* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != NVFP4_OK) return st;
  // every partial the quantise pass reads is written by this call's amax pass
  // first, so nothing needs clearing between calls
  return quantize_impl(x, in_dtype, rows, cols, ld, mode, flags, seed, offset, out, scratch,
                       sizeof(float) * kNoAllocPartials, static_cast<cudaStream_t>(stream));
}

namespace nvfp4 {

size_t swizzled_scale_bytes(int64_t rows, int64_t cols) {
  const int64_t prow = (rows + 127) / 128 * 128;
  const int64_t pcol = ((cols / 16) + 3) / 4 * 4;
  return (size_t)(prow * pcol);
}

nvfp4_status quantize_impl(const void* x, int32_t in_dtype, int64_t rows, int64_t cols,
                           int64_t ld, int32_t mode, uint32_t flags, uint64_t seed,
                           uint64_t offset, nvfp4_tensor* out, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
  if (!x || !out || !out->codes || !out->scales || !out->amax || !out->s_dec)
    return NVFP4_ERR_INVALID_ARG;
  if (in_dtype != NVFP4_IN_BF16 && in_dtype != NVFP4_IN_FP32) return NVFP4_ERR_INVALID_ARG;
  if (mode < NVFP4_ROW_1X16 || mode > NVFP4_BLOCK_16X16) return NVFP4_ERR_INVALID_ARG;
  if (flags & ~(uint32_t)(NVFP4_RHT | NVFP4_SR | NVFP4_EMIT_T | NVFP4_AMAX_GIVEN))
    return NVFP4_ERR_INVALID_ARG;
  if ((flags & NVFP4_EMIT_T) && mode != NVFP4_BLOCK_16X16) return NVFP4_ERR_INVALID_ARG;
  if ((flags & NVFP4_RHT) && mode == NVFP4_BLOCK_16X16) return NVFP4_ERR_INVALID_ARG;
  if ((flags & NVFP4_EMIT_T) && (!out->codes_t || !out->scales_t)) return NVFP4_ERR_INVALID_ARG;
  if (rows <= 0 || cols <= 0 || ld < cols) return NVFP4_ERR_SHAPE;
  if (cols % 8) return NVFP4_ERR_SHAPE;
  if (mode == NVFP4_ROW_1X16 && cols % 16) return NVFP4_ERR_SHAPE;
  if (mode == NVFP4_COL_1X16 && rows % 16) return NVFP4_ERR_SHAPE;
  if (mode == NVFP4_BLOCK_16X16 && (rows % 16 || cols % 16)) return NVFP4_ERR_SHAPE;
  const size_t esz = in_dtype == NVFP4_IN_BF16 ? 2 : 4;
  if (!aligned16(x) || (ld * (int64_t)esz) % 16) return NVFP4_ERR_ALIGN;
  if (!aligned16(out->scales) || ((reinterpret_cast<uintptr_t>(out->codes) & 3u) != 0))
    return NVFP4_ERR_ALIGN;
  if ((flags & NVFP4_EMIT_T) &&
      (!aligned16(out->scales_t) || (reinterpret_cast<uintptr_t>(out->codes_t) & 3u)))
    return NVFP4_ERR_ALIGN;
  const bool given = flags & NVFP4_AMAX_GIVEN;
  if (!given && (!workspace || workspace_bytes < kQuantWorkspaceBytes || !aligned16(workspace)))
    return NVFP4_ERR_WORKSPACE;

  DeviceInfo dev;
  nvfp4_status st = current_device(&dev);
  if (st != NVFP4_OK) return st;

  QParams p;
  p.x = x;
  p.rows = rows;
  p.cols = cols;
  p.ld = ld;
  p.flags = flags;
  p.seed = seed;
  p.offset = offset;
  p.codes = static_cast<uint8_t*>(out->codes);
  p.scales = static_cast<uint8_t*>(out->scales);
  p.codes_t = static_cast<uint8_t*>(out->codes_t);
  p.scales_t = static_cast<uint8_t*>(out->scales_t);
  p.amax_out = out->amax;
  p.s_dec_out = out->s_dec;
  p.amax_in = out->amax;
  p.partials = static_cast<float*>(workspace);

  const int64_t tiles_amax = num_tiles(
      (mode == NVFP4_COL_1X16 && (flags & NVFP4_RHT)) ? NVFP4_COL_1X16 : NVFP4_ROW_1X16, rows,
      cols);
  const int grid_amax = (int)std::min<int64_t>(
      std::min<int64_t>(tiles_amax, (int64_t)dev.sm_count * 4), kMaxPartials);
  p.num_partials = grid_amax;
  const int64_t tiles = num_tiles(mode, rows, cols);
  const int grid = (int)std::min<int64_t>(tiles, (int64_t)dev.sm_count * 8);

  if (!given) {
    if (in_dtype == NVFP4_IN_BF16) launch_amax<uint16_t>(p, mode, grid_amax, stream);
    else launch_amax<float>(p, mode, grid_amax, stream);
    if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;
  }
  if (in_dtype == NVFP4_IN_BF16) launch_quant<uint16_t>(p, mode, grid, stream);
  else launch_quant<float>(p, mode, grid, stream);
  if (cudaGetLastError() != cudaSuccess) return NVFP4_ERR_CUDA;

  if (mode == NVFP4_COL_1X16) {
    out->rows = cols;
    out->cols = rows;
  } else {
    out->rows = rows;
    out->cols = cols;
  }
  out->mode = mode;
  out->flags = flags;
  return NVFP4_OK;
}

}  // namespace nvfp4
