// quantize.cu -- NVFP4 quantisers for sm_103a ("NVFP4 pretraining recipe"
// page, bullets 1-5): per-tensor amax pre-pass, then one pass that computes
// the E4M3 block scales, encodes E2M1 codes (RNE via cvt.rn.satfinite, or
// stochastic rounding from Philox4x32-10) and writes the scales directly in
// the MMA's 128x4 atom layout.
//
// The quantise pass is a persistent, warp-specialised kernel: one producer
// thread streams input tiles into a ring of shared-memory stages with TMA
// (boxes of 128-byte rows, 128-byte swizzle, zeros past the tensor's edges)
// while eight consumer warps turn each stage into codes and scales.  A stage
// is handed back as soon as its values sit in registers, so HBM reads run
// ahead of the encoding.  Outputs leave through coalesced stores, staged in
// shared memory per warp (or, for the transposing mode, per CTA behind a
// bounded mbarrier).  The amax pre-pass is a plain bandwidth kernel with
// wide loads and several loads in flight per thread.
//
// Every wait is bounded (2 s via %globaltimer): on expiry the kernel records
// a code in the quantiser error word, raises its CTA's abort flag, the
// producer waits (bounded) for the copies it issued and the CTA exits.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace nvfp4 {

static __device__ unsigned int g_quant_error;
// Failure injection for tests of the bounded waits (nvfp4_debug_inject):
// while g_q_stall is set the quantise passes' producers issue no loads, so
// the consumers' waits run out; pipeline waits give up after g_q_wait_ns.
static __device__ unsigned int g_q_stall;
static __device__ unsigned long long g_q_wait_ns = 2000000000ull;

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kQThreads = kConsumers + 32;  // + one producer warp
constexpr int kAmaxThreads = 256;
constexpr uint64_t kQWaitNs = 2000000000ull;

struct QParams {
  int64_t rows, cols, ld;  // input [rows, cols], leading dim in elements
  uint32_t flags;
  uint64_t seed, offset;
  const void* x;           // amax pass only (the quantise pass reads through TMA)
  uint8_t* codes;
  uint8_t* scales;
  uint8_t* codes_t;
  uint8_t* scales_t;
  float* amax_out;
  float* s_dec_out;
  const float* amax_in;  // NVFP4_AMAX_GIVEN
  float* partials;       // amax pass: written; quantise pass: read
  int num_partials;
  int codes_vec16;       // codes (and rows of codes) 16-byte aligned
  int codes_t_vec8;      // transposed codes 8-byte aligned
  PhiloxKeys rk;         // round keys of the stochastic-rounding generator (key = seed)
};

// ---- tile geometry -------------------------------------------------------------
// A stage holds a tile of TR rows x TC columns of the input as NBOX TMA boxes
// of TR rows x 128 bytes, each box 128-byte swizzled (the 16-byte chunk c of
// row r sits at chunk c ^ (r % 8)), so row-wise and column-wise reads of the
// stage are free of bank conflicts.
template <typename T, int TR, int TC, int STAGES>
struct Geo {
  static constexpr int kTR = TR, kTC = TC, kStages = STAGES;
  static constexpr int kBoxCols = 128 / (int)sizeof(T);
  static constexpr int kNBox = TC / kBoxCols;
  static constexpr uint32_t kBoxBytes = TR * 128;
  static constexpr uint32_t kStageBytes = kNBox * kBoxBytes;
  static_assert(TC % kBoxCols == 0 && TR % 8 == 0, "tile shape");
};
template <typename T>
using RowGeo = Geo<T, 128, 64, sizeof(T) == 2 ? 4 : 3>;
template <typename T>
using ColGeo = Geo<T, 64, 128, sizeof(T) == 2 ? 4 : 3>;
template <typename T>
using BlkGeo = Geo<T, 128, 64, sizeof(T) == 2 ? 4 : 3>;

// Shared memory: stages (1024-byte aligned for the swizzle), kernel-specific
// staging, the encode table, reduction scratch, barriers, abort flag.
template <class G, int EXTRA>
struct QSmem {
  static constexpr uint32_t offExtra = G::kStages * G::kStageBytes;
  static constexpr uint32_t offTab = offExtra + EXTRA;
  static constexpr uint32_t offRed = offTab + 512;
  static constexpr uint32_t offBar = offRed + 64;  // full[S], empty[S], out[2]
  static constexpr uint32_t offMisc = offBar + 8 * (2 * G::kStages + 2);
  static constexpr uint32_t kBytes = offMisc + 16;
  static constexpr uint32_t kAlloc = kBytes + 1024;
  static_assert(EXTRA % 16 == 0, "staging alignment");
};

NVFP4_DEV uint8_t* align_smem_1024(uint8_t* raw) {
  return raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
}

// Tile row and column (tile = tr * ntc + tc) of a CTA's tiles, which step by
// the grid size: advanced by an add and a carry per tile instead of a 64-bit
// division and remainder.  32-bit: the launchers refuse more than 2^30 tiles
// (a tile is 8192 elements, so no tensor that fits in memory has as many).
struct TileWalk {
  int32_t tr, tc, dr, dc, ntc;
  NVFP4_DEV TileWalk(int32_t tile0, int32_t step, int32_t n)
      : tr(tile0 / n), tc(tile0 % n), dr(step / n), dc(step % n), ntc(n) {}
  NVFP4_DEV void next() {
    tc += dc;
    tr += dr;
    if (tc >= ntc) {
      tc -= ntc;
      ++tr;
    }
  }
};

// Byte offset of (row r, byte b of the tile row) inside a stage.
template <class G>
NVFP4_DEV uint32_t swz(int r, int b) {
  return (uint32_t)(b >> 7) * G::kBoxBytes + (uint32_t)r * 128u +
         ((uint32_t)(((b >> 4) & 7) ^ (r & 7)) << 4) + (uint32_t)(b & 15);
}

// 8 consecutive elements starting at column c of row r.
template <class G>
NVFP4_DEV void lds8(const uint8_t* st, int r, int c, const uint16_t*, float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(st + swz<G>(r, c * 2));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
template <class G>
NVFP4_DEV void lds8(const uint8_t* st, int r, int c, const float*, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(st + swz<G>(r, c * 4));
  const float4 b = *reinterpret_cast<const float4*>(st + swz<G>(r, c * 4 + 16));
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
// 2 consecutive elements starting at (even) column c of row r.
template <class G>
NVFP4_DEV float2 lds2(const uint8_t* st, int r, int c, const uint16_t*) {
  const uint32_t w = *reinterpret_cast<const uint32_t*>(st + swz<G>(r, c * 2));
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
template <class G>
NVFP4_DEV float2 lds2(const uint8_t* st, int r, int c, const float*) {
  return *reinterpret_cast<const float2*>(st + swz<G>(r, c * 4));
}
// As lds2, both elements negated where m has bit 31 set (one XOR of the
// loaded word: the transform's sign of their row).
template <class G>
NVFP4_DEV float2 lds2s(const uint8_t* st, int r, int c, uint32_t m, const uint16_t*) {
  const uint32_t w = *reinterpret_cast<const uint32_t*>(st + swz<G>(r, c * 2)) ^ (m | (m >> 16));
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
template <class G>
NVFP4_DEV float2 lds2s(const uint8_t* st, int r, int c, uint32_t m, const float*) {
  const float2 f = *reinterpret_cast<const float2*>(st + swz<G>(r, c * 4));
  return make_float2(__uint_as_float(__float_as_uint(f.x) ^ m),
                     __uint_as_float(__float_as_uint(f.y) ^ m));
}

// ---- bounded waits -------------------------------------------------------------
NVFP4_DEV bool q_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag, unsigned code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  const uint64_t limit = *reinterpret_cast<volatile unsigned long long*>(&g_q_wait_ns);
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit) {
      *abort_flag = 1;
      atomicCAS(&g_quant_error, 0u, code);
      return false;
    }
  }
}
NVFP4_DEV void q_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kQWaitNs) {
      atomicCAS(&g_quant_error, 0u, 0x4Fu);
      return;
    }
  }
}

// ---- loads (amax pass) -----------------------------------------------------------
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

// ---- random Hadamard transform of a block split over a lane pair --------------
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
  return e4m3_rn_satfinite(__fmul_rn(div6_rn(a_b), s_enc));
}

// Element encode factor s_enc / S for every scale byte a block can get
// (block amaxes are non-negative, so bytes 0..127), 0 where S = 0: the same
// binary32 quotient the per-block formula gives, divided once per CTA.
constexpr int kEncTable = 128;
NVFP4_DEV void fill_enc_table(float* tab, float s_enc) {
  for (int i = threadIdx.x; i < kEncTable; i += blockDim.x) {
    const float S = e4m3_value((uint32_t)i);
    tab[i] = S == 0.0f ? 0.0f : __fdiv_rn(s_enc, S);
  }
  __syncthreads();
}
NVFP4_DEV float encode_factor(const float* tab, uint32_t sc) { return tab[sc & 127u]; }

// 8 elements -> 32 bits of packed codes (element 0 in the lowest nibble).
// SR takes each magnitude as |v| * enc (= |v * enc|: enc >= 0, and binary32
// rounding is symmetric) and the eight signs from v in one gather.
template <bool SR>
NVFP4_DEV uint32_t encode8(const float (&v)[8], float enc, uint4 w0, uint4 w1) {
  uint32_t out = 0;
  if (SR) {
    const uint32_t r[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i)  // disjoint nibbles
      out += e2m1_sr_mag(__float_as_uint(__fmul_rn(fabsf(v[i]), enc)), r[i]) * (1u << (4 * i));
    out |= sign_nibbles8(v);
  } else {
    float y[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) y[i] = __fmul_rn(v[i], enc);
#pragma unroll
    for (int i = 0; i < 4; ++i) out |= e2m1x2_rn(y[2 * i], y[2 * i + 1]) << (8 * i);
  }
  return out;
}

// ---- shared-memory layouts of the three quantise kernels --------------------------
constexpr int kColOutWords = 9;                             // 8 code words per output row + pad
constexpr uint32_t kColOutBytes = 128 * kColOutWords * 4;   // staged codes of one tile
constexpr uint32_t kColBuf = kColOutBytes + 512;            // + its scale atom
constexpr int kBlkKWords = 9;                               // 8 code words per row + pad
constexpr uint32_t kBlkWarpK = 16 * kBlkKWords * 4;         // K-major codes of a warp's 16 rows
constexpr uint32_t kBlkWarpBytes = kBlkWarpK + 512;         // + transposed codes, 64 x 8 bytes
template <typename T>
using RowL = QSmem<RowGeo<T>, kConsumerWarps * 64>;
template <typename T>
using ColL = QSmem<ColGeo<T>, 2 * kColBuf>;
template <typename T>
using BlkL = QSmem<BlkGeo<T>, kConsumerWarps * kBlkWarpBytes>;

// ---- pipeline pieces shared by the quantise kernels ----------------------------
// Barriers: full[s] (count 1, completed by the TMA bytes), empty[s] (one
// arrive per consumer warp), out[2] (one arrive per consumer warp; used by the
// transposing kernel to hand its staged tile to the storing warps).
template <class G, class L>
NVFP4_DEV void q_init(uint8_t* smem) {
  if (threadIdx.x == 0) {
    const uint32_t bar = smem_u32(smem + L::offBar);
    for (int s = 0; s < G::kStages; ++s) {
      mbar_init(bar + 8 * s, 1);
      mbar_init(bar + 8 * (G::kStages + s), kConsumerWarps);
    }
    mbar_init(bar + 8 * (2 * G::kStages), kConsumerWarps);
    mbar_init(bar + 8 * (2 * G::kStages + 1), kConsumerWarps);
    *reinterpret_cast<volatile int*>(smem + L::offMisc) = 0;
    fence_mbar_init();
  }
}

// Producer (one thread): the CTA's tiles in order, tile = blockIdx.x +
// k * gridDim.x into stage k % S.
template <class G>
NVFP4_DEV void q_produce(const CUtensorMap* tm, uint32_t stage0, uint32_t bar_full,
                         uint32_t bar_empty, volatile int* abort_flag, int64_t ntiles,
                         int64_t ntc) {
  prefetch_tmap(tm);
  uint32_t k = 0;
  if (*reinterpret_cast<volatile unsigned int*>(&g_q_stall)) return;  // injected: no loads
  TileWalk tw((int32_t)blockIdx.x, (int32_t)gridDim.x, (int32_t)ntc);
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++k, tw.next()) {
    const int s = (int)(k % G::kStages);
    if (!q_wait(bar_empty + 8 * s, (uint32_t)((k / G::kStages) & 1) ^ 1u, abort_flag, 0x40u))
      break;
    const int32_t x = (int32_t)(tw.tc * G::kTC), y = (int32_t)(tw.tr * G::kTR);
    mbar_arrive_expect_tx(bar_full + 8 * s, G::kStageBytes);
#pragma unroll
    for (int b = 0; b < G::kNBox; ++b)
      tma_load_2d(stage0 + s * G::kStageBytes + b * G::kBoxBytes, tm, bar_full + 8 * s,
                  x + b * G::kBoxCols, y);
  }
  // wait for the last copy issued into each stage: none is in flight at exit
  for (int s = 0; s < G::kStages && s < k; ++s) {
    const int64_t kl = s + G::kStages * ((k - 1 - s) / G::kStages);
    q_drain(bar_full + 8 * s, (uint32_t)((kl / G::kStages) & 1));
  }
}

// =============================================================================
// ROW_1X16: tile = 128 rows x 64 columns (one scale atom).  Consumer thread t
// owns the 8-element chunk (row t/8 + 32 i, columns 8 (t%8) ..) for i = 0..3;
// lanes t and t^1 form a 16-element block.  Warp w's rows are 4w..4w+3 (+32 i),
// which is exactly bytes 64w..64w+63 of the tile's scale atom, so each warp
// writes its codes and its slice of the atom without waiting for the others.
// =============================================================================
template <typename T, bool RHT, bool SR>
__global__ void __launch_bounds__(kQThreads, 2)
    quant_row_kernel(const __grid_constant__ CUtensorMap tm, const QParams p) {
  using G = RowGeo<T>;
  using L = RowL<T>;
  extern __shared__ uint8_t q_smem_raw[];
  uint8_t* smem = align_smem_1024(q_smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t bar_full = smem_u32(smem + L::offBar);
  const uint32_t bar_empty = bar_full + 8 * G::kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::offMisc);
  float* tab = reinterpret_cast<float*>(smem + L::offTab);
  q_init<G, L>(smem);
  griddep_wait();
  const float s_enc = tensor_s_enc(p, reinterpret_cast<float*>(smem + L::offRed));
  fill_enc_table(tab, s_enc);  // ends with a CTA barrier

  const int64_t R = p.rows, C = p.cols;
  const int64_t ntc = (C + G::kTC - 1) / G::kTC, ntiles = ((R + G::kTR - 1) / G::kTR) * ntc;
  if (warp == kConsumerWarps) {
    if (lane == 0) q_produce<G>(&tm, smem_u32(smem), bar_full, bar_empty, abort_flag, ntiles, ntc);
    return;
  }
  const int c8 = tid & 7, rsub = tid >> 3, half = c8 & 1;
  const int64_t apr = ((C / 16) + 3) / 4;
  const uint32_t sign_bits = RHT ? rht_sign_bits(p.seed) : 0u;
  uint8_t* wat = smem + L::offExtra + warp * 64;
  uint32_t k = 0;
  TileWalk tw((int32_t)blockIdx.x, (int32_t)gridDim.x, (int32_t)ntc);
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++k, tw.next()) {
    const int s = (int)(k % G::kStages);
    if (!q_wait(bar_full + 8 * s, (uint32_t)((k / G::kStages) & 1), abort_flag, 0x41u)) break;
    const uint8_t* st = smem + s * G::kStageBytes;
    float v[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      lds8<G>(st, rsub + 32 * i, c8 * 8, static_cast<const T*>(nullptr), v[i]);
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * s);

    const int64_t tr = tw.tr, tc = tw.tc;
    const int64_t c0 = tc * G::kTC + c8 * 8;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t r = tr * G::kTR + i * 32 + rsub;
      const bool ok = r < R && c0 < C;
      if (RHT) rht16_pair(v[i], sign_bits, half);
      float m = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(v[i][e]));
      m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
      const uint32_t sc = ok ? block_scale_code(m, s_enc) : 0u;
      const float enc = encode_factor(tab, sc);
      uint4 w0 = make_uint4(0, 0, 0, 0), w1 = w0;
      if (SR && ok) {
        const uint64_t idx = (uint64_t)(r * C + c0);
        w0 = sr_words(p.rk, p.offset, idx);
        w1 = sr_words(p.rk, p.offset, idx + 4);
      }
      const uint32_t packed = encode8<SR>(v[i], enc, w0, w1);
      if (ok) *reinterpret_cast<uint32_t*>(p.codes + r * (C / 2) + c0 / 2) = packed;
      if (half == 0) wat[(rsub & 3) * 16 + i * 4 + (c8 >> 1)] = (uint8_t)sc;
    }
    __syncwarp();
    if (lane < 4)
      reinterpret_cast<uint4*>(p.scales + (tr * apr + tc) * 512 + warp * 64)[lane] =
          reinterpret_cast<const uint4*>(wat)[lane];
    __syncwarp();
  }
}

// One output row (input column c0 + ol) of a COL_1X16 tile: 16 values of the
// 16-row block j (with RHT: already sign-flipped at the load) -> the
// transform, scale, codes, staged for the coalesced store.
template <bool RHT, bool SR>
NVFP4_DEV void col_block(float (&v)[16], int ol, int j, bool rows_ok, int64_t c0, int64_t r0,
                         int64_t R, int64_t C, float s_enc, const float* tab,
                         const PhiloxKeys& rk, uint64_t offset, uint32_t* out_s, uint8_t* atom) {
  const int64_t col = c0 + ol;
  const bool ok = rows_ok && col < C;
  if (RHT) rht16_signed_block(v);
  float m = 0.0f;
#pragma unroll
  for (int e = 0; e < 16; ++e) m = fmaxf(m, fabsf(v[e]));
  const uint32_t sc = ok ? block_scale_code(m, s_enc) : 0u;
  const float enc = encode_factor(tab, sc);
  uint4 w[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                make_uint4(0, 0, 0, 0)};
  if (SR && ok) {
    const uint64_t idx = (uint64_t)(col * R + r0 + 16 * j);
#pragma unroll
    for (int q = 0; q < 4; ++q) w[q] = sr_words(rk, offset, idx + 4 * q);
  }
  float lo[8], hi[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    lo[e] = v[e];
    hi[e] = v[8 + e];
  }
  out_s[ol * kColOutWords + 2 * j] = encode8<SR>(lo, enc, w[0], w[1]);
  out_s[ol * kColOutWords + 2 * j + 1] = encode8<SR>(hi, enc, w[2], w[3]);
  atom[(ol & 31) * 16 + ((ol >> 5) & 3) * 4 + j] = (uint8_t)sc;
}

// =============================================================================
// COL_1X16 (transposing): tile = 64 input rows x 128 input columns, i.e. an
// output tile of 128 rows x 64 columns -- one scale atom.  Consumer warp w,
// lane l owns the column pair 2 (l + 32 (w % 2)), +1 and the 16-row block
// w / 2: 16 conflict-free 4- or 8-byte reads of the stage, then per column the
// RHT butterfly, block amax, scale and codes from registers.  Codes and the
// atom are staged in shared memory (double-buffered) and, after every warp
// has arrived on the out barrier, written out as coalesced rows.
// =============================================================================
template <typename T, bool RHT, bool SR>
__global__ void __launch_bounds__(kQThreads, 2)
    quant_col_kernel(const __grid_constant__ CUtensorMap tm, const QParams p) {
  using G = ColGeo<T>;
  using L = ColL<T>;
  constexpr int kOutWords = kColOutWords;
  constexpr uint32_t kOutBytes = kColOutBytes, kBuf = kColBuf;
  extern __shared__ uint8_t q_smem_raw[];
  uint8_t* smem = align_smem_1024(q_smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t bar_full = smem_u32(smem + L::offBar);
  const uint32_t bar_empty = bar_full + 8 * G::kStages;
  const uint32_t bar_out = bar_full + 16 * G::kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::offMisc);
  float* tab = reinterpret_cast<float*>(smem + L::offTab);
  q_init<G, L>(smem);
  griddep_wait();
  const float s_enc = tensor_s_enc(p, reinterpret_cast<float*>(smem + L::offRed));
  fill_enc_table(tab, s_enc);

  const int64_t R = p.rows, C = p.cols;  // output is [C, R]
  const int64_t ntc = (C + G::kTC - 1) / G::kTC, ntiles = ((R + G::kTR - 1) / G::kTR) * ntc;
  if (warp == kConsumerWarps) {
    if (lane == 0) q_produce<G>(&tm, smem_u32(smem), bar_full, bar_empty, abort_flag, ntiles, ntc);
    return;
  }
  const int cp = lane + 32 * (warp & 1), j = warp >> 1;
  const int64_t apr = ((R / 16) + 3) / 4;
  uint32_t smask[16] = {};  // the transform's sign of block row e (bit 31)
  if (RHT) rht_sign_masks(rht_sign_bits(p.seed), smask);
  uint32_t k = 0;
  TileWalk tw((int32_t)blockIdx.x, (int32_t)gridDim.x, (int32_t)ntc);
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++k, tw.next()) {
    const int s = (int)(k % G::kStages);
    if (!q_wait(bar_full + 8 * s, (uint32_t)((k / G::kStages) & 1), abort_flag, 0x41u)) break;
    const uint8_t* st = smem + s * G::kStageBytes;
    float va[16], vb[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float2 f = lds2s<G>(st, 16 * j + e, 2 * cp, smask[e], static_cast<const T*>(nullptr));
      va[e] = f.x;
      vb[e] = f.y;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * s);

    const int64_t tr = tw.tr, tc = tw.tc;
    const int64_t r0 = tr * G::kTR, c0 = tc * G::kTC;
    const int buf = (int)(k & 1);
    uint32_t* out_s = reinterpret_cast<uint32_t*>(smem + L::offExtra + buf * kBuf);
    uint8_t* atom = smem + L::offExtra + buf * kBuf + kOutBytes;
    const bool rows_ok = r0 + 16 * j < R;
    col_block<RHT, SR>(va, 2 * cp, j, rows_ok, c0, r0, R, C, s_enc, tab, p.rk, p.offset,
                       out_s, atom);
    col_block<RHT, SR>(vb, 2 * cp + 1, j, rows_ok, c0, r0, R, C, s_enc, tab, p.rk, p.offset,
                       out_s, atom);
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_out + 8 * buf);
    if (!q_wait(bar_out + 8 * buf, (uint32_t)((k >> 1) & 1), abort_flag, 0x42u)) break;
    // warp w stores output rows 16w..16w+15: lane -> row 16w + lane/2, words 4 (lane%2) ..
    const int orl = 16 * warp + (lane >> 1), wq = (lane & 1) * 4;
    const int64_t orow = c0 + orl;
    if (orow < C) {
      uint8_t* dst = p.codes + orow * (R / 2) + r0 / 2 + wq * 4;
      const uint32_t* src = out_s + orl * kOutWords + wq;
      if (p.codes_vec16 && r0 + 8 * (wq + 4) <= R) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(src[0], src[1], src[2], src[3]);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (r0 + 8 * (wq + q) < R) reinterpret_cast<uint32_t*>(dst)[q] = src[q];
      }
    }
    if (warp == 0)
      reinterpret_cast<uint4*>(p.scales + (tc * apr + tr) * 512)[lane] =
          reinterpret_cast<const uint4*>(atom)[lane];
  }
}

// =============================================================================
// ROW_1X16 and COL_1X16 from one read (the two quantisations a training step
// makes of an activation or a gradient: the FPROP / DGRAD operand and the
// WGRAD operand), bf16 input, both tensor amaxes given.  Tile = 64 input rows
// x 128 input columns, read once from the stage by two sets of lanes:
//   column role (as quant_col_kernel): lane = column pair, warp pair = 16-row
//     block -> one output atom of the transposed operand, staged and stored
//     as coalesced rows after the out barrier;
//   row role: thread t owns input row t / 4 and the two 16-element blocks at
//     columns 32 (t % 4) .. + 31 -> 16 bytes of row codes and two scale bytes
//     (one 16-bit word of the row operand's scale atom), stored directly.
// The row operand's tiles are half an atom high; the tile that ends the last
// atom's first half also writes the zero scale rows of its second half.
// =============================================================================
struct QRowColParams {
  int64_t rows, cols;
  uint64_t seed, row_offset, col_offset;
  uint8_t* row_codes;
  uint8_t* row_scales;
  uint8_t* col_codes;
  uint8_t* col_scales;
  float* row_s_dec;
  float* col_s_dec;
  const float* row_amax;
  const float* col_amax;
  int row_codes_vec16;  // row codes 16-byte aligned rows (else 8)
  int col_codes_vec16;
  PhiloxKeys rk;
};
using RowColL = QSmem<ColGeo<uint16_t>, 2 * kColBuf + 512>;  // + the row operand's encode table

template <bool RHT, bool SRR, bool SRC>
__global__ void __launch_bounds__(kQThreads, 2)
    quant_rowcol_kernel(const __grid_constant__ CUtensorMap tm, const QRowColParams p) {
  using G = ColGeo<uint16_t>;
  using L = RowColL;
  constexpr int kOutWords = kColOutWords;
  constexpr uint32_t kOutBytes = kColOutBytes, kBuf = kColBuf;
  extern __shared__ uint8_t q_smem_raw[];
  uint8_t* smem = align_smem_1024(q_smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t bar_full = smem_u32(smem + L::offBar);
  const uint32_t bar_empty = bar_full + 8 * G::kStages;
  const uint32_t bar_out = bar_full + 16 * G::kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::offMisc);
  float* tab_c = reinterpret_cast<float*>(smem + L::offTab);
  float* tab_r = reinterpret_cast<float*>(smem + L::offExtra + 2 * kBuf);
  q_init<G, L>(smem);
  griddep_wait();
  const float s_enc_r = per_tensor_s_enc(*p.row_amax), s_enc_c = per_tensor_s_enc(*p.col_amax);
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *p.row_s_dec = __fdiv_rn(1.0f, s_enc_r);
    *p.col_s_dec = __fdiv_rn(1.0f, s_enc_c);
  }
  fill_enc_table(tab_r, s_enc_r);
  fill_enc_table(tab_c, s_enc_c);

  const int64_t R = p.rows, C = p.cols;
  const int64_t ntc = (C + G::kTC - 1) / G::kTC, ntr = (R + G::kTR - 1) / G::kTR;
  const int64_t ntiles = ntr * ntc;
  if (warp == kConsumerWarps) {
    if (lane == 0) q_produce<G>(&tm, smem_u32(smem), bar_full, bar_empty, abort_flag, ntiles, ntc);
    return;
  }
  const int cp = lane + 32 * (warp & 1), j = warp >> 1;  // column role
  const int rr = tid >> 2, bp = tid & 3;                   // row role
  const int64_t apr_c = ((R / 16) + 3) / 4;  // atoms per 128 rows of the column operand
  const int64_t pc4_r = ((C / 16) + 3) / 4 * 4;  // padded scale columns of the row operand
  uint32_t smask[16] = {};  // the transform's sign of block row e (bit 31)
  if (RHT) rht_sign_masks(rht_sign_bits(p.seed), smask);
  uint32_t k = 0;
  TileWalk tw((int32_t)blockIdx.x, (int32_t)gridDim.x, (int32_t)ntc);
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++k, tw.next()) {
    const int s = (int)(k % G::kStages);
    if (!q_wait(bar_full + 8 * s, (uint32_t)((k / G::kStages) & 1), abort_flag, 0x41u)) break;
    const uint8_t* st = smem + s * G::kStageBytes;
    float va[16], vb[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float2 f =
          lds2s<G>(st, 16 * j + e, 2 * cp, smask[e], static_cast<const uint16_t*>(nullptr));
      va[e] = f.x;
      vb[e] = f.y;
    }
    // RNE forms: the row role's 32 values, still packed, are read now and the
    // stage goes back to the producer before either role computes (the SR
    // forms, short of registers, read them after the column role)
    constexpr bool kEarly = !SRR && !SRC;
    uint4 rw[4];
    if constexpr (kEarly) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        rw[q] = *reinterpret_cast<const uint4*>(st + swz<G>(rr, (32 * bp + 8 * q) * 2));
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);
    }

    const int64_t tr = tw.tr, tc = tw.tc;
    const int64_t r0 = tr * G::kTR, c0 = tc * G::kTC;
    // ---- column operand: staged for the coalesced stores below
    const int buf = (int)(k & 1);
    uint32_t* out_s = reinterpret_cast<uint32_t*>(smem + L::offExtra + buf * kBuf);
    uint8_t* atom = smem + L::offExtra + buf * kBuf + kOutBytes;
    const bool rows_ok = r0 + 16 * j < R;
    col_block<RHT, SRC>(va, 2 * cp, j, rows_ok, c0, r0, R, C, s_enc_c, tab_c, p.rk, p.col_offset,
                        out_s, atom);
    col_block<RHT, SRC>(vb, 2 * cp + 1, j, rows_ok, c0, r0, R, C, s_enc_c, tab_c, p.rk,
                        p.col_offset, out_s, atom);
    // ---- row operand: row r, columns cb .. cb + 31 (two blocks)
    {
      float vr[4][8];
      if constexpr (kEarly) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t w[4] = {rw[q].x, rw[q].y, rw[q].z, rw[q].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            vr[q][2 * i] = __uint_as_float(w[i] << 16);
            vr[q][2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
          }
        }
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          lds8<G>(st, rr, 32 * bp + 8 * q, static_cast<const uint16_t*>(nullptr), vr[q]);
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + 8 * s);
      }
      const int64_t r = r0 + rr, cb = c0 + 32 * bp;
      const bool row_ok = r < R;
      uint32_t words[4], scw = 0;
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        const bool ok = row_ok && cb + 16 * b < C;
        float m = 0.0f;
#pragma unroll
        for (int e = 0; e < 8; ++e) m = fmaxf(m, fmaxf(fabsf(vr[2 * b][e]), fabsf(vr[2 * b + 1][e])));
        const uint32_t sc = ok ? block_scale_code(m, s_enc_r) : 0u;
        const float enc = encode_factor(tab_r, sc);
        uint4 w0 = make_uint4(0, 0, 0, 0), w1 = w0, w2 = w0, w3 = w0;
        if (SRR && ok) {
          const uint64_t idx = (uint64_t)(r * C + cb + 16 * b);
          w0 = sr_words(p.rk, p.row_offset, idx);
          w1 = sr_words(p.rk, p.row_offset, idx + 4);
          w2 = sr_words(p.rk, p.row_offset, idx + 8);
          w3 = sr_words(p.rk, p.row_offset, idx + 12);
        }
        words[2 * b] = encode8<SRR>(vr[2 * b], enc, w0, w1);
        words[2 * b + 1] = encode8<SRR>(vr[2 * b + 1], enc, w2, w3);
        scw |= sc << (8 * b);
      }
      if (row_ok && cb < C) {
        uint8_t* dst = p.row_codes + r * (C / 2) + cb / 2;
        if (cb + 32 <= C && p.row_codes_vec16) {
          *reinterpret_cast<uint4*>(dst) = make_uint4(words[0], words[1], words[2], words[3]);
        } else {
          *reinterpret_cast<uint2*>(dst) = make_uint2(words[0], words[1]);
          if (cb + 16 < C) *reinterpret_cast<uint2*>(dst + 8) = make_uint2(words[2], words[3]);
        }
      }
      // scale bytes of scale columns cb/16, cb/16 + 1 (within one 4-byte group:
      // cb/16 is even); columns past C are zero padding
      if (cb / 16 < pc4_r)
        *reinterpret_cast<uint16_t*>(p.row_scales + sf_offset(r, cb / 16, pc4_r)) = (uint16_t)scw;
      // the second half of the last atom's rows, if no tile covers it: zeros
      if (tr == ntr - 1 && (r0 & 127) == 0 && cb / 16 < pc4_r)
        *reinterpret_cast<uint16_t*>(p.row_scales + sf_offset(r + 64, cb / 16, pc4_r)) = 0;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_out + 8 * buf);
    if (!q_wait(bar_out + 8 * buf, (uint32_t)((k >> 1) & 1), abort_flag, 0x42u)) break;
    // column operand rows 16 w .. 16 w + 15: lane -> row 16 w + lane / 2, words 4 (lane % 2) ..
    const int orl = 16 * warp + (lane >> 1), wq = (lane & 1) * 4;
    const int64_t orow = c0 + orl;
    if (orow < C) {
      uint8_t* dst = p.col_codes + orow * (R / 2) + r0 / 2 + wq * 4;
      const uint32_t* src = out_s + orl * kOutWords + wq;
      if (p.col_codes_vec16 && r0 + 8 * (wq + 4) <= R) {
        *reinterpret_cast<uint4*>(dst) = make_uint4(src[0], src[1], src[2], src[3]);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (r0 + 8 * (wq + q) < R) reinterpret_cast<uint32_t*>(dst)[q] = src[q];
      }
    }
    if (warp == 0)
      reinterpret_cast<uint4*>(p.col_scales + (tc * apr_c + tr) * 512)[lane] =
          reinterpret_cast<const uint4*>(atom)[lane];
  }
}

// =============================================================================
// BLOCK_16X16 (weights): tile = 128 rows x 64 columns = 8 x 4 scale tiles.
// Consumer warp w owns rows 16w..16w+15; lane -> (row lane % 16, half lane /
// 16), 8 elements of each of the 4 16x16 tiles, whose amax is one warp
// reduction.  Writes the K-major codes and, with EMIT_T, the nibble-transposed
// codes built from the same codes (the partner row's codes arrive by one
// shuffle), plus both scale layouts.  Every output of warp w comes from its
// own 16 rows, so warps never wait for each other.
// =============================================================================
template <typename T, bool SR, bool EMIT_T>
__global__ void __launch_bounds__(kQThreads, 2)
    quant_16x16_kernel(const __grid_constant__ CUtensorMap tm, const QParams p) {
  using G = BlkGeo<T>;
  using L = BlkL<T>;
  constexpr int kKWords = kBlkKWords;
  constexpr uint32_t kWarpK = kBlkWarpK, kWarpBytes = kBlkWarpBytes;
  extern __shared__ uint8_t q_smem_raw[];
  uint8_t* smem = align_smem_1024(q_smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t bar_full = smem_u32(smem + L::offBar);
  const uint32_t bar_empty = bar_full + 8 * G::kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::offMisc);
  float* tab = reinterpret_cast<float*>(smem + L::offTab);
  q_init<G, L>(smem);
  griddep_wait();
  const float s_enc = tensor_s_enc(p, reinterpret_cast<float*>(smem + L::offRed));
  fill_enc_table(tab, s_enc);

  const int64_t R = p.rows, C = p.cols;
  const int64_t ntc = (C + G::kTC - 1) / G::kTC, ntiles = ((R + G::kTR - 1) / G::kTR) * ntc;
  if (warp == kConsumerWarps) {
    if (lane == 0) q_produce<G>(&tm, smem_u32(smem), bar_full, bar_empty, abort_flag, ntiles, ntc);
    return;
  }
  const int rl16 = lane & 15, h = lane >> 4;
  const int rl = 16 * warp + rl16;
  const int64_t apr_k = ((C / 16) + 3) / 4;  // atoms per 128-row block, K-major view
  const int64_t apr_t = ((R / 16) + 3) / 4;  // transposed view
  uint32_t* ok_s = reinterpret_cast<uint32_t*>(smem + L::offExtra + warp * kWarpBytes);
  uint8_t* ot_s = smem + L::offExtra + warp * kWarpBytes + kWarpK;
  uint32_t k = 0;
  TileWalk tw((int32_t)blockIdx.x, (int32_t)gridDim.x, (int32_t)ntc);
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++k, tw.next()) {
    const int s = (int)(k % G::kStages);
    if (!q_wait(bar_full + 8 * s, (uint32_t)((k / G::kStages) & 1), abort_flag, 0x41u)) break;
    const uint8_t* st = smem + s * G::kStageBytes;
    float v[4][8];
#pragma unroll
    for (int b = 0; b < 4; ++b)
      lds8<G>(st, rl, 16 * b + 8 * h, static_cast<const T*>(nullptr), v[b]);
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + 8 * s);

    const int64_t tr = tw.tr, tc = tw.tc;
    const int64_t r0 = tr * G::kTR, c0 = tc * G::kTC;
    const int64_t r = r0 + rl;
    const bool row_ok = r0 + 16 * warp < R;  // rows come in whole 16-row strips
    const int64_t g = tr * 8 + warp;         // 16-row block: scale column of the transposed view
    // the four 16x16 blocks side by side, one step at a time, so that their
    // warp reductions, table reads and shuffles are in flight together
    uint32_t scw = 0, sc[4], packed[4];
    float mb[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      float m = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(v[b][e]));
      mb[b] = m;
    }
    // each block's maximum in one warp reduction: non-negative floats order
    // like their bit patterns read as unsigned integers
#pragma unroll
    for (int b = 0; b < 4; ++b)
      mb[b] = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(mb[b])));
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const bool ok = row_ok && (c0 + 16 * b < C);
      sc[b] = ok ? block_scale_code(mb[b], s_enc) : 0u;
      const float enc = encode_factor(tab, sc[b]);
      uint4 w0 = make_uint4(0, 0, 0, 0), w1 = w0;
      if (SR && ok) {
        const uint64_t idx = (uint64_t)(r * C + c0 + 16 * b + 8 * h);
        w0 = sr_words(p.rk, p.offset, idx);
        w1 = sr_words(p.rk, p.offset, idx + 4);
      }
      packed[b] = encode8<SR>(v[b], enc, w0, w1);
      ok_s[rl16 * kKWords + 2 * b + h] = packed[b];
      scw |= sc[b] << (8 * b);
    }
    if (EMIT_T) {
      uint32_t others[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) others[b] = __shfl_xor_sync(0xFFFFFFFFu, packed[b], 1);
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        // transposed byte of column e = code(even row, e) | code(odd row, e) << 4:
        // t holds columns 0, 2, 4, 6 and u columns 1, 3, 5, 7 of the lane
        // pair's 8 columns; the even lane stores columns 0-3, the odd 4-7
        const uint32_t other = others[b];  // row rl ^ 1
        const uint32_t lo = (lane & 1) ? other : packed[b], hi = (lane & 1) ? packed[b] : other;
        const uint32_t t = (lo & 0x0F0F0F0Fu) | ((hi & 0x0F0F0F0Fu) << 4);
        const uint32_t u = ((lo >> 4) & 0x0F0F0F0Fu) | (hi & 0xF0F0F0F0u);
        const uint32_t w = (lane & 1) ? __byte_perm(t, u, 0x7362) : __byte_perm(t, u, 0x5140);
        const int cb = 16 * b + 8 * h + 4 * (lane & 1);
#pragma unroll
        for (int k = 0; k < 4; ++k) ot_s[(cb + k) * 8 + (rl16 >> 1)] = (uint8_t)(w >> (8 * k));
        // transposed scale of output row c0 + 16 b + lane, scale column g
        if (lane < 16 && g < 4 * apr_t) {
          const int64_t orow = c0 + 16 * b + lane;
          p.scales_t[((orow >> 7) * apr_t + (g >> 2)) * 512 + (orow & 31) * 16 +
                     ((orow >> 5) & 3) * 4 + (g & 3)] = (uint8_t)sc[b];
        }
      }
    }
    // K-major scales: the 4 bytes of row rl form one word of the tile's atom
    if (h == 0)
      *reinterpret_cast<uint32_t*>(p.scales + (tr * apr_k + tc) * 512 + (rl & 31) * 16 +
                                   ((rl >> 5) & 3) * 4) = scw;
    // the transposed view's scale rows past the last 64-column tile, up to the
    // 128-row padding, belong to no tile: the CTA of that last tile zeroes them
    if (EMIT_T && (tc & 1) == 0 && tc == ntc - 1 && g < 4 * apr_t) {
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int64_t orow = c0 + 64 + lane + 32 * q;
        p.scales_t[((orow >> 7) * apr_t + (g >> 2)) * 512 + (orow & 31) * 16 +
                   ((orow >> 5) & 3) * 4 + (g & 3)] = 0;
      }
    }
    __syncwarp();
    {  // K-major codes: lane -> row 16 w + lane / 2, 16 bytes (32 columns) lane % 2
      const int rr = lane >> 1, hh = lane & 1;
      const int64_t row = r0 + 16 * warp + rr, col = c0 + 32 * hh;
      if (row < R && col < C) {
        uint8_t* dst = p.codes + row * (C / 2) + col / 2;
        const uint32_t* src = ok_s + rr * kKWords + 4 * hh;
        if (p.codes_vec16 && col + 32 <= C) {
          *reinterpret_cast<uint4*>(dst) = make_uint4(src[0], src[1], src[2], src[3]);
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (col + 8 * q < C) reinterpret_cast<uint32_t*>(dst)[q] = src[q];
        }
      }
    }
    if (EMIT_T && row_ok) {  // transposed codes: output rows c0 + lane (+32), 8 bytes each
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int c = lane + 32 * q;
        if (c0 + c < C) {
          uint8_t* dst = p.codes_t + (c0 + c) * (R / 2) + (r0 + 16 * warp) / 2;
          const uint2 val = *reinterpret_cast<const uint2*>(ot_s + c * 8);
          if (p.codes_t_vec8) {
            *reinterpret_cast<uint2*>(dst) = val;
          } else {
            reinterpret_cast<uint32_t*>(dst)[0] = val.x;
            reinterpret_cast<uint32_t*>(dst)[1] = val.y;
          }
        }
      }
    }
    __syncwarp();
  }
}

// =============================================================================
// Amax pre-pass: per-CTA partial maxima of |x| (or of |RHT(x)| along the
// dimension the quantiser transforms), written to the workspace.
// =============================================================================
// max |x|: 8-element chunks, eight 16-byte loads in flight per thread (the
// pass is bound by how many bytes each SM keeps in flight).
template <typename T>
__global__ void __launch_bounds__(kAmaxThreads) amax_plain_kernel(const QParams p) {
  constexpr int kU = 8;
  __shared__ float red[kAmaxThreads / 32];
  griddep_wait();
  const T* x = static_cast<const T*>(p.x);
  const int64_t C = p.cols, ld = p.ld, cpr = C / 8, n = p.rows * cpr;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  float m = 0.0f;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += kU * stride) {
    // all loads issued before any value is used: indices past the end are
    // clamped to the last chunk (a valid address) and their values dropped
    float v[kU][8];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t q = min(i + u * stride, n - 1);
      const int64_t r = ld == C ? 0 : q / cpr;
      const int64_t off = ld == C ? q * 8 : r * ld + (q - r * cpr) * 8;
      load8(x + off, v[u]);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (i + u * stride < n) {
#pragma unroll
        for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(v[u][e]));
      }
  }
  m = block_max(m, red);
  if (threadIdx.x == 0) p.partials[blockIdx.x] = m;
}

// max |RHT(x)| with the transform along columns (16-row blocks, the WGRAD
// operand quantised by COL_1X16): an item is one 16-row block of one
// 16-byte column chunk, sixteen 16-byte loads in flight per thread.  With
// PLAIN it also takes max |x| of the same values (every element, as rows are
// whole 16-row blocks), written to the upper half of the partials.
template <typename T, bool PLAIN>
__global__ void __launch_bounds__(kAmaxThreads) amax_rht_col_kernel(const QParams p) {
  __shared__ float red[kAmaxThreads / 32];
  float mp = 0.0f;
  constexpr int kCh = 16 / (int)sizeof(T);  // columns per 16-byte chunk
  const T* x = static_cast<const T*>(p.x);
  const int64_t ld = p.ld, cpr = p.cols / kCh, n = (p.rows / 16) * cpr;
  const uint32_t sign_bits = rht_sign_bits(p.seed);
  griddep_wait();
  float m = 0.0f;
  for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < n;
       q += (int64_t)gridDim.x * blockDim.x) {
    const int64_t jb = q / cpr, cc = q - jb * cpr;
    const T* base = x + jb * 16 * ld + cc * kCh;
    uint4 u[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      // row e of the block, negated where the transform's sign bit e is set
      const uint32_t me =
          ((sign_bits >> e) & 1u) ? (sizeof(T) == 2 ? 0x80008000u : 0x80000000u) : 0u;
      u[e] = __ldg(reinterpret_cast<const uint4*>(base + e * ld));
      u[e].x ^= me;
      u[e].y ^= me;
      u[e].z ^= me;
      u[e].w ^= me;
    }
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      if (sizeof(T) == 2) {
        float a[16], b[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const uint32_t w = wi == 0 ? u[e].x : wi == 1 ? u[e].y : wi == 2 ? u[e].z : u[e].w;
          a[e] = __uint_as_float(w << 16);
          b[e] = __uint_as_float(w & 0xFFFF0000u);
          if (PLAIN) mp = fmaxf(mp, fmaxf(fabsf(a[e]), fabsf(b[e])));
        }
        m = fmaxf(m, fmaxf(rht16_absmax_signed(a), rht16_absmax_signed(b)));
      } else {
        float a[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          a[e] = __uint_as_float(wi == 0 ? u[e].x : wi == 1 ? u[e].y : wi == 2 ? u[e].z : u[e].w);
          if (PLAIN) mp = fmaxf(mp, fabsf(a[e]));
        }
        m = fmaxf(m, rht16_absmax_signed(a));
      }
    }
  }
  m = block_max(__fmul_rn(m, 0.25f), red);  // the transform's x 1/4, on the maximum
  if (threadIdx.x == 0) p.partials[blockIdx.x] = m;
  if (PLAIN) {
    mp = block_max(mp, red);
    if (threadIdx.x == 0) p.partials[kMaxPartials / 2 + blockIdx.x] = mp;
  }
}

// Final reduction of an nvfp4_amax call: partials [0, n) to *out0 and, when
// out1 is set, partials [kMaxPartials / 2, + n) to *out1.
__global__ void __launch_bounds__(kAmaxThreads) amax_finalize_kernel(const float* partials,
                                                                     int n, float* out0,
                                                                     float* out1) {
  __shared__ float red[kAmaxThreads / 32];
  griddep_wait();
  float m0 = 0.0f, m1 = 0.0f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    m0 = fmaxf(m0, partials[i]);
    if (out1) m1 = fmaxf(m1, partials[kMaxPartials / 2 + i]);
  }
  m0 = block_max(m0, red);
  if (threadIdx.x == 0) *out0 = m0;
  if (out1) {
    m1 = block_max(m1, red);
    if (threadIdx.x == 0) *out1 = m1;
  }
}

// max |RHT(x)| with the transform along rows (ROW_1X16 with RHT): an item is
// one 16-element block of a row.
template <typename T>
__global__ void __launch_bounds__(kAmaxThreads) amax_rht_row_kernel(const QParams p) {
  __shared__ float red[kAmaxThreads / 32];
  const T* x = static_cast<const T*>(p.x);
  const int64_t bpr = p.cols / 16, n = p.rows * bpr;
  const uint32_t sign_bits = rht_sign_bits(p.seed);
  griddep_wait();
  float m = 0.0f;
  for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < n;
       q += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = q / bpr, b = q - r * bpr;
    const T* base = x + r * p.ld + b * 16;
    float lo[8], hi[8], v[16];
    load8(base, lo);
    load8(base + 8, hi);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      v[e] = lo[e];
      v[8 + e] = hi[e];
    }
    m = fmaxf(m, rht16_absmax_unscaled(v, sign_bits));
  }
  m = block_max(__fmul_rn(m, 0.25f), red);  // the transform's x 1/4, on the maximum
  if (threadIdx.x == 0) p.partials[blockIdx.x] = m;
}

// ---- host dispatch -------------------------------------------------------------
// Per-device launch state of one kernel: dynamic shared memory opted in and
// the number of CTAs that fit on an SM.
struct LaunchState {
  std::mutex mu;
  int per_sm[64] = {};
};

template <typename K>
int resident_per_sm(LaunchState& ls, K kern, int threads, uint32_t smem) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(ls.mu);
  if (ls.per_sm[dev] == 0) {
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
      return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem) != cudaSuccess)
      return 0;
    ls.per_sm[dev] = n;
  }
  return ls.per_sm[dev];
}

template <auto KERN, class L>
nvfp4_status launch_q(const CUtensorMap& tm, const QParams& p, int64_t ntiles, int sms,
                      cudaStream_t s) {
  static LaunchState ls;
  if (ntiles > (int64_t(1) << 30)) return NVFP4_ERR_SHAPE;  // the kernels' 32-bit tile walk
  const int per_sm = resident_per_sm(ls, KERN, kQThreads, L::kAlloc);
  if (per_sm <= 0) return NVFP4_ERR_CUDA;
  const int grid = (int)std::min<int64_t>(ntiles, (int64_t)sms * per_sm);
  return launch_pdl(KERN, grid, kQThreads, L::kAlloc, s, tm, p) == cudaSuccess ? NVFP4_OK
                                                                       : NVFP4_ERR_CUDA;
}

template <auto KERN>
nvfp4_status launch_amax_kernel(const QParams& p, int grid, cudaStream_t s) {
  return launch_pdl(KERN, grid, kAmaxThreads, 0, s, p) == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA;
}

// Grid of an amax kernel: as many CTAs as are resident at once, at most 4 per
// SM (the partial-maxima slots a workspace holds) and at most one per 256
// work items.
template <auto KERN>
int amax_grid(int sms, int64_t items) {
  static LaunchState ls;
  const int per_sm = std::min(4, std::max(1, resident_per_sm(ls, KERN, kAmaxThreads, 0)));
  const int64_t want = std::max<int64_t>(1, (items + kAmaxThreads - 1) / kAmaxThreads);
  return (int)std::min<int64_t>(std::min<int64_t>(want, (int64_t)sms * per_sm), kMaxPartials);
}

// Amax pre-pass for one quantiser call: returns the CTA count in *grid.
template <typename T>
nvfp4_status launch_amax(QParams& p, int mode, int sms, cudaStream_t s) {
  const bool rht = p.flags & NVFP4_RHT;
  int grid;
  if (mode == NVFP4_COL_1X16 && rht) {
    grid = amax_grid<amax_rht_col_kernel<T, false>>(
        sms, (p.rows / 16) * (p.cols * (int64_t)sizeof(T) / 16));
    p.num_partials = grid;
    return launch_amax_kernel<amax_rht_col_kernel<T, false>>(p, grid, s);
  }
  if (mode == NVFP4_ROW_1X16 && rht) {
    grid = amax_grid<amax_rht_row_kernel<T>>(sms, p.rows * (p.cols / 16));
    p.num_partials = grid;
    return launch_amax_kernel<amax_rht_row_kernel<T>>(p, grid, s);
  }
  grid = amax_grid<amax_plain_kernel<T>>(sms, p.rows * (p.cols / 8) / 4);
  p.num_partials = grid;
  return launch_amax_kernel<amax_plain_kernel<T>>(p, grid, s);
}

// 2-D tensor map over the input [rows, cols] (leading dimension ld): boxes of
// box_rows x 128 bytes, 128-byte swizzle, zeros outside the tensor.
template <typename T>
bool make_input_map(CUtensorMap* map, const void* x, int64_t rows, int64_t cols, int64_t ld,
                    int box_rows) {
  EncodeTiledFn enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(ld * (int64_t)sizeof(T))};
  const cuuint32_t box[2] = {(cuuint32_t)(128 / sizeof(T)), (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map,
             sizeof(T) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
             2, const_cast<void*>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename T>
nvfp4_status launch_quant(const QParams& p, int mode, int sms, cudaStream_t s) {
  const bool rht = p.flags & NVFP4_RHT, sr = p.flags & NVFP4_SR, et = p.flags & NVFP4_EMIT_T;
  const int64_t R = p.rows, C = p.cols;
  CUtensorMap tm;
  if (mode == NVFP4_ROW_1X16) {
    using G = RowGeo<T>;
    if (!make_input_map<T>(&tm, p.x, R, C, p.ld, G::kTR)) return NVFP4_ERR_CUDA;
    const int64_t nt = ((R + G::kTR - 1) / G::kTR) * ((C + G::kTC - 1) / G::kTC);
    if (rht && sr) return launch_q<quant_row_kernel<T, true, true>, RowL<T>>(tm, p, nt, sms, s);
    if (rht) return launch_q<quant_row_kernel<T, true, false>, RowL<T>>(tm, p, nt, sms, s);
    if (sr) return launch_q<quant_row_kernel<T, false, true>, RowL<T>>(tm, p, nt, sms, s);
    return launch_q<quant_row_kernel<T, false, false>, RowL<T>>(tm, p, nt, sms, s);
  }
  if (mode == NVFP4_COL_1X16) {
    using G = ColGeo<T>;
    if (!make_input_map<T>(&tm, p.x, R, C, p.ld, G::kTR)) return NVFP4_ERR_CUDA;
    const int64_t nt = ((R + G::kTR - 1) / G::kTR) * ((C + G::kTC - 1) / G::kTC);
    if (rht && sr) return launch_q<quant_col_kernel<T, true, true>, ColL<T>>(tm, p, nt, sms, s);
    if (rht) return launch_q<quant_col_kernel<T, true, false>, ColL<T>>(tm, p, nt, sms, s);
    if (sr) return launch_q<quant_col_kernel<T, false, true>, ColL<T>>(tm, p, nt, sms, s);
    return launch_q<quant_col_kernel<T, false, false>, ColL<T>>(tm, p, nt, sms, s);
  }
  using G = BlkGeo<T>;
  if (!make_input_map<T>(&tm, p.x, R, C, p.ld, G::kTR)) return NVFP4_ERR_CUDA;
  const int64_t nt = ((R + G::kTR - 1) / G::kTR) * ((C + G::kTC - 1) / G::kTC);
  if (sr && et) return launch_q<quant_16x16_kernel<T, true, true>, BlkL<T>>(tm, p, nt, sms, s);
  if (sr) return launch_q<quant_16x16_kernel<T, true, false>, BlkL<T>>(tm, p, nt, sms, s);
  if (et) return launch_q<quant_16x16_kernel<T, false, true>, BlkL<T>>(tm, p, nt, sms, s);
  return launch_q<quant_16x16_kernel<T, false, false>, BlkL<T>>(tm, p, nt, sms, s);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <auto KERN>
nvfp4_status launch_rowcol(const CUtensorMap& tm, const QRowColParams& p, int64_t ntiles, int sms,
                           cudaStream_t s) {
  static LaunchState ls;
  if (ntiles > (int64_t(1) << 30)) return NVFP4_ERR_SHAPE;  // the kernels' 32-bit tile walk
  const int per_sm = resident_per_sm(ls, KERN, kQThreads, RowColL::kAlloc);
  if (per_sm <= 0) return NVFP4_ERR_CUDA;
  const int grid = (int)std::min<int64_t>(ntiles, (int64_t)sms * per_sm);
  return launch_pdl(KERN, grid, kQThreads, RowColL::kAlloc, s, tm, p) == cudaSuccess
             ? NVFP4_OK
             : NVFP4_ERR_CUDA;
}

}  // namespace

nvfp4_status quantize_rowcol_impl(const void* x, int32_t in_dtype, int64_t rows, int64_t cols,
                                  int64_t ld, uint32_t row_flags, uint32_t col_flags,
                                  uint64_t seed, uint64_t row_offset, uint64_t col_offset,
                                  nvfp4_tensor* row_out, nvfp4_tensor* col_out,
                                  cudaStream_t stream) {
  if (!x || !row_out || !col_out) return NVFP4_ERR_INVALID_ARG;
  for (const nvfp4_tensor* t : {row_out, col_out})
    if (!t->codes || !t->scales || !t->amax || !t->s_dec) return NVFP4_ERR_INVALID_ARG;
  if (in_dtype != NVFP4_IN_BF16) return NVFP4_ERR_INVALID_ARG;
  if ((row_flags & ~(uint32_t)(NVFP4_SR | NVFP4_AMAX_GIVEN)) ||
      (col_flags & ~(uint32_t)(NVFP4_SR | NVFP4_RHT | NVFP4_AMAX_GIVEN)) ||
      !(row_flags & NVFP4_AMAX_GIVEN) || !(col_flags & NVFP4_AMAX_GIVEN))
    return NVFP4_ERR_INVALID_ARG;
  if (rows <= 0 || cols <= 0 || ld < cols || rows % 16 || cols % 16) return NVFP4_ERR_SHAPE;
  if (rows > INT32_MAX || cols > INT32_MAX) return NVFP4_ERR_SHAPE;
  if (!aligned16(x) || (ld * 2) % 16) return NVFP4_ERR_ALIGN;
  for (const nvfp4_tensor* t : {row_out, col_out})
    if (!aligned16(t->codes) || !aligned16(t->scales) ||
        (reinterpret_cast<uintptr_t>(t->amax) & 3u) || (reinterpret_cast<uintptr_t>(t->s_dec) & 3u))
      return NVFP4_ERR_ALIGN;
  DeviceInfo dev;
  nvfp4_status st = current_device(&dev);
  if (st != NVFP4_OK) return st;

  QRowColParams p;
  p.rows = rows;
  p.cols = cols;
  p.seed = seed;
  p.row_offset = row_offset;
  p.col_offset = col_offset;
  p.row_codes = static_cast<uint8_t*>(row_out->codes);
  p.row_scales = static_cast<uint8_t*>(row_out->scales);
  p.col_codes = static_cast<uint8_t*>(col_out->codes);
  p.col_scales = static_cast<uint8_t*>(col_out->scales);
  p.row_s_dec = row_out->s_dec;
  p.col_s_dec = col_out->s_dec;
  p.row_amax = row_out->amax;
  p.col_amax = col_out->amax;
  p.row_codes_vec16 = (cols / 2) % 16 == 0;
  p.col_codes_vec16 = (rows / 2) % 16 == 0;
  p.rk = philox_round_keys(seed);
  using G = ColGeo<uint16_t>;
  CUtensorMap tm;
  if (!make_input_map<uint16_t>(&tm, x, rows, cols, ld, G::kTR)) return NVFP4_ERR_CUDA;
  const int64_t nt = ((rows + G::kTR - 1) / G::kTR) * ((cols + G::kTC - 1) / G::kTC);
  const bool rht = col_flags & NVFP4_RHT, srr = row_flags & NVFP4_SR, src = col_flags & NVFP4_SR;
  const int sms = dev.sm_count;
  if (rht) {
    if (srr && src) st = launch_rowcol<quant_rowcol_kernel<true, true, true>>(tm, p, nt, sms, stream);
    else if (srr) st = launch_rowcol<quant_rowcol_kernel<true, true, false>>(tm, p, nt, sms, stream);
    else if (src) st = launch_rowcol<quant_rowcol_kernel<true, false, true>>(tm, p, nt, sms, stream);
    else st = launch_rowcol<quant_rowcol_kernel<true, false, false>>(tm, p, nt, sms, stream);
  } else {
    if (srr && src) st = launch_rowcol<quant_rowcol_kernel<false, true, true>>(tm, p, nt, sms, stream);
    else if (srr) st = launch_rowcol<quant_rowcol_kernel<false, true, false>>(tm, p, nt, sms, stream);
    else if (src) st = launch_rowcol<quant_rowcol_kernel<false, false, true>>(tm, p, nt, sms, stream);
    else st = launch_rowcol<quant_rowcol_kernel<false, false, false>>(tm, p, nt, sms, stream);
  }
  if (st != NVFP4_OK) return st;
  row_out->rows = rows;
  row_out->cols = cols;
  row_out->mode = NVFP4_ROW_1X16;
  row_out->flags = row_flags;
  col_out->rows = cols;
  col_out->cols = rows;
  col_out->mode = NVFP4_COL_1X16;
  col_out->flags = col_flags;
  return NVFP4_OK;
}

// One read of x for the amax of its row-wise and column-wise (RHT) quantisations.
nvfp4_status amax_impl(const void* x, int32_t in_dtype, int64_t rows, int64_t cols, int64_t ld,
                       uint64_t seed, float* amax_plain, float* amax_rht, void* workspace,
                       size_t workspace_bytes, cudaStream_t stream) {
  if (!x || (!amax_plain && !amax_rht)) return NVFP4_ERR_INVALID_ARG;
  if (in_dtype != NVFP4_IN_BF16 && in_dtype != NVFP4_IN_FP32) return NVFP4_ERR_INVALID_ARG;
  if (rows <= 0 || cols <= 0 || ld < cols || cols % 8) return NVFP4_ERR_SHAPE;
  if (amax_rht && rows % 16) return NVFP4_ERR_SHAPE;
  const int64_t esz = in_dtype == NVFP4_IN_BF16 ? 2 : 4;
  if (!aligned16(x) || (ld * esz) % 16) return NVFP4_ERR_ALIGN;
  if ((reinterpret_cast<uintptr_t>(amax_plain) & 3u) || (reinterpret_cast<uintptr_t>(amax_rht) & 3u))
    return NVFP4_ERR_ALIGN;
  if (!workspace || workspace_bytes < kQuantWorkspaceBytes || !aligned16(workspace))
    return NVFP4_ERR_WORKSPACE;
  DeviceInfo dev;
  nvfp4_status st = current_device(&dev);
  if (st != NVFP4_OK) return st;

  QParams p{};
  p.x = x;
  p.rows = rows;
  p.cols = cols;
  p.ld = ld;
  p.seed = seed;
  p.partials = static_cast<float*>(workspace);
  const bool bf = in_dtype == NVFP4_IN_BF16;
  int grid = 0;
  if (!amax_rht) {  // max |x| alone
    grid = bf ? amax_grid<amax_plain_kernel<uint16_t>>(dev.sm_count, rows * (cols / 8) / 4)
              : amax_grid<amax_plain_kernel<float>>(dev.sm_count, rows * (cols / 8) / 4);
    st = bf ? launch_amax_kernel<amax_plain_kernel<uint16_t>>(p, grid, stream)
            : launch_amax_kernel<amax_plain_kernel<float>>(p, grid, stream);
  } else {  // the RHT amax, with max |x| from the same loads when asked for
    const int64_t items = (rows / 16) * (cols * esz / 16);
    if (amax_plain) {
      grid = bf ? amax_grid<amax_rht_col_kernel<uint16_t, true>>(dev.sm_count, items)
                : amax_grid<amax_rht_col_kernel<float, true>>(dev.sm_count, items);
      grid = std::min(grid, kMaxPartials / 2);
      st = bf ? launch_amax_kernel<amax_rht_col_kernel<uint16_t, true>>(p, grid, stream)
              : launch_amax_kernel<amax_rht_col_kernel<float, true>>(p, grid, stream);
    } else {
      grid = bf ? amax_grid<amax_rht_col_kernel<uint16_t, false>>(dev.sm_count, items)
                : amax_grid<amax_rht_col_kernel<float, false>>(dev.sm_count, items);
      st = bf ? launch_amax_kernel<amax_rht_col_kernel<uint16_t, false>>(p, grid, stream)
              : launch_amax_kernel<amax_rht_col_kernel<float, false>>(p, grid, stream);
    }
  }
  if (st != NVFP4_OK) return st;
  float* out0 = amax_rht ? amax_rht : amax_plain;
  float* out1 = amax_rht ? amax_plain : nullptr;
  return launch_pdl(amax_finalize_kernel, 1, kAmaxThreads, 0, stream,
                    static_cast<const float*>(p.partials), grid, out0, out1) == cudaSuccess
             ? NVFP4_OK
             : NVFP4_ERR_CUDA;
}

nvfp4_status quant_set_injection(unsigned int stall, unsigned long long wait_ns) {
  if (cudaMemcpyToSymbol(g_q_stall, &stall, sizeof(stall)) != cudaSuccess ||
      cudaMemcpyToSymbol(g_q_wait_ns, &wait_ns, sizeof(wait_ns)) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  return NVFP4_OK;
}

nvfp4_status quant_read_error(unsigned int* code) {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_quant_error, sizeof(v)) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (v && cudaMemcpyToSymbol(g_quant_error, &zero, sizeof(zero)) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  *code = v;
  return NVFP4_OK;
}

// ---- entry point that allocates nothing ---------------------------------------
// Some callers cannot hand the library a workspace: code that runs while a
// CUDA graph is being captured (where cudaMalloc is not permitted), plugins
// that receive only input and output pointers from a host framework, or
// applications whose allocator owns all device memory.  For them the amax
// partial maxima live in a fixed array inside the library instead.
namespace {

constexpr int kNoAllocPartials = kMaxPartials;  // 1024 floats: 4 KB per device
// every amax grid is capped at kMaxPartials CTAs, one partial each
static_assert(kNoAllocPartials >= kMaxPartials, "the array holds every partial maximum");
// Lives on every device that loads the library, until the process exits.
// In host code this name is only a stand-in: kernels receive the device
// address obtained with cudaGetSymbolAddress below.
static __device__ __align__(256) float g_noalloc_partials[kNoAllocPartials];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[64] = {};

// Device address of the array on the current device.  Outside stream capture
// it is looked up on every call (cudaDeviceReset reloads the module, and the
// array may then sit at another address); during capture the address found
// by the last call outside capture on this device is used, so the first call
// on a device must come before any capture.
nvfp4_status noalloc_scratch(cudaStream_t stream, void** addr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return NVFP4_ERR_CUDA;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return NVFP4_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (cap == cudaStreamCaptureStatusNone || !g_noalloc_addr[dev]) {
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
  void* scratch = nullptr;
  st = noalloc_scratch(static_cast<cudaStream_t>(stream), &scratch);
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

  if (rows > INT32_MAX || cols > INT32_MAX) return NVFP4_ERR_SHAPE;  // TMA coordinates

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
  p.rk = philox_round_keys(seed);
  p.codes = static_cast<uint8_t*>(out->codes);
  p.scales = static_cast<uint8_t*>(out->scales);
  p.codes_t = static_cast<uint8_t*>(out->codes_t);
  p.scales_t = static_cast<uint8_t*>(out->scales_t);
  p.amax_out = out->amax;
  p.s_dec_out = out->s_dec;
  p.amax_in = out->amax;
  p.partials = static_cast<float*>(workspace);
  p.num_partials = 0;
  // 16-byte code stores need 16-byte aligned rows of codes
  const int64_t code_row_bytes = mode == NVFP4_COL_1X16 ? rows / 2 : cols / 2;
  p.codes_vec16 = aligned16(out->codes) && code_row_bytes % 16 == 0;
  p.codes_t_vec8 = (flags & NVFP4_EMIT_T) && (reinterpret_cast<uintptr_t>(out->codes_t) & 7u) == 0;

  if (!given) {
    st = in_dtype == NVFP4_IN_BF16 ? launch_amax<uint16_t>(p, mode, dev.sm_count, stream)
                                   : launch_amax<float>(p, mode, dev.sm_count, stream);
    if (st != NVFP4_OK) return st;
  }
  st = in_dtype == NVFP4_IN_BF16 ? launch_quant<uint16_t>(p, mode, dev.sm_count, stream)
                                 : launch_quant<float>(p, mode, dev.sm_count, stream);
  if (st != NVFP4_OK) return st;

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
