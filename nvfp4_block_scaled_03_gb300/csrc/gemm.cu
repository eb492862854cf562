// gemm.cu -- NVFP4 block-scaled GEMM for sm_103a: D = alpha * A . B^T with
// A [M, K], B [N, K] E2M1 K-major and one UE4M3 scale per 16 elements
// ("NVFP4 pretraining recipe" page: FPROP, DGRAD and WGRAD consume NVFP4
// inputs and emit BF16 outputs, Figure 1 text).
//
// Design (one CTA per SM, persistent over output tiles of 128 x BN):
//   warp 0      TMA producer: A/B code tiles (cp.async.bulk.tensor, 128-byte
//               swizzle) and the scale atoms (cp.async.bulk, already in the
//               MMA layout) into a STAGES-deep shared-memory ring;
//   warp 1      allocates tensor memory; one thread copies each stage's scale
//               atoms to tensor memory (tcgen05.cp) and issues
//               tcgen05.mma.kind::mxf4nvf4.block_scale (K = 64 per
//               instruction, 4 per stage), then tcgen05.commit frees the
//               stage and, after the last K block, signals the accumulator;
//   warps 2..9  epilogue: tcgen05.ld of the FP32 accumulator (each warp one
//               32-lane quarter and half of the columns) into registers,
//               release of the accumulator to the MMA warp, then x alpha
//               (= s_dec(A) * s_dec(B) read on the device), BF16 rounding
//               and global stores while the next tile's MMAs run.
// Every mbarrier wait is bounded (2 s); on expiry the kernel records a code
// in the device error word, the other roles stop at their next wait, copies
// and MMAs in flight are drained (again bounded) and tensor memory is freed.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace nvfp4 {

static __device__ unsigned int g_gemm_error;
// Failure injection for tests of the bounded waits (nvfp4_debug_inject):
// while g_gemm_stall is set the producers of every GEMM kernel issue no
// loads, and the pipeline waits give up after g_gemm_wait_ns.
static __device__ unsigned int g_gemm_stall;
static __device__ unsigned long long g_gemm_wait_ns = 2000000000ull;

namespace {

constexpr uint64_t kWaitTimeoutNs = 2000000000ull;
constexpr int kThreads = 320;      // producer, MMA, 8 epilogue warps
constexpr int kBM = 128;            // rows of A per tile (one MMA, cta_group::1)
constexpr int kBKBytes = 128;       // K bytes per stage (256 FP4 elements)
constexpr uint32_t kTmemCols = 512;

struct GemmArgs {
  const uint8_t* sfa;
  const uint8_t* sfb;
  const float* sdec_a;
  const float* sdec_b;
  void* D;
  const void* C;
  int M, N, K;
  int kg;         // scale atoms per 128-row block along K (= K / 64)
  int num_m_blk;  // ceil(M / 128)
  int num_n_blk;  // ceil(N / BN)
  int nrb_b;      // 128-row blocks of B's scale tensor (ceil(N / 128))
  int nrb_a;      // 128-row blocks of A's scale tensor (ceil(M / 128))
};

template <int BN, int STAGES, int BKB>
struct Smem {
  static constexpr int kAtoms = BKB / 32;                        // scale atoms per 128 rows per stage
  static constexpr uint32_t kA = kBM * BKB;                      // 16/8 KB
  static constexpr uint32_t kB = BN * BKB;
  static constexpr uint32_t kSFA = kAtoms * 512;
  static constexpr uint32_t kSFB = (BN / 128) * kAtoms * 512;
  static constexpr uint32_t offA = 0;
  static constexpr uint32_t offB = offA + STAGES * kA;
  static constexpr uint32_t offSFA = offB + STAGES * kB;
  static constexpr uint32_t offSFB = offSFA + STAGES * kSFA;
  static constexpr uint32_t offBar = offSFB + STAGES * kSFB;
  static constexpr uint32_t kNumBars = 2 * STAGES + 3;  // full, empty, acc_full, acc_empty, drain
  static constexpr uint32_t offMisc = offBar + kNumBars * 8;
  static constexpr uint32_t kBytes = offMisc + 16;
  static constexpr uint32_t kAlloc = kBytes + 1024;  // room to align the base to 1024
  // tensor memory columns: accumulator [0, BN), then per-stage scales
  static constexpr uint32_t kSfCol0 = BN;
  static constexpr uint32_t kSfColsPerStage = (16 + BN / 8) * kAtoms / 4;
  static_assert(kSfCol0 + STAGES * kSfColsPerStage <= kTmemCols, "tensor memory overflow");
  static_assert(kAlloc <= 232448, "shared memory overflow");
};

// K-major operand descriptor for a stage row width of BKB bytes (128-byte or
// 64-byte swizzle; 8-row swizzle atoms stacked 8*BKB bytes apart).
template <int BKB>
NVFP4_DEV uint64_t smem_desc_kmajor(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)((8 * BKB) >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(BKB == 128 ? 2 : 4) << 61;  // SWIZZLE_128B or SWIZZLE_64B
  return d;
}


// Drain wait used after an abort: bounded, ignores the abort flag.
NVFP4_DEV void wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
      atomicCAS(&g_gemm_error, 0u, 0xDEu);
      return;
    }
  }
}

// Bounded wait of the single-SM kernel: on expiry it raises the CTA's abort
// flag and records `code` in the error word.
NVFP4_DEV bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                            unsigned int code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  const uint64_t limit = *reinterpret_cast<volatile unsigned long long*>(&g_gemm_wait_ns);
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit) {
      *abort_flag = 1;
      atomicCAS(&g_gemm_error, 0u, code);
      return false;
    }
  }
}

NVFP4_DEV uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

template <int DMODE>
NVFP4_DEV void store_row_chunk(const GemmArgs& a, int64_t row, int64_t col0, const uint32_t (&r)[32],
                               float alpha) {
  if (DMODE == NVFP4_D_BF16 || DMODE == NVFP4_D_BF16_ADD_C) {
    __nv_bfloat16* D = static_cast<__nv_bfloat16*>(a.D) + row * a.N + col0;
    const __nv_bfloat16* Cp = static_cast<const __nv_bfloat16*>(a.C) + row * a.N + col0;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      if (col0 + g * 8 >= a.N) break;
      float f[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = __fmul_rn(__uint_as_float(r[g * 8 + e]), alpha);
      if (DMODE == NVFP4_D_BF16_ADD_C) {
        const uint4 c = *reinterpret_cast<const uint4*>(Cp + g * 8);
        const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          f[2 * e] = __fadd_rn(f[2 * e], __uint_as_float(cw[e] << 16));
          f[2 * e + 1] = __fadd_rn(f[2 * e + 1], __uint_as_float(cw[e] & 0xFFFF0000u));
        }
      }
      uint4 o;
      o.x = pack_bf16x2(f[0], f[1]);
      o.y = pack_bf16x2(f[2], f[3]);
      o.z = pack_bf16x2(f[4], f[5]);
      o.w = pack_bf16x2(f[6], f[7]);
      *reinterpret_cast<uint4*>(D + g * 8) = o;
    }
  } else {  // NVFP4_D_F32_ACCUM: D += float(bf16(alpha * acc))
    // the loads of four 16-byte pieces before their stores: the stores may
    // alias later loads as far as the compiler knows, so interleaving them
    // one by one would serialise eight memory round trips per chunk
    float* D = static_cast<float*>(a.D) + row * a.N + col0;
#pragma unroll
    for (int g0 = 0; g0 < 8; g0 += 4) {
      float4 d[4];
#pragma unroll
      for (int g = 0; g < 4; ++g)
        if (col0 + (g0 + g) * 4 < a.N) d[g] = *reinterpret_cast<const float4*>(D + (g0 + g) * 4);
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        if (col0 + (g0 + g) * 4 >= a.N) break;
        float t[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          t[e] = __bfloat162float(
              __float2bfloat16_rn(__fmul_rn(__uint_as_float(r[(g0 + g) * 4 + e]), alpha)));
        d[g].x = __fadd_rn(d[g].x, t[0]);
        d[g].y = __fadd_rn(d[g].y, t[1]);
        d[g].z = __fadd_rn(d[g].z, t[2]);
        d[g].w = __fadd_rn(d[g].w, t[3]);
        *reinterpret_cast<float4*>(D + (g0 + g) * 4) = d[g];
      }
    }
  }
}

// Pulls the part of D that a row of a later tile's epilogue reads (128-byte
// lines from col0 on, `bytes` of them) into L2 while the tile's MMAs run.
NVFP4_DEV void prefetch_l2_row(const void* p, int bytes) {
  const char* c = static_cast<const char*>(p);
  for (int o = 0; o < bytes; o += 128)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(c + o)));
}

// Epilogue helper: one warp's 32 rows x 32 bf16 columns (lane = row, 16
// packed pairs) into its staging box, then one tensor store at (x, y).  The
// box is rewritten only after the previous store has read it; the 16-byte
// pieces are rotated so a warp's writes hit distinct banks.
NVFP4_DEV void store_box_bf16(uint8_t* box, int lane, const uint32_t (&pk)[16],
                              const CUtensorMap* tmD, int32_t x, int32_t y) {
  if (lane == 0) bulk_wait_group_read<0>();
  __syncwarp();
#pragma unroll
  for (int pc = 0; pc < 4; ++pc) {
    const int piece = (pc + (lane >> 1)) & 3;
    uint4 v;
    switch (piece) {
      case 0: v = make_uint4(pk[0], pk[1], pk[2], pk[3]); break;
      case 1: v = make_uint4(pk[4], pk[5], pk[6], pk[7]); break;
      case 2: v = make_uint4(pk[8], pk[9], pk[10], pk[11]); break;
      default: v = make_uint4(pk[12], pk[13], pk[14], pk[15]); break;
    }
    *reinterpret_cast<uint4*>(box + lane * 64 + piece * 16) = v;
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tmD, smem_u32(box), x, y);
    bulk_commit_group();
  }
}

// The FP32 fold from 32 bf16 results already rounded and packed in pairs:
// D[row, col0 + i] += float(bf16 result i), the same single FP32 add as
// store_row_chunk's F32_ACCUM branch.
NVFP4_DEV void fold_row_chunk_packed(const GemmArgs& a, int64_t row, int64_t col0,
                                     const uint32_t (&pk)[16]) {
  float* D = static_cast<float*>(a.D) + row * a.N + col0;
#pragma unroll
  for (int g0 = 0; g0 < 8; g0 += 4) {
    float4 d[4];
#pragma unroll
    for (int g = 0; g < 4; ++g)
      if (col0 + (g0 + g) * 4 < a.N) d[g] = *reinterpret_cast<const float4*>(D + (g0 + g) * 4);
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      if (col0 + (g0 + g) * 4 >= a.N) break;
      const uint32_t p0 = pk[(g0 + g) * 2], p1 = pk[(g0 + g) * 2 + 1];
      d[g].x = __fadd_rn(d[g].x, __uint_as_float(p0 << 16));
      d[g].y = __fadd_rn(d[g].y, __uint_as_float(p0 & 0xFFFF0000u));
      d[g].z = __fadd_rn(d[g].z, __uint_as_float(p1 << 16));
      d[g].w = __fadd_rn(d[g].w, __uint_as_float(p1 & 0xFFFF0000u));
      *reinterpret_cast<float4*>(D + (g0 + g) * 4) = d[g];
    }
  }
}

template <int BN, int STAGES, int DMODE, int BKB>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_nvf4_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, const GemmArgs args) {
  using L = Smem<BN, STAGES, BKB>;
  constexpr int kAt = L::kAtoms;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::offBar;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  const uint32_t acc_full = bar0 + 8u * (2 * STAGES);
  const uint32_t acc_empty = acc_full + 8;
  const uint32_t drain_bar = acc_full + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::offMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::offMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_kb = (args.K + 2 * BKB - 1) / (2 * BKB);
  const int num_mu = args.num_m_blk;
  const int num_units = num_mu * args.num_n_blk;
  const int unit0 = blockIdx.x, unit_step = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 8);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      uint32_t s = 0, ph = 0;
      int armed[STAGES];
      for (int i = 0; i < STAGES; ++i) armed[i] = -1;
      // injected stall: no loads, so the MMA thread's first wait runs out
      bool ok = *reinterpret_cast<volatile unsigned int*>(&g_gemm_stall) == 0u;
      for (int unit = unit0; ok && unit < num_units; unit += unit_step) {
        const int m_blk = unit % num_mu, n_blk = unit / num_mu;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_bounded(empty_bar(s), ph ^ 1u, abort_flag, 0x10u)) {
            ok = false;
            break;
          }
          const int natoms = min(kAt, args.kg - kb * kAt);
          int nb_valid = 0;
          for (int j = 0; j < BN / 128; ++j) nb_valid += (n_blk * (BN / 128) + j) < args.nrb_b;
          const uint32_t sf_bytes = (uint32_t)natoms * 512u * (1u + (uint32_t)nb_valid);
          mbar_arrive_expect_tx(full_bar(s), L::kA + L::kB + sf_bytes);
          armed[s] = (int)ph;
          tma_load_2d(sbase + L::offA + s * L::kA, &tmA, full_bar(s), kb * BKB, m_blk * kBM);
          tma_load_2d(sbase + L::offB + s * L::kB, &tmB, full_bar(s), kb * BKB, n_blk * BN);
          bulk_load(sbase + L::offSFA + s * L::kSFA,
                    args.sfa + ((int64_t)m_blk * args.kg + kb * kAt) * 512,
                    natoms * 512u, full_bar(s));
          for (int j = 0; j < BN / 128; ++j) {
            const int rb = n_blk * (BN / 128) + j;
            if (rb < args.nrb_b)
              bulk_load(sbase + L::offSFB + s * L::kSFB + j * (kAt * 512),
                        args.sfb + ((int64_t)rb * args.kg + kb * kAt) * 512,
                        natoms * 512u, full_bar(s));
          }
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok) {  // let the copies already issued land before the CTA exits
        for (int i = 0; i < STAGES; ++i)
          if (armed[i] >= 0) wait_drain(full_bar(i), (uint32_t)armed[i]);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA
      constexpr uint32_t idesc = idesc_nvf4(kBM, BN);
      uint32_t s = 0, ph = 0, acc_ph = 0;
      bool ok = true, issued = false;
      for (int unit = unit0; ok && unit < num_units; unit += unit_step) {
        if (!wait_bounded(acc_empty, acc_ph ^ 1u, abort_flag, 0x20u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_bounded(full_bar(s), ph, abort_flag, 0x21u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int natoms = min(kAt, args.kg - kb * kAt);
          const uint32_t sfa_t = tmem + L::kSfCol0 + s * L::kSfColsPerStage;
          const uint32_t sfb_t = sfa_t + 16;
          const uint32_t sa = sbase + L::offSFA + s * L::kSFA;
          const uint32_t sb = sbase + L::offSFB + s * L::kSFB;
          const uint32_t a0 = sbase + L::offA + s * L::kA;
          const uint32_t b0 = sbase + L::offB + s * L::kB;
          // per K step: its scale atoms to tensor memory, then its MMA, so the
          // copies of step j+1 proceed while the MMA of step j runs
          for (int j = 0; j < natoms; ++j) {
            tc_cp_32x128b_warpx4(sfa_t + 4 * j, smem_desc_sf(sa + j * 512));
#pragma unroll
            for (int b = 0; b < BN / 128; ++b)
              tc_cp_32x128b_warpx4(sfb_t + j * (BN / 32) + 4 * b,
                                   smem_desc_sf(sb + b * (kAt * 512) + j * 512));
            tc_mma_nvf4(tmem, smem_desc_kmajor<BKB>(a0 + 32 * j), smem_desc_kmajor<BKB>(b0 + 32 * j), idesc,
                        sfa_t + 4 * j, sfb_t + j * (BN / 32), (kb | j) != 0 ? 1u : 0u);
          }
          issued = true;
          tc_commit(empty_bar(s));
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        tc_commit(acc_full);
        acc_ph ^= 1u;
      }
      if (!ok && issued) {  // MMAs in flight must finish before tensor memory is freed
        tc_commit(drain_bar);
        wait_drain(drain_bar, 0);
      }
    }
  } else {
    // -------------------------------------------------------------- epilogue
    // Warp w reads lane quarter w % 4 of tensor memory and one half of the
    // tile's columns.  It drains its part of the accumulator into registers,
    // releases the accumulator to the MMA warp, then scales and stores.
    constexpr int kCols = BN / 2, kChunks = kCols / 32;
    const int q = warp & 3, h = (warp - 2) >> 2;
    const float alpha = __fmul_rn(__ldg(args.sdec_a), __ldg(args.sdec_b));
    uint32_t acc_ph = 0;
    for (int unit = unit0; unit < num_units; unit += unit_step) {
      const int m_blk = unit % num_mu, n_blk = unit / num_mu;
      if (!wait_bounded(acc_full, acc_ph, abort_flag, 0x30u)) break;
      tc_fence_after();
      uint32_t r[kChunks][32];
#pragma unroll
      for (int c = 0; c < kChunks; ++c)
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * kCols + c * 32), r[c]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
      acc_ph ^= 1u;
      const int64_t row = (int64_t)m_blk * kBM + q * 32 + lane;
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        const int64_t col0 = (int64_t)n_blk * BN + h * kCols + c * 32;
        if (row < args.M && col0 < args.N) store_row_chunk<DMODE>(args, row, col0, r[c], alpha);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// =============================================================================
// CTA-pair kernel: output tiles of 256 x 256 computed by a cluster of two
// CTAs with tcgen05 cta_group::2.  CTA r loads A rows [128 r, 128 r + 128)
// and B rows [128 r, 128 r + 128) of the tile, the scale atoms of its A rows
// and all scale atoms of the tile's B rows (each CTA's MMA reads all of B's
// scales from its own tensor memory).  The A and B loads complete on the
// leader's (rank 0) full barrier.  Per SM this moves two thirds of the
// operand bytes of the single-CTA 128 x 256 tile.
//
// The block scales reach tensor memory in one of two ways.  NVFP4 (stored
// scales): each CTA's scale atoms land on its own barrier, and four scale
// warps per CTA -- one per 32-lane quarter -- read them from shared memory
// and write them into their quarter with tcgen05.st, in the replicated
// layout the block-scaled MMA reads; each waits for its stores
// (tcgen05.wait::st), fences (tcgen05.fence::before_thread_sync) and arrives
// on the leader's scales-ready barrier.  A scale copy (tcgen05.cp) runs in
// the tensor pipe in order with the MMAs, at about 44 bytes of tensor memory
// a cycle, so a stage's 24 KB of replicated scales took longer than its four
// MMAs; the stores take a few tens of cycles beside them.  The MX formats
// (copied scales): two copy warps issue the stage's tcgen05.cp copies into
// both CTAs' tensor memory, B's scales as 4x-replicated images, and arrive
// on the same barrier.  The MMA thread waits for the stage's data and its
// scales, fences (tcgen05.fence::after_thread_sync) and issues only the MMAs
// and the commit that frees the stage.  A tensor-memory scale slot is
// rewritten only after its stage was refilled, i.e. after the MMAs that read
// it completed.  Each CTA's epilogue drains its 128 accumulator rows and
// releases them on the leader's barrier.  5 stages of 38 KB (NVFP4).
// =============================================================================
constexpr int kPairBN = 256;

constexpr int kPairCopyWarps = 2;

// Operand formats of the pair kernel.  Every format stages 128 bytes of K per
// row and issues four MMAs of 32 bytes of K per stage; the scale atoms (128
// rows x 4 scale bytes, 512 bytes) cover 64 K elements for NVFP4 (one per
// 16) and 128 for the MX formats (one per 32).
enum { kFmtNVF4 = 0, kFmtMXF4 = 1, kFmtMXF8 = 2 };
template <int FMT>
struct PairFmt {
  static constexpr int kAtoms = FMT == kFmtNVF4 ? 4 : (FMT == kFmtMXF4 ? 2 : 1);  // per stage
  static constexpr int kStageK = FMT == kFmtMXF8 ? 128 : 256;  // K elements per stage
  static constexpr int kMmaPerAtom = 4 / kAtoms;
};

// Warp roles of a pair CTA.  With the scales copied (IMG, the MX formats):
// 12 warps -- producer, MMA, two copy warps, eight epilogue warps.  With the
// scales stored (ST, NVFP4): 16 warps in four warpgroups -- warpgroup 0 the
// producer, the MMA warp and two idle warps; warpgroup 1 four scale warps,
// one per 32-lane quarter; warpgroups 2-3 the epilogue.  With 16 warps a
// sub-partition holds four, so each starts at 128 registers; warpgroups 0-1
// hand registers to the epilogue (setmaxnreg).
template <bool ST>
struct PairRoles {
  static constexpr int kEpi0 = ST ? 8 : 2 + kPairCopyWarps;  // first of 8 epilogue warps
  static constexpr int kThreads = (kEpi0 + 8) * 32;
  static constexpr int kRegsIssue = 96, kRegsEpilogue = 160;  // ST only
  static constexpr int kSplitRegs = 2 * 128 * kRegsIssue + 2 * 128 * kRegsEpilogue;
  static_assert(!ST || kSplitRegs <= kThreads * 128, "register split exceeds the launch's");
};

// Instruction descriptor of the MX block-scaled MMAs: element format code for
// A and B (E2M1 = 1 in the FP4 kinds, E4M3 = 0 in kind::mxf8f6f4), N / 8,
// scale type UE8M0 (bit 23), M / 16; the scale factor IDs (bits 4-5 for B,
// 29-30 for A: the first byte of each row's scale word the MMA reads) are
// ORed in per MMA.
__host__ __device__ constexpr uint32_t idesc_mx(int M, int N, uint32_t fmt) {
  return (fmt << 7) | (fmt << 10) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
         ((uint32_t)(M >> 4) << 24);
}

// The pair MMA of a format: NVFP4 (16-element blocks, UE4M3 scales), MXFP4
// (32-element blocks: two UE8M0 scales per 64-deep MMA), MXFP8 (E4M3
// elements, one UE8M0 scale per 32-deep MMA).
template <int FMT>
NVFP4_DEV void tc_mma_pair_bs(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                              uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  if constexpr (FMT == kFmtNVF4) {
    tc_mma_pair_nvf4(d_tmem, adesc, bdesc, idesc, sfa_tmem, sfb_tmem, accumulate);
  } else if constexpr (FMT == kFmtMXF4) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::2X"
        " [%0], %1, %2, %3, [%5], [%6], p;\n}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
  } else {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X"
        " [%0], %1, %2, %3, [%5], [%6], p;\n}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
        : "memory");
  }
}

template <int STAGES, int FMT, bool IMG>
struct PairSmem {
  // NVFP4 stores its scales into tensor memory from the scale warps; the MX
  // formats copy them (IMG: B's scales as images)
  static_assert(IMG == (FMT != kFmtNVF4), "scale path of the format");
  static constexpr bool kST = !IMG;  // scales through tcgen05.st
  static constexpr int kAt = PairFmt<FMT>::kAtoms;
  static constexpr uint32_t kA = 128 * kBKBytes;               // this CTA's 128 A rows
  static constexpr uint32_t kB = 128 * kBKBytes;               // this CTA's 128 B rows
  // B's scales either as the plain atoms of the tile's two 128-row blocks
  // (stored), or as 4 KB images, one per scale atom along K (the two row
  // halves' atoms, each repeated for the four 32-lane quarters), that one
  // 128-lane x 256-bit copy each moves into tensor memory
  static constexpr uint32_t kSFA = kAt * 512;                  // own A rows' scale atoms
  static constexpr uint32_t kSFB = IMG ? kAt * 4096 : kAt * 1024;
  // bytes counted on the leader's full barrier: both CTAs' A and B, and with
  // the scales copied also their scale atoms (stored scales land on each
  // CTA's own scale barrier)
  static constexpr uint32_t kStageTx = 2 * (kA + kB) + (kST ? 0 : 2 * (kSFA + kSFB));
  static constexpr uint32_t offA = 0;
  static constexpr uint32_t offB = offA + STAGES * kA;
  static constexpr uint32_t offSFA = offB + STAGES * kB;
  static constexpr uint32_t offSFB = offSFA + STAGES * kSFA;
  static constexpr uint32_t offBar = offSFB + STAGES * kSFB;
  // full, empty, scales-ready, scales-landed (ST) per stage; acc full, acc
  // empty; drains (MMA warp, copy warps)
  static constexpr uint32_t kNumBars = 4 * STAGES + 3 + kPairCopyWarps;
  static constexpr uint32_t offMisc = offBar + kNumBars * 8;
  // bf16 output staging for tensor stores: one box of 32 rows x 64 bytes per
  // epilogue warp
  static constexpr uint32_t kStoreBox = 32 * 64;
  static constexpr uint32_t offStore = (offMisc + 16 + 127) / 128 * 128;
  static constexpr uint32_t kBytes = offStore + 8 * kStoreBox;
  static constexpr uint32_t kAlloc = kBytes + 1024;
  static constexpr uint32_t kSfCol0 = kPairBN;
  static constexpr uint32_t kSfColsPerStage = kAt * (4 + 8);  // A (4 per atom), B (8 per atom)
  static_assert(kSfCol0 + STAGES * kSfColsPerStage <= kTmemCols, "tensor memory overflow");
  static_assert(kAlloc <= 232448, "shared memory overflow");
};

// Bounded wait for the pair: a timeout also raises the peer CTA's abort flag.
NVFP4_DEV bool wait_bounded_pair(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                 uint32_t peer_abort_addr, unsigned int code) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  const uint64_t limit = *reinterpret_cast<volatile unsigned long long*>(&g_gemm_wait_ns);
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit) {
      *abort_flag = 1;
      st_cluster_u32(peer_abort_addr, 1u);
      atomicCAS(&g_gemm_error, 0u, code);
      return false;
    }
  }
}

template <int STAGES, int DMODE, int FMT, bool IMG>
__global__ void __cluster_dims__(2, 1, 1)
__launch_bounds__(PairRoles<!IMG>::kThreads, 1)
    gemm_nvf4_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                          const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmSFA,
                          const __grid_constant__ CUtensorMap tmSFB,
                          const __grid_constant__ CUtensorMap tmD, const GemmArgs args) {
  using L = PairSmem<STAGES, FMT, IMG>;
  constexpr bool ST = L::kST;
  using R = PairRoles<ST>;
  constexpr int kAt = PairFmt<FMT>::kAtoms;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::offBar;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto sf_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };
  auto scf_bar = [&](int s) { return bar0 + 8u * (3 * STAGES + s); };  // ST: this CTA's scales
  const uint32_t acc_full = bar0 + 8u * (4 * STAGES);
  const uint32_t acc_empty = acc_full + 8;
  const uint32_t drain_bar = acc_full + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::offMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::offMisc + 4);

  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const uint32_t peer_abort = mapa_shared(smem_u32(smem + L::offMisc + 4), rank ^ 1u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_kb = (args.K + PairFmt<FMT>::kStageK - 1) / PairFmt<FMT>::kStageK;
  const int num_tiles = args.num_m_blk * args.num_n_blk;  // 256 x 256 tiles
  const int pair = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
      mbar_init(sf_bar(s), ST ? 8 : kPairCopyWarps);  // ST: four scale warps per CTA
      mbar_init(scf_bar(s), 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, 16);  // 8 epilogue warps in each CTA of the pair
    for (int d = 0; d <= kPairCopyWarps; ++d) mbar_init(drain_bar + 8u * d, 1);  // MMA, copy warps
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();

  if (warp < R::kEpi0) {
  // issue warps (the register hint sits inside the branch so that the code it
  // governs is known to the register allocator)
  if constexpr (ST) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R::kRegsIssue));
  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      prefetch_tmap(&tmSFA);
      prefetch_tmap(&tmSFB);
      uint32_t s = 0, ph = 0;
      // injected stall: no loads, so every consumer's first wait runs out
      bool ok = *reinterpret_cast<volatile unsigned int*>(&g_gemm_stall) == 0u;
      for (int tile = pair; ok && tile < num_tiles; tile += num_pairs) {
        const int m_blk = tile % args.num_m_blk, n_blk = tile / args.num_m_blk;
        const int a_rb = m_blk * 2 + (int)rank;  // this CTA's 128-row block of A
        const int b_rb0 = n_blk * 2;             // the tile's first 128-row block of B
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_bounded_pair(empty_bar(s), ph ^ 1u, abort_flag, peer_abort, 0x11u)) {
            ok = false;
            break;
          }
          const uint32_t fb = mapa_shared(full_bar(s), 0);
          if (leader) mbar_arrive_expect_tx(full_bar(s), L::kStageTx);
          tma_load_2d_pair(sbase + L::offA + s * L::kA, &tmA, fb, kb * kBKBytes, a_rb * 128);
          tma_load_2d_pair(sbase + L::offB + s * L::kB, &tmB, fb, kb * kBKBytes,
                           (b_rb0 + (int)rank) * 128);
          if (ST) {
            // this CTA's scale atoms (its A rows' and the tile's B rows', 128-byte
            // rows, 4 per atom) on its own barrier, for its scale warps
            mbar_arrive_expect_tx(scf_bar(s), L::kSFA + L::kSFB);
            tma_load_2d(sbase + L::offSFA + s * L::kSFA, &tmSFA, scf_bar(s), 0,
                        (a_rb * args.kg + kb * kAt) * 4);
            tma_load_2d(sbase + L::offSFB + s * L::kSFB, &tmSFB, scf_bar(s), 0,
                        (b_rb0 * args.kg + kb * kAt) * 4);
            tma_load_2d(sbase + L::offSFB + s * L::kSFB + kAt * 512, &tmSFB, scf_bar(s), 0,
                        ((b_rb0 + 1) * args.kg + kb * kAt) * 4);
            if (++s == STAGES) { s = 0; ph ^= 1u; }
            continue;
          }
          // A's scale atoms as 128-byte rows (4 per atom), B's as images
          tma_load_2d_pair(sbase + L::offSFA + s * L::kSFA, &tmSFA, fb, 0,
                           (a_rb * args.kg + kb * kAt) * 4);
          tma_load_5d_pair(sbase + L::offSFB + s * L::kSFB, &tmSFB, fb, b_rb0, kb * kAt);
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok) {  // give copies already issued time to land before exit
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
      }
    }
  } else if (ST && warp >= 4) {
    // ------------------------------------------------------------ scale warps
    // Warp q (= warp % 4) stores each stage's 12 scale atoms into its 32-lane
    // quarter of this CTA's tensor memory: lane i gets the 16-byte line i of
    // an atom (the scale words of rows i, i + 32, i + 64, i + 96) in 4
    // columns, for A's atoms j (columns 4 j ..) and B's atoms j of both row
    // blocks (16 + 8 j .., 20 + 8 j ..) -- the layout the block-scaled MMA
    // reads, which the four quarters all hold.  The stores are waited
    // for and fenced (tcgen05.fence::before_thread_sync) before the arrive;
    // the MMA thread's fence after its wait orders its MMAs behind them.
    const int q = warp & 3;
    const uint32_t sf_leader = mapa_shared(sf_bar(0), 0);
    uint32_t s = 0, ph = 0;
    bool ok = true;
    for (int tile = pair; ok && tile < num_tiles; tile += num_pairs) {
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!wait_bounded_pair(scf_bar(s), ph, abort_flag, peer_abort, 0x26u)) {
          ok = false;
          break;
        }
        const uint8_t* sa = smem + L::offSFA + s * L::kSFA + lane * 16;
        const uint8_t* sb = smem + L::offSFB + s * L::kSFB + lane * 16;
        uint32_t v[12 * kAt];
#pragma unroll
        for (int j = 0; j < kAt; ++j) {
          const uint4 a = *reinterpret_cast<const uint4*>(sa + j * 512);
          const uint4 b0 = *reinterpret_cast<const uint4*>(sb + j * 512);
          const uint4 b1 = *reinterpret_cast<const uint4*>(sb + (kAt + j) * 512);
          v[4 * j] = a.x;
          v[4 * j + 1] = a.y;
          v[4 * j + 2] = a.z;
          v[4 * j + 3] = a.w;
          v[4 * kAt + 8 * j] = b0.x;
          v[4 * kAt + 8 * j + 1] = b0.y;
          v[4 * kAt + 8 * j + 2] = b0.z;
          v[4 * kAt + 8 * j + 3] = b0.w;
          v[4 * kAt + 8 * j + 4] = b1.x;
          v[4 * kAt + 8 * j + 5] = b1.y;
          v[4 * kAt + 8 * j + 6] = b1.z;
          v[4 * kAt + 8 * j + 7] = b1.w;
        }
        const uint32_t taddr =
            tmem + ((uint32_t)(32 * q) << 16) + L::kSfCol0 + s * L::kSfColsPerStage;
#pragma unroll
        for (int c = 0; c < 12 * kAt; c += 16) tmem_st16(taddr + c, v + c);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        // relaxed: the stores have completed (wait::st) and are fenced; the
        // thread published nothing else
        if (lane == 0) mbar_arrive_cluster_relaxed(sf_leader + 8u * s);
        if (++s == STAGES) { s = 0; ph ^= 1u; }
      }
    }
  } else if (!ST && warp >= 2 && warp < 2 + kPairCopyWarps) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------- scale copies
      // the stage's copies: A's atom j (index j) and B's image of atom j (both
      // row halves; index kAt + j); copy warp cw issues the indices equal to
      // cw modulo the number of copy warps
      const int cw = warp - 2;
      uint32_t s = 0, ph = 0;
      bool ok = true, issued = false;
      for (int tile = pair; ok && tile < num_tiles; tile += num_pairs) {
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_bounded_pair(full_bar(s), ph, abort_flag, peer_abort, 0x24u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int natoms = min(kAt, args.kg - kb * kAt);
          const uint32_t sfa_t = tmem + L::kSfCol0 + s * L::kSfColsPerStage;
          const uint32_t sfb_t = sfa_t + 4 * kAt;
          const uint32_t sa = sbase + L::offSFA + s * L::kSFA;
          const uint32_t sb = sbase + L::offSFB + s * L::kSFB;
          for (int j = 0; j < natoms; ++j) {
            if (j % kPairCopyWarps == cw)
              tc_cp_pair_32x128b_warpx4(sfa_t + 4 * j, smem_desc_sf(sa + j * 512));
            if ((kAt + j) % kPairCopyWarps == cw)
              tc_cp_pair_128x256b(sfb_t + 8 * j, smem_desc_sf_image(sb + j * 4096));
          }
          issued = true;
          // the MMA thread may issue as soon as these copies are issued: the
          // fence before this arrive and the MMA thread's fence after its wait
          // order its MMAs behind them in the tensor pipe
          tc_fence_before();
          mbar_arrive(sf_bar(s));
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok && issued) {  // copies in flight must land before tensor memory is freed
        tc_commit_pair(drain_bar + 8u * (1 + cw), 1);
        wait_drain(drain_bar + 8u * (1 + cw), 0);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------------- MMA
      constexpr uint32_t idesc = FMT == kFmtNVF4 ? idesc_nvf4(256, kPairBN)
                                 : idesc_mx(256, kPairBN, FMT == kFmtMXF8 ? 0u : 1u);
      uint32_t s = 0, ph = 0, acc_ph = 0;
      bool ok = true, issued = false;
      for (int tile = pair; ok && tile < num_tiles; tile += num_pairs) {
        if (!wait_bounded_pair(acc_empty, acc_ph ^ 1u, abort_flag, peer_abort, 0x22u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < num_kb; ++kb) {
          // the copy warps observed the stage's data and issued its scale
          // copies; with stored scales the stage's A and B are waited for
          // here and the scales on the scale warps' barrier
          if ((ST && !wait_bounded_pair(full_bar(s), ph, abort_flag, peer_abort, 0x24u)) ||
              !wait_bounded_pair(sf_bar(s), ph, abort_flag, peer_abort, 0x23u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nmma = min(kAt, args.kg - kb * kAt) * PairFmt<FMT>::kMmaPerAtom;
          const uint32_t sfa_t = tmem + L::kSfCol0 + s * L::kSfColsPerStage;
          const uint32_t sfb_t = sfa_t + 4 * kAt;
          const uint32_t a0 = sbase + L::offA + s * L::kA;
          const uint32_t b0 = sbase + L::offB + s * L::kB;
          for (int j = 0; j < nmma; ++j) {
            // MMA j reads 32 bytes of K per row; its scales are atom
            // j / kMmaPerAtom, starting at byte (j % kMmaPerAtom) * kAt of
            // each row's 4-byte scale word (the scale factor ID)
            const int atom = j / PairFmt<FMT>::kMmaPerAtom;
            const uint32_t sfid = (uint32_t)(j % PairFmt<FMT>::kMmaPerAtom) * kAt;
            tc_mma_pair_bs<FMT>(tmem, smem_desc_sw128(a0 + 32 * j), smem_desc_sw128(b0 + 32 * j),
                                idesc | (sfid << 4) | (sfid << 29), sfa_t + 4 * atom,
                                sfb_t + 8 * atom, (kb | j) != 0 ? 1u : 0u);
          }
          issued = true;
          tc_commit_pair(empty_bar(s), 3);
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        tc_commit_pair(acc_full, 3);
        acc_ph ^= 1u;
      }
      if (!ok && issued) {
        tc_commit_pair(drain_bar, 1);
        wait_drain(drain_bar, 0);
      }
    }
  }
  } else {
    // -------------------------------------------------------------- epilogue
    if constexpr (ST)
      asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R::kRegsEpilogue));
    constexpr int kCols = kPairBN / 2, kChunks = kCols / 32;
    const int ew = warp - R::kEpi0;  // epilogue warp 0..7
    const int q = warp & 3, h = ew >> 2;
    const uint32_t acc_empty_leader = mapa_shared(acc_empty, 0);
    const float alpha =
        FMT == kFmtNVF4 ? __fmul_rn(__ldg(args.sdec_a), __ldg(args.sdec_b)) : 1.0f;
    uint8_t* stage_out = smem + L::offStore + ew * L::kStoreBox;
    if (DMODE == NVFP4_D_BF16 && lane == 0) prefetch_tmap(&tmD);
    uint32_t acc_ph = 0;
    for (int tile = pair; tile < num_tiles; tile += num_pairs) {
      const int m_blk = tile % args.num_m_blk, n_blk = tile / args.num_m_blk;
      if (DMODE != NVFP4_D_BF16) {
        // the rows of D (F32_ACCUM) or C (BF16_ADD_C) this warp reads for the
        // tile: into L2 while the MMAs still run
        const int64_t row = (int64_t)m_blk * 256 + rank * 128 + q * 32 + lane;
        const int64_t col0 = (int64_t)n_blk * kPairBN + h * kCols;
        if (row < args.M && col0 < args.N) {
          const int esz = DMODE == NVFP4_D_F32_ACCUM ? 4 : 2;
          const void* base = DMODE == NVFP4_D_F32_ACCUM ? args.D : args.C;
          const int64_t ncol = args.N - col0 < kCols ? args.N - col0 : kCols;
          prefetch_l2_row(static_cast<const char*>(base) + (row * args.N + col0) * esz,
                          (int)(ncol * esz));
        }
      }
      if (!wait_bounded_pair(acc_full, acc_ph, abort_flag, peer_abort, 0x33u)) break;
      tc_fence_after();
      uint32_t r[kChunks][32];
#pragma unroll
      for (int c = 0; c < kChunks; ++c)
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * kCols + c * 32), r[c]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      // the loads above have completed; a release here would also wait for
      // this warp's tensor stores of the previous tile
      if (lane == 0) mbar_arrive_cluster_relaxed(acc_empty_leader);
      acc_ph ^= 1u;
      if (DMODE == NVFP4_D_BF16) {
        // each 32-column chunk: bf16 rows into a staging box (lane = row; the
        // 16-byte pieces rotated so a warp's writes hit distinct banks), then
        // one tensor store; the box is rewritten once the store has read it
        const int32_t row0 = m_blk * 256 + (int)rank * 128 + q * 32;
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
          uint8_t* box = stage_out;
          if (lane == 0) bulk_wait_group_read<0>();
          __syncwarp();
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack_bf16x2(__fmul_rn(__uint_as_float(r[c][2 * e]), alpha),
                                __fmul_rn(__uint_as_float(r[c][2 * e + 1]), alpha));
#pragma unroll
          for (int pc = 0; pc < 4; ++pc) {
            const int piece = (pc + (lane >> 1)) & 3;
            uint4 v;
            switch (piece) {
              case 0: v = make_uint4(pk[0], pk[1], pk[2], pk[3]); break;
              case 1: v = make_uint4(pk[4], pk[5], pk[6], pk[7]); break;
              case 2: v = make_uint4(pk[8], pk[9], pk[10], pk[11]); break;
              default: v = make_uint4(pk[12], pk[13], pk[14], pk[15]); break;
            }
            *reinterpret_cast<uint4*>(box + lane * 64 + piece * 16) = v;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmD, smem_u32(box), n_blk * kPairBN + h * kCols + c * 32, row0);
            bulk_commit_group();
          }
        }
      } else {
        const int64_t row = (int64_t)m_blk * 256 + rank * 128 + q * 32 + lane;
#pragma unroll
        for (int c = 0; c < kChunks; ++c) {
          const int64_t col0 = (int64_t)n_blk * kPairBN + h * kCols + c * 32;
          if (row < args.M && col0 < args.N) store_row_chunk<DMODE>(args, row, col0, r[c], alpha);
        }
      }
    }
    if (DMODE == NVFP4_D_BF16 && lane == 0) bulk_wait_group<0>();  // stores done before exit
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}


// =============================================================================
// Wide CTA-pair kernel (NVFP4): output tiles of 256 x 384.  Per K step two
// MMAs -- N = 256 into accumulator columns [0, 256), issued by warp 1, and
// N = 128 into [256, 384), issued by warp 2 -- from one A and one B stage:
// CTA r holds A rows [128 r, 128 r + 128), B rows [128 r, 128 r + 128) (the
// first MMA's half) and [256 + 64 r, 256 + 64 r + 64) (the second's) of the
// tile, its A rows' scale atoms and all three of the tile's B row blocks'.
// A stage is 48 KB per SM for 1.5x the work of a 256-wide stage's 38 KB; the
// scales are stored by the four scale warps of each CTA, as in the pair
// kernel.  The 384 accumulator columns leave 128 of tensor memory: two scale
// slots of 64 columns ([B's third row block: 4 per atom] [A: 4 per atom]
// [B's first two row blocks: 8 per atom]); a slot is rewritten once the MMAs
// two stages back completed (this CTA's empty barrier of that stage), and
// shared memory holds 4 stages.  Each epilogue warp drains 192 columns,
// rounding each 32-column chunk to bf16 as it arrives (96 packed registers),
// then stores them (bf16 out) or folds them into FP32 (F32_ACCUM).  16
// warps: warpgroup 0 = producer, the two MMA warps, an idle warp;
// warpgroup 1 = scale warps; warpgroups 2-3 = epilogue (setmaxnreg split).
// =============================================================================
struct Pair384Smem {
  static constexpr int kStages = 4, kAt = 4;
  static constexpr uint32_t kA = 128 * kBKBytes, kB = 192 * kBKBytes;
  static constexpr uint32_t kSFA = kAt * 512, kSFB = kAt * 512 * 3;
  static constexpr uint32_t offA = 0, offB = kStages * kA, offSFA = offB + kStages * kB;
  static constexpr uint32_t offSFB = offSFA + kStages * kSFA, offBar = offSFB + kStages * kSFB;
  // full, empty, scales-ready, scales-landed per stage; acc full, acc empty;
  // a drain barrier per MMA warp
  static constexpr uint32_t kNumBars = 4 * kStages + 4;
  static constexpr uint32_t offMisc = offBar + kNumBars * 8;
  static constexpr uint32_t kStoreBox = 32 * 64;
  static constexpr uint32_t offStore = (offMisc + 16 + 127) / 128 * 128;
  static constexpr uint32_t kBytes = offStore + 8 * kStoreBox;
  static constexpr uint32_t kAlloc = kBytes + 1024;
  static constexpr uint32_t kSfCol0 = 384, kSlotCols = 64;
  static constexpr uint32_t kColB2 = 0, kColA = 16, kColB01 = 32;  // inside a slot
  static constexpr int kSlots = 2;
  static constexpr int kThreads = 512;
  static constexpr int kRegsIssue = 88, kRegsEpilogue = 168;
  static constexpr int kSplitRegs = 2 * 128 * kRegsIssue + 2 * 128 * kRegsEpilogue;
  static_assert(kSfCol0 + kSlots * kSlotCols <= kTmemCols, "tensor memory overflow");
  static_assert(kAlloc <= 232448, "shared memory overflow");
  static_assert(kSplitRegs <= kThreads * 128, "register split exceeds the launch's");
};

template <int DMODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Pair384Smem::kThreads, 1)
    gemm_nvf4_pair384_kernel(const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmB2,
                             const __grid_constant__ CUtensorMap tmSFA,
                             const __grid_constant__ CUtensorMap tmSFB,
                             const __grid_constant__ CUtensorMap tmD, const GemmArgs args) {
  static_assert(DMODE != NVFP4_D_BF16_ADD_C, "384-wide tiles take no bf16 C input");
  using L = Pair384Smem;
  constexpr int S = L::kStages, kAt = L::kAt;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::offBar;
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto sf_bar = [&](int s) { return bar0 + 8u * (2 * S + s); };
  auto scf_bar = [&](int s) { return bar0 + 8u * (3 * S + s); };
  const uint32_t acc_full = bar0 + 8u * (4 * S);
  const uint32_t acc_empty = acc_full + 8;
  const uint32_t drain_bar = acc_full + 16;  // MMA warps 1 and 2
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::offMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::offMisc + 4);
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const uint32_t peer_abort = mapa_shared(smem_u32(smem + L::offMisc + 4), rank ^ 1u);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_kb = (args.K + 255) / 256;
  const int num_tiles = args.num_m_blk * args.num_n_blk;  // 256 x 384 tiles
  const int pair = blockIdx.x >> 1, num_pairs = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 2);  // one commit per MMA warp
      mbar_init(sf_bar(s), 8);     // four scale warps in each CTA
      mbar_init(scf_bar(s), 1);
    }
    mbar_init(acc_full, 2);
    mbar_init(acc_empty, 16);  // 8 epilogue warps in each CTA
    mbar_init(drain_bar, 1);
    mbar_init(drain_bar + 8, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();

  if (warp < 8) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(L::kRegsIssue));
  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      prefetch_tmap(&tmB2);
      prefetch_tmap(&tmSFA);
      prefetch_tmap(&tmSFB);
      uint32_t s = 0, ph = 0;
      // injected stall: no loads, so every consumer's first wait runs out
      bool ok = *reinterpret_cast<volatile unsigned int*>(&g_gemm_stall) == 0u;
      for (int tile = pair; ok && tile < num_tiles; tile += num_pairs) {
        const int m_blk = tile % args.num_m_blk, n_blk = tile / args.num_m_blk;
        const int a_rb = m_blk * 2 + (int)rank;  // this CTA's 128-row block of A
        const int b_rb0 = n_blk * 3;             // the tile's first 128-row block of B
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!wait_bounded_pair(empty_bar(s), ph ^ 1u, abort_flag, peer_abort, 0x11u)) {
            ok = false;
            break;
          }
          const uint32_t fb = mapa_shared(full_bar(s), 0);
          if (leader) mbar_arrive_expect_tx(full_bar(s), 2 * (L::kA + L::kB));
          tma_load_2d_pair(sbase + L::offA + s * L::kA, &tmA, fb, kb * kBKBytes, a_rb * 128);
          tma_load_2d_pair(sbase + L::offB + s * L::kB, &tmB, fb, kb * kBKBytes,
                           n_blk * 384 + (int)rank * 128);
          tma_load_2d_pair(sbase + L::offB + s * L::kB + 128 * kBKBytes, &tmB2, fb,
                           kb * kBKBytes, n_blk * 384 + 256 + (int)rank * 64);
          // this CTA's scale atoms on its own barrier (a block past N reads as zeros)
          mbar_arrive_expect_tx(scf_bar(s), L::kSFA + L::kSFB);
          tma_load_2d(sbase + L::offSFA + s * L::kSFA, &tmSFA, scf_bar(s), 0,
                      (a_rb * args.kg + kb * kAt) * 4);
#pragma unroll
          for (int i = 0; i < 3; ++i)
            tma_load_2d(sbase + L::offSFB + s * L::kSFB + i * kAt * 512, &tmSFB, scf_bar(s), 0,
                        ((b_rb0 + i) * args.kg + kb * kAt) * 4);
          if (++s == S) { s = 0; ph ^= 1u; }
        }
      }
      if (!ok) {  // give copies already issued time to land before exit
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) {
        }
      }
    }
  } else if (warp == 1 || warp == 2) {
    if (lane == 0 && leader) {
      // ---------------------------------------------------------------- MMA
      const bool second = warp == 2;
      const uint32_t idesc = second ? idesc_nvf4(256, 128) : idesc_nvf4(256, 256);
      const uint32_t d_tmem = tmem + (second ? 256u : 0u);
      const uint32_t b_off = second ? 128u * kBKBytes : 0u;
      const uint32_t sfb_col = second ? L::kColB2 : L::kColB01;
      const uint32_t sfb_step = second ? 4u : 8u;  // columns per atom
      const uint32_t my_drain = drain_bar + (second ? 8u : 0u);
      uint32_t s = 0, ph = 0, acc_ph = 0, it = 0;
      bool ok = true, issued = false;
      for (int tile = pair; ok && tile < num_tiles; tile += num_pairs) {
        if (!wait_bounded_pair(acc_empty, acc_ph ^ 1u, abort_flag, peer_abort, 0x22u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          if (!wait_bounded_pair(full_bar(s), ph, abort_flag, peer_abort, 0x24u) ||
              !wait_bounded_pair(sf_bar(s), ph, abort_flag, peer_abort, 0x23u)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int nmma = min(kAt, args.kg - kb * kAt);
          const uint32_t slot = tmem + L::kSfCol0 + (it % L::kSlots) * L::kSlotCols;
          const uint32_t a0 = sbase + L::offA + s * L::kA;
          const uint32_t b0 = sbase + L::offB + s * L::kB + b_off;
          for (int j = 0; j < nmma; ++j)
            tc_mma_pair_nvf4(d_tmem, smem_desc_sw128(a0 + 32 * j), smem_desc_sw128(b0 + 32 * j),
                             idesc, slot + L::kColA + 4 * j, slot + sfb_col + sfb_step * j,
                             (kb | j) != 0 ? 1u : 0u);
          issued = true;
          tc_commit_pair(empty_bar(s), 3);
          if (++s == S) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        tc_commit_pair(acc_full, 3);
        acc_ph ^= 1u;
      }
      if (!ok && issued) {
        tc_commit_pair(my_drain, 1);
        wait_drain(my_drain, 0);
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ scale warps
    // as in the pair kernel, 16 atoms a stage (B's third row block, A, B's
    // first two), into the slot of the stage's iteration
    const int q = warp & 3;
    const uint32_t sf_leader = mapa_shared(sf_bar(0), 0);
    uint32_t s = 0, ph = 0, it = 0;
    bool ok = true;
    for (int tile = pair; ok && tile < num_tiles; tile += num_pairs) {
      for (int kb = 0; kb < num_kb; ++kb, ++it) {
        if (!wait_bounded_pair(scf_bar(s), ph, abort_flag, peer_abort, 0x26u)) {
          ok = false;
          break;
        }
        if (it >= (uint32_t)L::kSlots) {
          // the slot's previous stage: its MMAs completed (its empty barrier)
          const uint32_t prev = it - L::kSlots;
          if (!wait_bounded_pair(empty_bar(prev % S), (prev / S) & 1u, abort_flag, peer_abort,
                                 0x25u)) {
            ok = false;
            break;
          }
        }
        const uint8_t* sa = smem + L::offSFA + s * L::kSFA + lane * 16;
        const uint8_t* sb = smem + L::offSFB + s * L::kSFB + lane * 16;
        uint32_t v[64];
#pragma unroll
        for (int j = 0; j < kAt; ++j) {
          const uint4 b2 = *reinterpret_cast<const uint4*>(sb + (2 * kAt + j) * 512);
          const uint4 a = *reinterpret_cast<const uint4*>(sa + j * 512);
          const uint4 b0 = *reinterpret_cast<const uint4*>(sb + j * 512);
          const uint4 b1 = *reinterpret_cast<const uint4*>(sb + (kAt + j) * 512);
          const uint32_t w[16] = {b2.x, b2.y, b2.z, b2.w, a.x, a.y, a.z, a.w,
                                  b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            v[L::kColB2 + 4 * j + e] = w[e];
            v[L::kColA + 4 * j + e] = w[4 + e];
            v[L::kColB01 + 8 * j + e] = w[8 + e];
            v[L::kColB01 + 8 * j + 4 + e] = w[12 + e];
          }
        }
        const uint32_t taddr =
            tmem + ((uint32_t)(32 * q) << 16) + L::kSfCol0 + (it % L::kSlots) * L::kSlotCols;
#pragma unroll
        for (int c = 0; c < 64; c += 16) tmem_st16(taddr + c, v + c);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster_relaxed(sf_leader + 8u * s);
        if (++s == S) { s = 0; ph ^= 1u; }
      }
    }
  }
  } else {
    // -------------------------------------------------------------- epilogue
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(L::kRegsEpilogue));
    constexpr int kCols = 192, kChunks = kCols / 32;
    const int ew = warp - 8;  // epilogue warp 0..7
    const int q = warp & 3, h = ew >> 2;
    const uint32_t acc_empty_leader = mapa_shared(acc_empty, 0);
    const float alpha = __fmul_rn(__ldg(args.sdec_a), __ldg(args.sdec_b));
    uint8_t* stage_out = smem + L::offStore + ew * L::kStoreBox;
    if (DMODE == NVFP4_D_BF16 && lane == 0) prefetch_tmap(&tmD);
    uint32_t acc_ph = 0;
    for (int tile = pair; tile < num_tiles; tile += num_pairs) {
      const int m_blk = tile % args.num_m_blk, n_blk = tile / args.num_m_blk;
      const int64_t row = (int64_t)m_blk * 256 + rank * 128 + q * 32 + lane;
      const int32_t row0 = m_blk * 256 + (int)rank * 128 + q * 32;
      if (DMODE == NVFP4_D_F32_ACCUM) {  // this warp's rows of D into L2 while the MMAs run
        const int64_t col0 = (int64_t)n_blk * 384 + h * kCols;
        if (row < args.M && col0 < args.N) {
          const int64_t ncol = args.N - col0 < kCols ? args.N - col0 : kCols;
          prefetch_l2_row(static_cast<const char*>(args.D) + (row * args.N + col0) * 4,
                          (int)(ncol * 4));
        }
      }
      if (!wait_bounded_pair(acc_full, acc_ph, abort_flag, peer_abort, 0x33u)) break;
      tc_fence_after();
      uint32_t pk[kChunks][16];
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        uint32_t r[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(h * kCols + c * 32), r);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[c][e] = pack_bf16x2(__fmul_rn(__uint_as_float(r[2 * e]), alpha),
                                 __fmul_rn(__uint_as_float(r[2 * e + 1]), alpha));
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(acc_empty_leader);
      acc_ph ^= 1u;
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        const int64_t col0 = (int64_t)n_blk * 384 + h * kCols + c * 32;
        if (DMODE == NVFP4_D_BF16) {
          store_box_bf16(stage_out, lane, pk[c], &tmD, (int32_t)col0, row0);
        } else if (row < args.M && col0 < args.N) {
          fold_row_chunk_packed(args, row, col0, pk[c]);
        }
      }
    }
    if (DMODE == NVFP4_D_BF16 && lane == 0) bulk_wait_group<0>();  // stores done before exit
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// ---- host side -----------------------------------------------------------------
EncodeTiledFn encode_fn() { return tensor_map_encoder(); }

// 2-D map over a K-major code matrix [rows, kbytes] with a box of box_bytes
// (128: 128-byte swizzle, 64: 64-byte swizzle) x box_rows.
bool make_code_map(CUtensorMap* map, const void* base, int64_t rows, int64_t kbytes,
                   int box_rows, int box_bytes = kBKBytes) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kbytes, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kbytes};
  const cuuint32_t box[2] = {(cuuint32_t)box_bytes, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             box_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over a scale tensor viewed as rows of 128 bytes (4 rows per atom),
// box of 16 rows (the 4 atoms of one stage).
bool make_sf_map(CUtensorMap* map, const void* base, size_t bytes, int box_rows = 16) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {128, (cuuint64_t)(bytes / 128)};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 5-D map over a scale tensor (atoms of 4 rows x 128 bytes, kg per 128-row
// block) that reads each atom four times: dimensions (byte, atom row, copy
// [stride 0], row block, atom along K); a box of (128, 4, 4, 2, atoms) brings
// one stage's B scales (its atoms x 2 row blocks) as 4 KB images, each two
// 2 KB planes of one atom repeated for the four 32-lane quarters.
bool make_sf_image_map(CUtensorMap* map, const void* base, int kg, int64_t row_blocks,
                       int atoms) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[5] = {128, 4, 4, (cuuint64_t)row_blocks, (cuuint64_t)kg};
  const cuuint64_t strides[4] = {128, 0, (cuuint64_t)kg * 512, 512};
  const cuuint32_t box[5] = {128, 4, 4, 2, (cuuint32_t)atoms};
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over a bf16 output [rows, cols] with 32 x 32 boxes (no swizzle);
// tensor stores skip the part of a box outside the matrix.
bool make_out_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)(cols * 2)};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Per-device, once-per-kernel launch set-up of a GEMM kernel, under a lock:
// its dynamic shared memory attribute, for a kernel that splits registers
// with setmaxnreg the check that the compiled count covers the split
// (setmaxnreg.inc waits until the registers it asks for are free in the
// block's launch allotment, so a split above it would wait forever), and
// for a CTA-pair kernel how many pairs are resident at once (cluster
// placement can leave SMs of a GPC unpaired).  Returns the resident pairs
// (1 for a single-SM kernel), 0 when the set-up failed.
struct GemmLaunchState {
  std::mutex mu;
  int resident[64] = {};  // per device: 0 not yet set up, -1 refused for good
};

template <typename K>
int gemm_setup(GemmLaunchState& ls, K kern, uint32_t smem, int threads, int split_regs,
               bool pair, int sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(ls.mu);
  if (ls.resident[dev] == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
      return 0;
    if (split_regs > 0) {
      cudaFuncAttributes fa;
      if (cudaFuncGetAttributes(&fa, kern) != cudaSuccess) return 0;
      if (fa.numRegs * threads < split_regs) {
        ls.resident[dev] = -1;  // the compiled kernel can never run
        return 0;
      }
    }
    int n = 1;
    if (pair) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * (sms / 2));
      cfg.blockDim = dim3(threads);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr;
      attr.id = cudaLaunchAttributeClusterDimension;
      attr.val.clusterDim.x = 2;
      attr.val.clusterDim.y = 1;
      attr.val.clusterDim.z = 1;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) n = sms / 2;
      n = std::min(n, sms / 2);
    }
    ls.resident[dev] = n;
  }
  return ls.resident[dev] > 0 ? ls.resident[dev] : 0;
}

template <int STAGES, int DMODE, int FMT, bool IMG>
nvfp4_status launch_pair(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& msa,
                         const CUtensorMap& msb, const CUtensorMap& md, const GemmArgs& a, int sms,
                         cudaStream_t stream) {
  using L = PairSmem<STAGES, FMT, IMG>;
  auto kern = gemm_nvf4_pair_kernel<STAGES, DMODE, FMT, IMG>;
  using R = PairRoles<L::kST>;
  static GemmLaunchState ls;
  // persistent grid: as many pairs as are resident at once, at most one per tile
  const int max_pairs =
      gemm_setup(ls, kern, L::kAlloc, R::kThreads, L::kST ? R::kSplitRegs : 0, true, sms);
  if (max_pairs <= 0) return NVFP4_ERR_CUDA;
  const int tiles = a.num_m_blk * a.num_n_blk;
  const int grid = 2 * std::min(tiles, max_pairs);
  return launch_pdl(kern, grid, R::kThreads, L::kAlloc, stream, ma, mb, msa, msb, md, a) ==
                 cudaSuccess
             ? NVFP4_OK
             : NVFP4_ERR_CUDA;
}


template <int DMODE>
nvfp4_status launch_pair384(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mb2,
                            const CUtensorMap& msa, const CUtensorMap& msb, const CUtensorMap& md,
                            const GemmArgs& a, int sms, cudaStream_t stream) {
  using L = Pair384Smem;
  auto kern = gemm_nvf4_pair384_kernel<DMODE>;
  static GemmLaunchState ls;
  const int max_pairs = gemm_setup(ls, kern, L::kAlloc, L::kThreads, L::kSplitRegs, true, sms);
  if (max_pairs <= 0) return NVFP4_ERR_CUDA;
  const int tiles = a.num_m_blk * a.num_n_blk;
  const int grid = 2 * std::min(tiles, max_pairs);
  return launch_pdl(kern, grid, L::kThreads, L::kAlloc, stream, ma, mb, mb2, msa, msb, md, a) ==
                 cudaSuccess
             ? NVFP4_OK
             : NVFP4_ERR_CUDA;
}

template <int BN, int STAGES, int DMODE, int BKB>
nvfp4_status launch(const CUtensorMap& ma, const CUtensorMap& mb, const GemmArgs& a, int sms,
                    cudaStream_t stream) {
  using L = Smem<BN, STAGES, BKB>;
  auto kern = gemm_nvf4_kernel<BN, STAGES, DMODE, BKB>;
  static GemmLaunchState ls;
  if (gemm_setup(ls, kern, L::kAlloc, kThreads, 0, false, sms) <= 0) return NVFP4_ERR_CUDA;
  // persistent grid: one CTA per SM (tensor memory and shared memory admit
  // one), at most one per output tile
  const int units = a.num_m_blk * a.num_n_blk;
  return launch_pdl(kern, std::min(units, sms), kThreads, L::kAlloc, stream, ma, mb, a) ==
                 cudaSuccess
             ? NVFP4_OK
             : NVFP4_ERR_CUDA;
}

template <int BN, int STAGES, int BKB>
nvfp4_status launch_mode(int d_mode, const CUtensorMap& ma, const CUtensorMap& mb,
                         const GemmArgs& a, int sms, cudaStream_t s) {
  switch (d_mode) {
    case NVFP4_D_BF16: return launch<BN, STAGES, NVFP4_D_BF16, BKB>(ma, mb, a, sms, s);
    case NVFP4_D_F32_ACCUM:
      return launch<BN, STAGES, NVFP4_D_F32_ACCUM, BKB>(ma, mb, a, sms, s);
    default: return launch<BN, STAGES, NVFP4_D_BF16_ADD_C, BKB>(ma, mb, a, sms, s);
  }
}

template <int STAGES>
nvfp4_status launch_pair_mode(int d_mode, const CUtensorMap& ma, const CUtensorMap& mb,
                              const CUtensorMap& msa, const CUtensorMap& msb,
                              const CUtensorMap& md, const GemmArgs& a, int sms, cudaStream_t s) {
  switch (d_mode) {
    case NVFP4_D_BF16:
      return launch_pair<STAGES, NVFP4_D_BF16, kFmtNVF4, false>(ma, mb, msa, msb, md, a, sms, s);
    case NVFP4_D_F32_ACCUM:
      return launch_pair<STAGES, NVFP4_D_F32_ACCUM, kFmtNVF4, false>(ma, mb, msa, msb, md, a, sms,
                                                                     s);
    default:
      return launch_pair<STAGES, NVFP4_D_BF16_ADD_C, kFmtNVF4, false>(ma, mb, msa, msb, md, a, sms,
                                                                      s);
  }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

EncodeTiledFn tensor_map_encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

nvfp4_status gemm_set_injection(unsigned int stall, unsigned long long wait_ns) {
  if (cudaMemcpyToSymbol(g_gemm_stall, &stall, sizeof(stall)) != cudaSuccess ||
      cudaMemcpyToSymbol(g_gemm_wait_ns, &wait_ns, sizeof(wait_ns)) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  return NVFP4_OK;
}

nvfp4_status gemm_read_error(unsigned int* code) {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemm_error, sizeof(v)) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (v && cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(zero)) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  *code = v;
  return NVFP4_OK;
}

nvfp4_status gemm_impl(const nvfp4_tensor* A, int32_t a_view, const nvfp4_tensor* B,
                       int32_t b_view, void* D, int32_t d_mode, const void* C, int64_t M,
                       int64_t N, int64_t K, int32_t tile, cudaStream_t stream) {
  if (!A || !B || !D) return NVFP4_ERR_INVALID_ARG;
  if (a_view < 0 || a_view > 1 || b_view < 0 || b_view > 1) return NVFP4_ERR_INVALID_ARG;
  if (d_mode < NVFP4_D_BF16 || d_mode > NVFP4_D_BF16_ADD_C) return NVFP4_ERR_INVALID_ARG;
  if (d_mode == NVFP4_D_BF16_ADD_C && !C) return NVFP4_ERR_INVALID_ARG;
  if (tile < NVFP4_TILE_AUTO || tile > NVFP4_TILE_PAIR_256X384 || tile == 4)
    return NVFP4_ERR_INVALID_ARG;  // 4: a retired configuration
  if (tile == NVFP4_TILE_PAIR_256X384 && d_mode == NVFP4_D_BF16_ADD_C)
    return NVFP4_ERR_INVALID_ARG;
  const void* a_codes = a_view ? A->codes_t : A->codes;
  const void* a_sf = a_view ? A->scales_t : A->scales;
  const void* b_codes = b_view ? B->codes_t : B->codes;
  const void* b_sf = b_view ? B->scales_t : B->scales;
  if (!a_codes || !a_sf || !b_codes || !b_sf || !A->s_dec || !B->s_dec)
    return NVFP4_ERR_INVALID_ARG;
  const int64_t a_rows = a_view ? A->cols : A->rows, a_cols = a_view ? A->rows : A->cols;
  const int64_t b_rows = b_view ? B->cols : B->rows, b_cols = b_view ? B->rows : B->cols;
  if (M <= 0 || N <= 0 || K <= 0 || K % 64 || N % 8) return NVFP4_ERR_SHAPE;
  if (a_rows != M || b_rows != N || a_cols != K || b_cols != K) return NVFP4_ERR_SHAPE;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return NVFP4_ERR_SHAPE;
  if (!aligned16(a_codes) || !aligned16(b_codes) || !aligned16(a_sf) || !aligned16(b_sf) ||
      !aligned16(D) || (C && !aligned16(C)))
    return NVFP4_ERR_ALIGN;

  DeviceInfo dev;
  nvfp4_status st = current_device(&dev);
  if (st != NVFP4_OK) return st;

  if (tile == NVFP4_TILE_AUTO) {
    // the CTA pair when its 256 x 256 tiles still give every pair of SMs
    // work; smaller problems keep more, smaller tiles.  Between the pair's
    // two widths, the one whose rounds of tiles per pair cost less: a
    // 384-wide tile took 1.2x the time of a 256-wide one on the Llama-3-8B
    // shapes (same K); bf16 C input stays on the 256-wide tile.
    const int64_t pairs = std::max(1, dev.sm_count / 2);
    const int64_t mt = (M + 255) / 256;
    const int64_t t256 = mt * ((N + 255) / 256), t384 = mt * ((N + 383) / 384);
    if (N <= 128) {
      tile = NVFP4_TILE_128X128;
    } else if (t256 >= pairs) {
      const int64_t w256 = (t256 + pairs - 1) / pairs, w384 = (t384 + pairs - 1) / pairs;
      tile = (d_mode != NVFP4_D_BF16_ADD_C && 6 * w384 < 5 * w256) ? NVFP4_TILE_PAIR_256X384
                                                                  : NVFP4_TILE_PAIR_256X256;
    } else {
      tile = NVFP4_TILE_128X256;
    }
  }
  GemmArgs a;
  a.sfa = static_cast<const uint8_t*>(a_sf);
  a.sfb = static_cast<const uint8_t*>(b_sf);
  a.sdec_a = A->s_dec;
  a.sdec_b = B->s_dec;
  a.D = D;
  a.C = C;
  a.M = (int)M;
  a.N = (int)N;
  a.K = (int)K;
  a.kg = (int)(K / 64);
  a.nrb_b = (int)((N + 127) / 128);
  a.nrb_a = (int)((M + 127) / 128);
  CUtensorMap ma, mb;
  if (tile == NVFP4_TILE_PAIR_256X384) {
    // B's last 128 tile rows arrive as 64-row boxes, one per CTA
    CUtensorMap mb2, msa, msb, md;
    if (!make_code_map(&ma, a_codes, M, K / 2, 128) || !make_code_map(&mb, b_codes, N, K / 2, 128) ||
        !make_code_map(&mb2, b_codes, N, K / 2, 64) ||
        !make_sf_map(&msa, a_sf, swizzled_scale_bytes(M, K)) ||
        !make_sf_map(&msb, b_sf, swizzled_scale_bytes(N, K)))
      return NVFP4_ERR_CUDA;
    if (d_mode == NVFP4_D_BF16) {
      if (!make_out_map(&md, D, M, N)) return NVFP4_ERR_CUDA;
    } else {
      md = ma;
    }
    a.num_m_blk = (int)((M + 255) / 256);
    a.num_n_blk = (int)((N + 383) / 384);
    return d_mode == NVFP4_D_BF16
               ? launch_pair384<NVFP4_D_BF16>(ma, mb, mb2, msa, msb, md, a, dev.sm_count, stream)
               : launch_pair384<NVFP4_D_F32_ACCUM>(ma, mb, mb2, msa, msb, md, a, dev.sm_count,
                                                   stream);
  }
  if (tile == NVFP4_TILE_PAIR_256X256) {
    CUtensorMap msa, msb, md;
    if (!make_code_map(&ma, a_codes, M, K / 2, 128) || !make_code_map(&mb, b_codes, N, K / 2, 128) ||
        !make_sf_map(&msa, a_sf, swizzled_scale_bytes(M, K)) ||
        !make_sf_map(&msb, b_sf, swizzled_scale_bytes(N, K)))
      return NVFP4_ERR_CUDA;
    // bf16 output map for the tensor-store epilogue (other modes do not use it)
    if (d_mode == NVFP4_D_BF16) {
      if (!make_out_map(&md, D, M, N)) return NVFP4_ERR_CUDA;
    } else {
      md = ma;
    }
    a.num_m_blk = (int)((M + 255) / 256);
    a.num_n_blk = (int)((N + 255) / 256);
    return launch_pair_mode<5>(d_mode, ma, mb, msa, msb, md, a, dev.sm_count, stream);
  }
  const int bn = tile == NVFP4_TILE_128X128 ? 128 : 256;
  const int bkb = tile == NVFP4_TILE_128X256_K128 ? 64 : 128;  // stage K bytes per row
  if (!make_code_map(&ma, a_codes, M, K / 2, kBM, bkb) ||
      !make_code_map(&mb, b_codes, N, K / 2, bn, bkb))
    return NVFP4_ERR_CUDA;
  a.num_m_blk = (int)((M + kBM - 1) / kBM);
  a.num_n_blk = (int)((N + bn - 1) / bn);
  if (bkb == 64) return launch_mode<256, 8, 64>(d_mode, ma, mb, a, dev.sm_count, stream);
  if (bn == 256) return launch_mode<256, 4, 128>(d_mode, ma, mb, a, dev.sm_count, stream);
  return launch_mode<128, 6, 128>(d_mode, ma, mb, a, dev.sm_count, stream);
}

// D bf16 [M, N] = A . B^T for MX operands (codes K-major; scales in the MMA
// layout, one atom per 128 rows and 128 K elements), on the CTA-pair kernel.
nvfp4_status gemm_mx_impl(const void* a_codes, const void* a_sf, const void* b_codes,
                          const void* b_sf, int32_t fmt, void* D, int64_t M, int64_t N,
                          int64_t K, cudaStream_t stream) {
  if (!a_codes || !a_sf || !b_codes || !b_sf || !D) return NVFP4_ERR_INVALID_ARG;
  if (fmt != NVFP4_MXFP4 && fmt != NVFP4_MXFP8) return NVFP4_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || K % 128 || N % 8) return NVFP4_ERR_SHAPE;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return NVFP4_ERR_SHAPE;
  if (!aligned16(a_codes) || !aligned16(b_codes) || !aligned16(a_sf) || !aligned16(b_sf) ||
      !aligned16(D))
    return NVFP4_ERR_ALIGN;
  DeviceInfo dev;
  nvfp4_status st = current_device(&dev);
  if (st != NVFP4_OK) return st;
  GemmArgs a = {};
  a.sfa = static_cast<const uint8_t*>(a_sf);
  a.sfb = static_cast<const uint8_t*>(b_sf);
  a.D = D;
  a.M = (int)M;
  a.N = (int)N;
  a.K = (int)K;
  a.kg = (int)(K / 128);  // scale atoms per 128-row block along K
  a.nrb_b = (int)((N + 127) / 128);
  a.nrb_a = (int)((M + 127) / 128);
  a.num_m_blk = (int)((M + 255) / 256);
  a.num_n_blk = (int)((N + 255) / 256);
  const int64_t kbytes = fmt == NVFP4_MXFP4 ? K / 2 : K;
  const int atoms = fmt == NVFP4_MXFP4 ? PairFmt<kFmtMXF4>::kAtoms : PairFmt<kFmtMXF8>::kAtoms;
  CUtensorMap ma, mb, msa, msb, md;
  if (!make_code_map(&ma, a_codes, M, kbytes, 128) || !make_code_map(&mb, b_codes, N, kbytes, 128) ||
      !make_sf_map(&msa, a_sf, (size_t)a.nrb_a * a.kg * 512, 4 * atoms) ||
      !make_sf_image_map(&msb, b_sf, a.kg, a.nrb_b, atoms) ||
      !make_out_map(&md, D, M, N))
    return NVFP4_ERR_CUDA;
  return fmt == NVFP4_MXFP4
             ? launch_pair<5, NVFP4_D_BF16, kFmtMXF4, true>(ma, mb, msa, msb, md, a, dev.sm_count,
                                                            stream)
             : launch_pair<5, NVFP4_D_BF16, kFmtMXF8, true>(ma, mb, msa, msb, md, a, dev.sm_count,
                                                            stream);
}

}  // namespace nvfp4
