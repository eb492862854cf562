// common.cuh -- device helpers shared by the NVFP4 kernels (sm_103a only):
// inline-PTX wrappers for mbarrier, TMA, tcgen05 and the FP4/FP8 conversion
// instructions, the Philox4x32-10 counter RNG, and E4M3/E2M1 helpers.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/nvfp4.h"

#define NVFP4_DEV __device__ __forceinline__

namespace nvfp4 {

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): ten rounds of the
// published multiply-xor S-box; the key is bumped by the Weyl constants
// between rounds.
// ---------------------------------------------------------------------------
NVFP4_DEV uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

// The twenty round keys of Philox4x32-10 for one 64-bit key (round i uses
// key + i * Weyl constants): computed once on the host and read by the
// kernels from their parameters, so a call costs only the ten S-box rounds.
struct PhiloxKeys {
  uint32_t k[20];
};
inline PhiloxKeys philox_round_keys(uint64_t seed) {
  PhiloxKeys r;
  uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
  for (int i = 0; i < 10; ++i) {
    r.k[2 * i] = k0;
    r.k[2 * i + 1] = k1;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return r;
}
NVFP4_DEV uint4 philox4x32_10_rk(uint4 c, const PhiloxKeys& rk) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint32_t lo0 = 0xD2511F53u * c.x, hi0 = __umulhi(0xD2511F53u, c.x);
    const uint32_t lo1 = 0xCD9E8D57u * c.z, hi1 = __umulhi(0xCD9E8D57u, c.z);
    c = make_uint4(hi1 ^ c.y ^ rk.k[2 * round], lo1, hi0 ^ c.w ^ rk.k[2 * round + 1], lo0);
  }
  return c;
}

// Stochastic-rounding words for the 4 consecutive output elements starting at
// linear index idx4 (a multiple of 4): counter (idx4/4, stream 0, offset).
NVFP4_DEV uint4 sr_words(const PhiloxKeys& rk, uint64_t offset, uint64_t idx4) {
  const uint64_t g = idx4 >> 2;
  return philox4x32_10_rk(make_uint4((uint32_t)g, (uint32_t)(g >> 32), 0u, (uint32_t)offset), rk);
}

// 16 RHT sign bits (bit i set -> sign -1): word 0 of counter (0, 0, 1, 0).
NVFP4_DEV uint32_t rht_sign_bits(uint64_t seed) {
  return philox4x32_10(make_uint4(0u, 0u, 1u, 0u), (uint32_t)seed, (uint32_t)(seed >> 32)).x &
         0xFFFFu;
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

// max |(H16 diag(s) v)_i| over one block whose random signs s were applied
// already, without the transform's x 1/4 (applied by the caller to its final
// maximum: rounding is monotone, so that maximum is the same bit for bit).
// Butterfly stages h = 1, 2, 4 as in the full transform; the last stage
// turns each pair (a, b) into a + b and a - b, and the larger magnitude of
// the two rounded results is exactly the rounded |a| + |b| (one of them is
// that sum, the other is no larger), so the stage is one add per pair.  v is
// overwritten.
NVFP4_DEV float rht16_absmax_signed(float (&v)[16]) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if ((i & h) == 0) {
        const float a = v[i], b = v[i + h];
        v[i] = __fadd_rn(a, b);
        v[i + h] = __fsub_rn(a, b);
      }
    }
  }
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, __fadd_rn(fabsf(v[i]), fabsf(v[i + 8])));
  return m;
}
// As rht16_absmax_signed, with the random signs applied here.
NVFP4_DEV float rht16_absmax_unscaled(float (&v)[16], uint32_t sign_bits) {
#pragma unroll
  for (int i = 0; i < 16; ++i)
    if ((sign_bits >> i) & 1u) v[i] = -v[i];
  return rht16_absmax_signed(v);
}

// The 16-point transform of one register-resident block whose random signs
// were applied as it was loaded (rht_sign_masks): stages h = 1, 2, 4, 8,
// then x 1/4.
NVFP4_DEV void rht16_signed_block(float (&v)[16]) {
  butterfly_local<16>(v);
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __fmul_rn(v[i], 0.25f);
}

// The transform's signs as XOR masks, one per row e of a 16-row block: bit 31
// set where sign bit e negates that row.
NVFP4_DEV void rht_sign_masks(uint32_t sign_bits, uint32_t (&m)[16]) {
#pragma unroll
  for (int e = 0; e < 16; ++e) m[e] = ((sign_bits >> e) & 1u) << 31;
}

// ---------------------------------------------------------------------------
// Format conversions.  E4M3 here is the FN variant (max 448, no infinity).
// ---------------------------------------------------------------------------
// RNE + saturation of one non-negative float to an E4M3 byte.
NVFP4_DEV uint32_t e4m3_rn_satfinite(float t) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(t));
  return r & 0xFFu;  // the second source lands in the low byte
}

// Exact value of an E4M3FN byte (no NaN expected: scales are finite).
NVFP4_DEV float e4m3_value(uint32_t b) {
  const uint32_t e = (b >> 3) & 15u, m = b & 7u;
  float mag;
  if (e == 0) mag = (float)m * 0.001953125f;  // m * 2^-9
  else mag = __uint_as_float(((e + 120u) << 23) | (m << 20));
  return (b & 0x80u) ? -mag : mag;
}

// Two floats -> one byte of E2M1 codes with RNE and saturation to +-6:
// `lo` goes to the low nibble (even element), `hi` to the high nibble.
NVFP4_DEV uint32_t e2m1x2_rn(float lo, float hi) {
  uint16_t r;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u16.u8 %0, t;\n}"
      : "=h"(r) : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

// Stochastic rounding of a magnitude onto the E2M1 grid {0,.5,1,1.5,2,3,4,6}:
// a = the bits of |y|; rounds |y| up to the next grid value iff
// r < floor(frac * 2^32), frac = (|y| - lo) / (hi - lo).  Returns the 3-bit
// magnitude code; |y| >= 6 saturates (the caller adds the sign).  Evaluated
// exactly and without branches on the float's bits: for |y| >= 1 the grid
// keeps one mantissa bit and frac * 2^32 is the 22 bits below it shifted
// left by 10, so r < thr iff the 22-bit complement of r's top 22 bits, added
// to those bits, carries into the kept bit -- adding it to the whole word
// performs the round-up, binade changes included, and the code is read off
// bits 22 and up.  On [0.5, 1) the same holds with 23 bits (the carry
// reaches the exponent); below 0.5 the threshold is floor(|y| * 2^33), an
// exact power-of-two scaling.
NVFP4_DEV uint32_t e2m1_sr_mag(uint32_t a, uint32_t r) {
  const bool ge1 = a >= 0x3F800000u;
  const uint32_t t = a + ((~r) >> (ge1 ? 10 : 9));
  const uint32_t code_hi = ge1 ? (t >> 22) - 252u : (t >> 23) - 125u;
  const uint32_t thr = __float2uint_rz(__fmul_rn(__uint_as_float(a), 8589934592.0f));
  const uint32_t code = a < 0x3F000000u ? (thr > r ? 1u : 0u) : code_hi;
  // |y| >= 6 (or not finite) saturates: code_hi is at least 7 there, and never
  // above 7 below it (lo = 4 rounds up to code 7 at most)
  return min(code, 7u);
}

// The sign bits of eight values at the sign positions of their 4-bit codes
// (bit 4 i + 3 = sign of v[i]): the top bytes of v[1], v[3], v[5], v[7]
// gathered into bytes 0..3 put each sign at bit 8 k + 7; those of the even
// elements, gathered likewise and shifted down by 4, at bit 8 k + 3.
NVFP4_DEV uint32_t sign_nibbles8(const float (&v)[8]) {
  uint32_t b[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) b[i] = __float_as_uint(v[i]);
  const uint32_t odd =
      __byte_perm(__byte_perm(b[1], b[3], 0x0073), __byte_perm(b[5], b[7], 0x0073), 0x5410);
  const uint32_t even =
      __byte_perm(__byte_perm(b[0], b[2], 0x0073), __byte_perm(b[4], b[6], 0x0073), 0x5410);
  return (odd & 0x80808080u) | ((even >> 4) & 0x08080808u);
}

// Correctly rounded a / 6 for a >= 2^-100 without a division: the product
// with RN(1/6), one exact FMA residual and one FMA correction (Markstein's
// correction step; correct rounding checked exhaustively over every binary32
// finite a >= 2^-100).  Smaller a (subnormal quotients), infinities and NaN
// take the IEEE division.
NVFP4_DEV float div6_rn(float a) {
  const float c = 0x1.555556p-3f;  // RN(1/6)
  if (!(a >= 0x1p-100f && a <= 0x1.fffffep127f)) return __fdiv_rn(a, 6.0f);
  const float q0 = __fmul_rn(a, c);
  const float res = __fmaf_rn(-q0, 6.0f, a);
  return __fmaf_rn(res, c, q0);
}

// Per-tensor encode scale from the amax: 6*448/amax, 1 for 0, FLT_MAX if the
// quotient is not finite.
NVFP4_DEV float per_tensor_s_enc(float amax) {
  if (amax == 0.0f) return 1.0f;
  float s = __fdiv_rn(2688.0f, amax);
  if (!isfinite(s)) s = 3.402823466e38f;
  return s;
}

// Byte offset of (row r, scale column c) in the MMA scale layout of an
// operand whose padded scale-column count is pc4 (a multiple of 4).
NVFP4_DEV int64_t sf_offset(int64_t r, int64_t c, int64_t pc4) {
  return ((r >> 7) * (pc4 >> 2) + (c >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (c & 3);
}


// ---------------------------------------------------------------------------
// Shared memory / mbarrier / TMA
// ---------------------------------------------------------------------------
NVFP4_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

NVFP4_DEV void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization (launch_pdl) may be scheduled while the kernel before it on
// the stream is still finishing, so it runs its on-chip setup (barriers,
// tensor memory, tables) early and waits here -- for that kernel to complete
// and its writes to be visible -- before it reads or writes global memory.
// Returns at once in a kernel launched without the attribute.  Then lets the
// next kernel on the stream be scheduled (its CTAs take whatever room this
// grid leaves and wait in their own griddep_wait): every CTA of this grid is
// resident and running by the time all of them have passed this point.
NVFP4_DEV void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

NVFP4_DEV void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
NVFP4_DEV void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
NVFP4_DEV void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
NVFP4_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
NVFP4_DEV uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

NVFP4_DEV void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x,
                           int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
NVFP4_DEV void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// Tensor store of a shared-memory box to global memory (bulk async group of
// the issuing thread); elements outside the tensor are not written.
NVFP4_DEV void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
NVFP4_DEV void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until at most N of this thread's bulk groups still read shared memory.
template <int N>
NVFP4_DEV void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until at most N of this thread's bulk groups are incomplete.
template <int N>
NVFP4_DEV void bulk_wait_group() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
// Generic-proxy shared-memory writes made visible to the async proxy (TMA).
NVFP4_DEV void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
NVFP4_DEV void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor cores, accumulators in tensor memory)
// ---------------------------------------------------------------------------
NVFP4_DEV void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
NVFP4_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
NVFP4_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
NVFP4_DEV void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
NVFP4_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Arrive on `bar` once every tcgen05 operation this thread issued completes.
NVFP4_DEV void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
// Copy 32 rows x 128 bits of shared memory to tensor memory, replicated into
// each of the four 32-lane quarters (the scale-factor copy).
NVFP4_DEV void tc_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}
// D(tmem) (+)= A(smem) . B(smem)^T with E2M1 operands and one UE4M3 scale per
// 16 elements of K (scales in tensor memory); K = 64 per instruction.
NVFP4_DEV void tc_mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                           uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}
// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp receives
// lane (quarter base + i), columns taddr.col .. +31.
NVFP4_DEV void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
NVFP4_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// 32 lanes x 16 consecutive 32-bit columns: thread i of the warp stores r to
// lane (quarter base + i), columns taddr.col .. +15.
NVFP4_DEV void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
NVFP4_DEV void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------------------
// CTA pair (cluster of 2, tcgen05 cta_group::2): one MMA spans both SMs.
// Each CTA holds its half of A and of B in its own shared memory, its own
// rows' A scales and the full B scales; tensor-memory allocations and scale
// copies happen in both CTAs, the leader (rank 0) issues copies and MMAs.
// ---------------------------------------------------------------------------
NVFP4_DEV uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
NVFP4_DEV void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
}
// Address of the same shared-memory location in cluster CTA `rank`.
NVFP4_DEV uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Relaxed arrive on an mbarrier of any CTA in the cluster: no release fence,
// so it does not wait for the thread's earlier memory operations (bulk tensor
// stores still in flight, for one).  For signals whose ordering is already
// established otherwise, e.g. tensor-memory loads completed by
// tcgen05.wait::ld and fenced by tcgen05.fence::before_thread_sync.
NVFP4_DEV void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
NVFP4_DEV void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
// TMA tile load into this CTA's shared memory whose completion is counted on
// an mbarrier of either CTA of the pair (the leader's).
NVFP4_DEV void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}
// 5-D variant (coordinates 0, 0, 0, x3, x4) completing on a pair barrier.
NVFP4_DEV void tma_load_5d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                int32_t x3, int32_t x4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %3, %3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(0), "r"(x3), "r"(x4)
      : "memory");
}
NVFP4_DEV void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
NVFP4_DEV void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
NVFP4_DEV void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Arrive on the same-offset mbarrier of every CTA in `mask` when all prior
// tcgen05 operations of this thread complete.
NVFP4_DEV void tc_commit_pair(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}
// Scale-atom copy in both CTAs: each CTA's shared memory to its own tensor
// memory, replicated into the four 32-lane quarters.
NVFP4_DEV void tc_cp_pair_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}
// 128 lanes x 256 bits in both CTAs: row L of each CTA's image (two 16-byte
// chunks) to lane L, columns base .. base + 7.
NVFP4_DEV void tc_cp_pair_128x256b(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// Descriptor of a 128-row x 32-byte image stored as two 2 KB chunk planes
// (bytes 0-15 of row L at L * 16, bytes 16-31 at 2048 + L * 16); the copy
// puts plane 0 in columns base .. base + 3 and plane 1 in base + 4 .. + 7.
NVFP4_DEV uint64_t smem_desc_sf_image(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(2048 >> 4) << 16;  // leading byte offset: the second 16-byte chunk
  d |= (uint64_t)(128 >> 4) << 32;   // stride byte offset: next 8 rows
  d |= (uint64_t)1 << 46;
  return d;
}
// Pair MMA: D (M = 256 split over the two CTAs' tensor memory) (+)= A . B^T.
NVFP4_DEV void tc_mma_pair_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// Shared-memory matrix descriptor, K-major operand with the 128-byte swizzle:
// rows of 128 bytes, 8-row (1024-byte) swizzle atoms stacked 1024 bytes apart.
NVFP4_DEV uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)1 << 16;                 // leading byte offset (unused when swizzled)
  d |= (uint64_t)(1024 >> 4) << 32;       // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                 // descriptor version for tcgen05
  d |= (uint64_t)2 << 61;                 // SWIZZLE_128B
  return d;
}
// Descriptor of a 32-row x 16-byte scale-factor block (no swizzle, 8-row core
// matrices of 128 contiguous bytes).
NVFP4_DEV uint64_t smem_desc_sf(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(128 >> 4) << 32;        // stride byte offset: next 8 rows
  d |= (uint64_t)1 << 46;
  return d;
}

// Instruction descriptor for kind::mxf4nvf4: E2M1 A and B (K-major), UE4M3
// scales, dense, M x N tile.
__host__ __device__ constexpr uint32_t idesc_nvf4(int M, int N) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

}  // namespace nvfp4
