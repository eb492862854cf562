/*
 * nvfp4_oracle.c -- plain, slow, single-threaded CPU oracle (TEST
 * INFRASTRUCTURE ONLY; see nvfp4_oracle.h for who may use it).
 *
 * Every step follows the "NVFP4 pretraining recipe" page (re-post of NVIDIA's
 * NVFP4 pretraining blog), written from its description in the order the
 * recipe gives it:
 *   - 16-element micro-blocks  ("NVFP4 pretraining recipe", bullet 1);
 *   - E4M3 block scale under an FP32 per-tensor scale (bullet 2, and the
 *     "two-level microscaling" of "NVFP4 format and advantages");
 *   - random Hadamard transform on the WGRAD inputs only (bullet 3);
 *   - one E4M3 scale per 16x16 weight tile, shared by FPROP and the
 *     transposed DGRAD (bullet 4);
 *   - stochastic rounding on gradients, RNE on weights/activations (bullet 5);
 *   - NVFP4 inputs, BF16 outputs for FPROP/DGRAD/WGRAD (Figure 1 text).
 * Constants the page does not print (E2M1 grid, E4M3 maximum 448, the 6*448
 * per-tensor mapping, the 16-point Sylvester Hadamard, Philox4x32-10) are the
 * plain readings recorded in the design notes.
 *
 * Build: cc -O2 -std=c11 -ffp-contract=off -fno-fast-math -shared -fPIC
 */
#include "nvfp4_oracle.h"

#include <float.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ======================================================================== */
/* E2M1 ("NVFP4 format and advantages"; element format of bullet 1).
 * Bit layout s.ee.m, exponent bias 1, ee == 0 is subnormal (0 or 0.5).     */
/* ======================================================================== */
float orc_e2m1_value(uint8_t code) {
  int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  float mag;
  if (e == 0) mag = 0.5f * (float)m;                                   /* subnormal */
  else        mag = (1.0f + 0.5f * (float)m) * (float)(1 << (e - 1));  /* 2^(e-1)(1+m/2) */
  return s ? -mag : mag;
}

/* Magnitude of 3-bit code i, from the bit definition above. */
static float e2m1_mag(int i) { return orc_e2m1_value((uint8_t)i); }

/* Round-to-nearest-even onto the E2M1 grid with saturation to +-6 (bullet 5:
 * weights and activations use RNE).  A tie goes to the code whose mantissa
 * bit is 0.  The sign is kept, so a negative value that rounds to zero gives
 * the negative-zero code 0x8. */
uint8_t orc_e2m1_rne(float y) {
  uint8_t sign = signbit(y) ? 0x8 : 0x0;
  float a = fabsf(y);
  if (isnan(y)) return (uint8_t)(sign | 0x7);  /* out of contract: saturate */
  if (a >= 6.0f) return (uint8_t)(sign | 0x7);
  int lo = 0;
  while (lo < 7 && e2m1_mag(lo + 1) <= a) lo++;
  if (e2m1_mag(lo) == a) return (uint8_t)(sign | lo);
  int hi = lo + 1;
  float mid = 0.5f * (e2m1_mag(lo) + e2m1_mag(hi)); /* exact: grid has 3 bits */
  int pick;
  if (a < mid) pick = lo;
  else if (a > mid) pick = hi;
  else pick = ((lo & 1) == 0) ? lo : hi;            /* tie: even mantissa */
  return (uint8_t)(sign | pick);
}

/* Stochastic rounding onto the E2M1 grid (bullet 5: gradients).  lo/hi are
 * the grid neighbours of |y|; the value rounds up iff rbits < floor(frac *
 * 2^32), frac = (|y| - lo) / (hi - lo).  |y| >= 6 saturates to 6; grid
 * points never move.  frac is exact in binary32 because hi - lo is a power
 * of two and |y| - lo is exact (lo <= |y| < 2 lo, or lo == 0). */
uint8_t orc_e2m1_sr(float y, uint32_t rbits) {
  uint8_t sign = signbit(y) ? 0x8 : 0x0;
  float a = fabsf(y);
  if (isnan(y)) return (uint8_t)(sign | 0x7);
  if (a >= 6.0f) return (uint8_t)(sign | 0x7);
  int lo = 0;
  while (lo < 7 && e2m1_mag(lo + 1) <= a) lo++;
  float flo = e2m1_mag(lo);
  if (flo == a) return (uint8_t)(sign | lo);
  float fhi = e2m1_mag(lo + 1);
  float frac = (a - flo) / (fhi - flo);
  double thr = floor((double)frac * 4294967296.0);  /* exact: frac has 24 bits */
  int up = (double)rbits < thr;
  return (uint8_t)(sign | (up ? lo + 1 : lo));
}

/* ======================================================================== */
/* E4M3 ("NVFP4 pretraining recipe", bullet 2: E4M3 block scale factors;
 * bullet 4: "FP8 scale").  Reading: the FN variant -- bias 7, no infinity,
 * 0x7F/0xFF are NaN, largest finite 448, smallest subnormal 2^-9.          */
/* ======================================================================== */
float orc_e4m3_value(uint8_t code) {
  int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  float mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) mag = ldexpf((float)m, -9);
  else        mag = ldexpf(1.0f + (float)m / 8.0f, e - 7);
  return s ? -mag : mag;
}

/* Round-to-nearest-even to E4M3FN, saturating finite values above 448 (and
 * infinities) to 448. */
uint8_t orc_e4m3_rne_sat(float t) {
  uint8_t sign = signbit(t) ? 0x80 : 0x00;
  if (isnan(t)) return 0x7F;
  double a = fabs((double)t);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  if (a < ldexp(1.0, -6)) {                      /* subnormal range: step 2^-9 */
    double n = rint(a * 512.0);                  /* ties to even; 8 -> 2^-6    */
    return (uint8_t)(sign | (int)n);
  }
  int e2;
  double m = frexp(a, &e2);      /* a = m 2^e2, m in [0.5, 1) */
  int e = e2 - 1;                /* a = (2m) 2^e, 2m in [1, 2) */
  double q = rint((2.0 * m - 1.0) * 8.0);        /* mantissa, ties to even   */
  if (q == 8.0) { q = 0.0; e += 1; }
  int code = ((e + 7) << 3) | (int)q;
  if (code > 0x7E) code = 0x7E;                  /* cannot happen below 448 */
  return (uint8_t)(sign | code);
}

/* ======================================================================== */
/* BF16 (outputs of the three GEMMs are BF16: Figure 1 text).               */
/* ======================================================================== */
float orc_bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* Round a double directly to the nearest bf16 (ties to even), no double
 * rounding through binary32.  Overflow gives infinity. */
uint16_t orc_bf16_from_double(double x) {
  if (isnan(x)) return 0x7FC0;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (a == 0.0) return sign;
  int e2;
  frexp(a, &e2);                  /* a in [2^(e2-1), 2^e2) */
  int lsb_exp = (e2 - 1) - 7;     /* 8 significant bits    */
  if (lsb_exp < -133) lsb_exp = -133;  /* bf16 subnormal spacing */
  double q = rint(ldexp(a, -lsb_exp));
  double r = ldexp(q, lsb_exp);
  if (r > 3.3895313892515355e38) return (uint16_t)(sign | 0x7F80); /* inf */
  float rf = (float)r;            /* exact: r has <= 8 significant bits */
  uint32_t u;
  memcpy(&u, &rf, 4);
  return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

void orc_bf16_round_array(const double* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_from_double(x[i]);
}

/* ======================================================================== */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
 * easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies with the
 * published multipliers, key bumped by the Weyl constants between rounds.   */
/* ======================================================================== */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
    uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Stochastic-rounding bits of the element with linear index idx in the
 * quantised operand's logical output layout.  key = seed; counter =
 * (idx/4 low, idx/4 high, stream 0, offset low); word idx%4. */
uint32_t orc_sr_word(uint64_t seed, uint64_t offset, uint64_t idx) {
  uint64_t g = idx >> 2;
  uint32_t ctr[4] = {(uint32_t)g, (uint32_t)(g >> 32), 0u, (uint32_t)offset};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  orc_philox4x32_10(ctr, key, out);
  return out[idx & 3];
}

/* The 16 random signs of the Hadamard transform: key = seed, counter =
 * (0, 0, stream 1, 0); sign i is -1 when bit i of word 0 is set.  One sign
 * vector per seed, shared by both operands of a WGRAD GEMM. */
void orc_rht_signs(uint64_t seed, float signs[16]) {
  uint32_t ctr[4] = {0u, 0u, 1u, 0u};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  orc_philox4x32_10(ctr, key, out);
  for (int i = 0; i < 16; ++i) signs[i] = ((out[0] >> i) & 1u) ? -1.0f : 1.0f;
}

/* ======================================================================== */
/* Random Hadamard transform ("NVFP4 pretraining recipe", bullet 3).
 * v <- (1/4) H16 D v with H16[i][j] = (-1)^popcount(i & j) (Sylvester order)
 * and D = diag(signs).  Evaluated as: signs first, then the butterfly stages
 * h = 1, 2, 4, 8 with (v_i, v_{i+h}) <- (v_i + v_{i+h}, v_i - v_{i+h}) for
 * every i with (i & h) == 0, then a multiply by 0.25.                      */
/* ======================================================================== */
void orc_rht16(float v[16], const float signs[16]) {
  for (int i = 0; i < 16; ++i) v[i] = v[i] * signs[i];
  for (int h = 1; h < 16; h <<= 1) {
    for (int i = 0; i < 16; ++i) {
      if ((i & h) == 0) {
        float a = v[i], b = v[i + h];
        v[i] = a + b;
        v[i + h] = a - b;
      }
    }
  }
  for (int i = 0; i < 16; ++i) v[i] = v[i] * 0.25f;
}

/* ======================================================================== */
/* Quantiser                                                                */
/* ======================================================================== */
void orc_out_shape(int mode, int64_t rows, int64_t cols, int64_t* orows, int64_t* ocols) {
  if (mode == ORC_COL_1X16) { *orows = cols; *ocols = rows; }
  else                      { *orows = rows; *ocols = cols; }
}

/* Scale-factor layout read by the block-scaled MMA: atoms of 128 rows x 4
 * scale columns (512 bytes); inside an atom row r, column c sits at
 * (r % 32) * 16 + ((r / 32) % 4) * 4 + c % 4; atoms are ordered row-block
 * major.  Rows pad to 128 and scale columns to 4 with zero bytes. */
int64_t orc_swizzled_bytes(int64_t orows, int64_t ocols) {
  int64_t nsc = ocols / 16;
  int64_t prow = (orows + 127) / 128 * 128;
  int64_t pcol = (nsc + 3) / 4 * 4;
  return prow * pcol;
}

int64_t orc_swizzle_offset(int64_t r, int64_t c, int64_t ocols) {
  int64_t nsc = ocols / 16;
  int64_t atoms_per_row = (nsc + 3) / 4;
  int64_t atom = (r / 128) * atoms_per_row + c / 4;
  return atom * 512 + (r % 32) * 16 + ((r / 32) % 4) * 4 + (c % 4);
}

static float load_in(const void* x, int in_dtype, int64_t idx) {
  if (in_dtype == ORC_IN_BF16) return orc_bf16_value(((const uint16_t*)x)[idx]);
  return ((const float*)x)[idx];
}

/* Widen the input to binary32 in the operand's logical output layout
 * [orows][ocols] (COL_1X16 transposes), then apply the RHT along each
 * 16-element block if asked. */
static float* load_operand(const void* x, int in_dtype, int64_t rows, int64_t cols, int64_t ld,
                           int mode, uint32_t flags, uint64_t seed) {
  int64_t orows, ocols;
  orc_out_shape(mode, rows, cols, &orows, &ocols);
  float* v = (float*)malloc(sizeof(float) * (size_t)(orows * ocols > 0 ? orows * ocols : 1));
  if (!v) return NULL;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      float f = load_in(x, in_dtype, r * ld + c);
      if (mode == ORC_COL_1X16) v[c * ocols + r] = f;
      else                      v[r * ocols + c] = f;
    }
  if ((flags & ORC_RHT) && mode != ORC_BLOCK_16X16) {
    float signs[16];
    orc_rht_signs(seed, signs);
    for (int64_t r = 0; r < orows; ++r)
      for (int64_t b = 0; b < ocols / 16; ++b) orc_rht16(v + r * ocols + b * 16, signs);
  }
  return v;
}

static int check_args(int in_dtype, int64_t rows, int64_t cols, int64_t ld, int mode,
                      uint32_t flags) {
  if (in_dtype != ORC_IN_BF16 && in_dtype != ORC_IN_FP32) return 1;
  if (rows < 0 || cols < 0 || ld < cols) return 1;
  if (mode < 0 || mode > 2) return 1;
  if (mode == ORC_ROW_1X16 && cols % 16) return 1;
  if (mode == ORC_COL_1X16 && rows % 16) return 1;
  if (mode == ORC_BLOCK_16X16 && ((rows % 16) || (cols % 16) || (flags & ORC_RHT))) return 1;
  if ((flags & ORC_EMIT_T) && mode != ORC_BLOCK_16X16) return 1;
  return 0;
}

static float amax_of(const float* v, int64_t n) {
  float m = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float a = fabsf(v[i]);
    if (a > m) m = a;
  }
  return m;
}

float orc_amax(const void* x, int in_dtype, int64_t rows, int64_t cols, int64_t ld,
               int mode, uint32_t flags, uint64_t seed) {
  if (check_args(in_dtype, rows, cols, ld, mode, flags)) return NAN;
  float* v = load_operand(x, in_dtype, rows, cols, ld, mode, flags, seed);
  if (!v) return NAN;
  float m = amax_of(v, rows * cols);
  free(v);
  return m;
}

/* Per-tensor scale (bullet 2: the FP32 scale beneath the E4M3 block
 * scales).  Reading: map the tensor amax onto the top of the two-level range,
 * s_enc = (6 * 448) / amax; amax == 0 gives 1; a non-finite quotient gives
 * FLT_MAX.  s_dec = 1 / s_enc. */
static float per_tensor_s_enc(float amax) {
  if (amax == 0.0f) return 1.0f;
  float s = 2688.0f / amax;
  if (!isfinite(s)) s = FLT_MAX;
  return s;
}

/* Block scale (bullets 1, 2, 4): S_b = E4M3_rne_sat((a_b / 6) * s_enc). */
static uint8_t block_scale(float a_b, float s_enc) {
  float t = (a_b / 6.0f) * s_enc;
  return orc_e4m3_rne_sat(t);
}

/* Element encode factor: s_enc / S_b, or 0 for a zero block scale. */
static float encode_factor(uint8_t scale_code, float s_enc) {
  float S = orc_e4m3_value(scale_code);
  return (S == 0.0f) ? 0.0f : s_enc / S;
}

static void put_code(uint8_t* row, int64_t j, uint8_t code) {
  if ((j & 1) == 0) row[j / 2] = (uint8_t)((row[j / 2] & 0xF0) | (code & 0xF));
  else              row[j / 2] = (uint8_t)((row[j / 2] & 0x0F) | ((code & 0xF) << 4));
}

static void swizzle_scales(const uint8_t* rm, int64_t orows, int64_t ocols, uint8_t* sw) {
  memset(sw, 0, (size_t)orc_swizzled_bytes(orows, ocols));
  int64_t nsc = ocols / 16;
  for (int64_t r = 0; r < orows; ++r)
    for (int64_t c = 0; c < nsc; ++c) sw[orc_swizzle_offset(r, c, ocols)] = rm[r * nsc + c];
}

int orc_quantize(const void* x, int in_dtype, int64_t rows, int64_t cols, int64_t ld,
                 int mode, uint32_t flags, uint64_t seed, uint64_t offset,
                 float amax_given, orc_qout* out) {
  return orc_quantize_window(x, in_dtype, rows, cols, ld, mode, flags, seed, offset, amax_given,
                             0, out);
}

int orc_quantize_window(const void* x, int in_dtype, int64_t rows, int64_t cols, int64_t ld,
                        int mode, uint32_t flags, uint64_t seed, uint64_t offset,
                        float amax_given, uint64_t sr_index_base, orc_qout* out) {
  if (check_args(in_dtype, rows, cols, ld, mode, flags)) return 1;
  if (!out || !out->codes || !out->scales) return 1;
  if ((flags & ORC_EMIT_T) && (!out->codes_t || !out->scales_t)) return 1;
  int64_t orows, ocols;
  orc_out_shape(mode, rows, cols, &orows, &ocols);

  /* steps 1-2: widen (and transpose for COL_1X16), RHT along the blocks */
  float* v = load_operand(x, in_dtype, rows, cols, ld, mode, flags, seed);
  if (!v) return 2;

  /* steps 3-4: tensor amax and per-tensor scales */
  float amax = (flags & ORC_AMAX_GIVEN) ? amax_given : amax_of(v, orows * ocols);
  float s_enc = per_tensor_s_enc(amax);
  float s_dec = 1.0f / s_enc;
  out->amax = amax;
  out->s_enc = s_enc;
  out->s_dec = s_dec;

  int64_t nsc = ocols / 16;
  memset(out->codes, 0, (size_t)(orows * ocols / 2));

  /* step 5: block scales -- one per 1x16 block, or one per 16x16 tile
   * broadcast to each of the tile's rows (and columns of the transpose) */
  if (mode == ORC_BLOCK_16X16) {
    for (int64_t tr = 0; tr < orows / 16; ++tr)
      for (int64_t tc = 0; tc < nsc; ++tc) {
        float a_b = 0.0f;
        for (int64_t i = 0; i < 16; ++i)
          for (int64_t j = 0; j < 16; ++j) {
            float a = fabsf(v[(tr * 16 + i) * ocols + tc * 16 + j]);
            if (a > a_b) a_b = a;
          }
        uint8_t sc = block_scale(a_b, s_enc);
        for (int64_t i = 0; i < 16; ++i) out->scales[(tr * 16 + i) * nsc + tc] = sc;
        if (flags & ORC_EMIT_T)
          for (int64_t j = 0; j < 16; ++j)
            out->scales_t[(tc * 16 + j) * (orows / 16) + tr] = sc;
      }
  } else {
    for (int64_t r = 0; r < orows; ++r)
      for (int64_t b = 0; b < nsc; ++b)
        out->scales[r * nsc + b] = block_scale(amax_of(v + r * ocols + b * 16, 16), s_enc);
  }

  /* steps 6-8: encode each element with its block's factor, pack */
  if (flags & ORC_EMIT_T) memset(out->codes_t, 0, (size_t)(orows * ocols / 2));
  for (int64_t r = 0; r < orows; ++r) {
    for (int64_t c = 0; c < ocols; ++c) {
      float enc = encode_factor(out->scales[r * nsc + c / 16], s_enc);
      float y = v[r * ocols + c] * enc;
      uint8_t code;
      if (flags & ORC_SR) code = orc_e2m1_sr(y, orc_sr_word(seed, offset, sr_index_base + (uint64_t)(r * ocols + c)));
      else                code = orc_e2m1_rne(y);
      put_code(out->codes + r * (ocols / 2), c, code);
      if (flags & ORC_EMIT_T) put_code(out->codes_t + c * (orows / 2), r, code);
    }
  }

  /* step 9: scales in the MMA layout */
  if (out->scales_sw) swizzle_scales(out->scales, orows, ocols, out->scales_sw);
  if ((flags & ORC_EMIT_T) && out->scales_t_sw)
    swizzle_scales(out->scales_t, ocols, orows, out->scales_t_sw);
  free(v);
  return 0;
}

/* ======================================================================== */
/* Dequantise and FP64 GEMM (Figure 1 text: the GEMMs consume NVFP4 inputs).
 * deq = e2m1(code) * S_b * s_dec, all in FP64 (exact).                     */
/* ======================================================================== */
static double deq_elem(const uint8_t* codes, const uint8_t* scales, double s_dec,
                       int64_t r, int64_t c, int64_t cols) {
  uint8_t byte = codes[r * (cols / 2) + c / 2];
  uint8_t code = (c & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 0xF);
  double S = (double)orc_e4m3_value(scales[r * (cols / 16) + c / 16]);
  return (double)orc_e2m1_value(code) * S * s_dec;
}

void orc_dequant(const uint8_t* codes, const uint8_t* scales, float s_dec,
                 int64_t rows, int64_t cols, double* out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c)
      out[r * cols + c] = deq_elem(codes, scales, (double)s_dec, r, c, cols);
}

/* out[m][n] = sum_k deqA[m][k] * deqB[n][k] in FP64 (both operands K-major). */
void orc_gemm_fp64(const uint8_t* codes_a, const uint8_t* scales_a, float s_dec_a,
                   const uint8_t* codes_b, const uint8_t* scales_b, float s_dec_b,
                   int64_t M, int64_t N, int64_t K, double* out) {
  double* a = (double*)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
  double* b = (double*)malloc(sizeof(double) * (size_t)(N * K > 0 ? N * K : 1));
  if (!a || !b) { free(a); free(b); return; }
  orc_dequant(codes_a, scales_a, s_dec_a, M, K, a);
  orc_dequant(codes_b, scales_b, s_dec_b, N, K, b);
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k) acc += a[m * K + k] * b[n * K + k];
      out[m * N + n] = acc;
    }
  free(a);
  free(b);
}

void orc_gemm_fp64_sampled(const uint8_t* codes_a, const uint8_t* scales_a, float s_dec_a,
                           const uint8_t* codes_b, const uint8_t* scales_b, float s_dec_b,
                           int64_t K, const int64_t* m_idx, const int64_t* n_idx,
                           int64_t n_samples, double* out) {
  for (int64_t s = 0; s < n_samples; ++s) {
    double acc = 0.0;
    for (int64_t k = 0; k < K; ++k)
      acc += deq_elem(codes_a, scales_a, (double)s_dec_a, m_idx[s], k, K) *
             deq_elem(codes_b, scales_b, (double)s_dec_b, n_idx[s], k, K);
    out[s] = acc;
  }
}

/* ======================================================================== */
/* SwiGLU between the MLP GEMMs (the MLP is the part of the block the
 * recipe quantises: Figure 1 text).  h = silu(g) * u, silu(g) = g *
 * sigmoid(g), evaluated in FP64 and rounded once to bf16.                  */
/* ======================================================================== */
static double sigmoid_d(double g) { return 1.0 / (1.0 + exp(-g)); }

void orc_swiglu_fwd(const uint16_t* g, const uint16_t* u, int64_t n, uint16_t* h) {
  for (int64_t i = 0; i < n; ++i) {
    double gv = (double)orc_bf16_value(g[i]), uv = (double)orc_bf16_value(u[i]);
    h[i] = orc_bf16_from_double(gv * sigmoid_d(gv) * uv);
  }
}

/* dU = dH * silu(g);  dG = dH * u * sigmoid(g) * (1 + g * (1 - sigmoid(g))). */
void orc_swiglu_bwd(const uint16_t* dh, const uint16_t* g, const uint16_t* u, int64_t n,
                    uint16_t* dg, uint16_t* du) {
  for (int64_t i = 0; i < n; ++i) {
    double d = (double)orc_bf16_value(dh[i]);
    double gv = (double)orc_bf16_value(g[i]), uv = (double)orc_bf16_value(u[i]);
    double s = sigmoid_d(gv);
    du[i] = orc_bf16_from_double(d * gv * s);
    dg[i] = orc_bf16_from_double(d * uv * s * (1.0 + gv * (1.0 - s)));
  }
}

/* ======================================================================== */
/* MX comparison formats ("NVFP4 pretraining recipe" page, "NVFP4 format
 * and advantages": MXFP4 takes 32-element blocks and power-of-two E8M0
 * scales, against NVFP4's 16-element E4M3 blocks; the Triton-on-Blackwell
 * quote: MXFP8 and MXFP4 block-scaled GEMMs).  The pages link the OCP
 * Microscaling specification for the formats; its conversion is restated
 * here: the block's shared exponent is floor(log2(amax)) minus the largest
 * normal exponent of the element format (2 for E2M1, 8 for E4M3), clamped
 * to the E8M0 range [-127, 127]; each element is v / 2^shared rounded to
 * nearest-even and saturated to the element format's largest finite value.
 * Readings (the spec leaves them to the implementation): an all-zero block
 * gets scale byte 0 and zero codes; a block whose amax is not finite gets
 * scale byte 0xFF (the E8M0 NaN) and zero codes; negative values that round
 * to zero keep their sign (E2M1 code 0x8, E4M3 byte 0x80).                 */
/* ======================================================================== */
float orc_e8m0_value(uint8_t b) {
  if (b == 0xFF) return NAN;
  return ldexpf(1.0f, (int)b - 127);
}

/* floor(log2(a)) of a positive finite float, from frexp (exact). */
static int floor_log2f(float a) {
  int e;
  (void)frexpf(a, &e);  /* a = m 2^e, m in [0.5, 1) */
  return e - 1;
}

uint8_t orc_e8m0_scale(float amax, int fmt) {
  if (!isfinite(amax)) return 0xFF;
  if (amax == 0.0f) return 0;
  const int emax = fmt == ORC_MXFP8 ? 8 : 2;
  int shared = floor_log2f(amax) - emax;
  if (shared < -127) shared = -127;
  if (shared > 127) shared = 127;
  return (uint8_t)(shared + 127);
}

void orc_mx_out_shape(int mode, int64_t rows, int64_t cols, int64_t* orows, int64_t* ocols) {
  orc_out_shape(mode == ORC_MX_COL ? ORC_COL_1X16 : ORC_ROW_1X16, rows, cols, orows, ocols);
}

int orc_mx_quantize(const void* x, int in_dtype, int64_t rows, int64_t cols, int64_t ld,
                    int mode, int fmt, uint8_t* codes, uint8_t* scales) {
  if ((in_dtype != ORC_IN_BF16 && in_dtype != ORC_IN_FP32) || rows <= 0 || cols <= 0 ||
      ld < cols || (mode != ORC_MX_ROW && mode != ORC_MX_COL) ||
      (fmt != ORC_MXFP4 && fmt != ORC_MXFP8))
    return 1;
  if ((mode == ORC_MX_ROW && cols % 32) || (mode == ORC_MX_COL && rows % 32)) return 1;
  int64_t orows, ocols;
  orc_mx_out_shape(mode, rows, cols, &orows, &ocols);
  const int64_t cbytes = fmt == ORC_MXFP4 ? ocols / 2 : ocols;
  float v[32];
  for (int64_t r = 0; r < orows; ++r) {
    for (int64_t b = 0; b < ocols / 32; ++b) {
      float a = 0.0f;
      int nonfinite = 0;
      for (int i = 0; i < 32; ++i) {
        const int64_t c = b * 32 + i;   /* output column */
        const int64_t idx = mode == ORC_MX_ROW ? r * ld + c : c * ld + r;
        v[i] = load_in(x, in_dtype, idx);
        if (!isfinite(v[i])) nonfinite = 1;
        else if (fabsf(v[i]) > a) a = fabsf(v[i]);
      }
      const uint8_t sb = orc_e8m0_scale(nonfinite ? INFINITY : a, fmt);
      scales[r * (ocols / 32) + b] = sb;
      uint8_t* row = codes + r * cbytes;
      for (int i = 0; i < 32; ++i) {
        const int64_t c = b * 32 + i;
        uint8_t code = 0;
        if (sb != 0xFF && a != 0.0f) {
          /* v / 2^shared: exact in FP64, then to float (only values far below
           * the element format's smallest step can round there) */
          const float y = (float)ldexp((double)v[i], -((int)sb - 127));
          code = fmt == ORC_MXFP4 ? orc_e2m1_rne(y) : orc_e4m3_rne_sat(y);
        } else if (sb != 0xFF && signbit(v[i])) {
          code = fmt == ORC_MXFP4 ? 0x8 : 0x80;  /* -0 in an all-zero block */
        }
        if (fmt == ORC_MXFP4) put_code(row, c, code);
        else row[c] = code;
      }
    }
  }
  return 0;
}

void orc_mx_dequant(const uint8_t* codes, const uint8_t* scales, int fmt, int64_t rows,
                    int64_t cols, double* out) {
  const int64_t cbytes = fmt == ORC_MXFP4 ? cols / 2 : cols;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      const uint8_t sb = scales[r * (cols / 32) + c / 32];
      double e;
      if (fmt == ORC_MXFP4) {
        const uint8_t byte = codes[r * cbytes + c / 2];
        e = orc_e2m1_value((uint8_t)((c & 1) ? byte >> 4 : byte & 15));
      } else {
        e = orc_e4m3_value(codes[r * cbytes + c]);
      }
      out[r * cols + c] = e * (double)orc_e8m0_value(sb);
    }
}
