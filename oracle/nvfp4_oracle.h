/*
 * nvfp4_oracle.h -- plain, slow, single-threaded CPU oracle for the NVFP4
 * linear-layer hot path (quantisers, FP64 GEMM, SwiGLU).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this code: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no source, header, table or helper with the
 * CUDA library, and it never reads a value produced by the CUDA library.
 *
 * Source: "NVFP4 pretraining recipe" page (re-post of NVIDIA's blog on the
 * NVFP4 recipe in TransformerEngine / MaxText), sections "NVFP4 format and
 * advantages" and "NVFP4 pretraining recipe" (its five bullets and the
 * Figure 1 data-flow text).  Where that page is silent the readings are the
 * ones listed in the repository's design notes; each function below names its
 * passage and, where applicable, the reading it takes.
 *
 * Arithmetic: IEEE binary32 with round-to-nearest-even unless a function says
 * FP64; no FMA contraction (build with -ffp-contract=off); each expression is
 * evaluated in the order written.
 */
#ifndef NVFP4_ORACLE_H
#define NVFP4_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Modes and flags of the oracle quantiser (same meaning as the library's). */
enum { ORC_ROW_1X16 = 0, ORC_COL_1X16 = 1, ORC_BLOCK_16X16 = 2 };
enum { ORC_RHT = 1, ORC_SR = 2, ORC_EMIT_T = 4, ORC_AMAX_GIVEN = 8 };
enum { ORC_IN_BF16 = 0, ORC_IN_FP32 = 1 };

/* ---- element formats ---------------------------------------------------- */
float   orc_e2m1_value(uint8_t code);          /* 4-bit code -> value        */
uint8_t orc_e2m1_rne(float y);                 /* nearest, ties to even code */
uint8_t orc_e2m1_sr(float y, uint32_t rbits);  /* stochastic rounding        */
float   orc_e4m3_value(uint8_t code);          /* E4M3FN byte -> value       */
uint8_t orc_e4m3_rne_sat(float t);             /* RNE + saturate to 448      */
uint16_t orc_bf16_from_double(double x);       /* RNE double -> bf16 bits    */
float   orc_bf16_value(uint16_t b);
void    orc_bf16_round_array(const double* x, int64_t n, uint16_t* out);

/* ---- counter-based RNG (Philox4x32-10, Salmon et al., SC'11) ------------ */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
uint32_t orc_sr_word(uint64_t seed, uint64_t offset, uint64_t idx);
void orc_rht_signs(uint64_t seed, float signs[16]);

/* ---- 16-point random Hadamard transform --------------------------------- */
void orc_rht16(float v[16], const float signs[16]);

/* ---- quantiser ----------------------------------------------------------- */
typedef struct {
  uint8_t* codes;        /* [orows][ocols/2] packed, element 2i in low nibble */
  uint8_t* scales;       /* [orows][ocols/16] row-major E4M3                  */
  uint8_t* scales_sw;    /* swizzled + padded (may be NULL)                   */
  uint8_t* codes_t;      /* 16x16 + EMIT_T: [ocols][orows/2]   (else NULL)    */
  uint8_t* scales_t;     /* 16x16 + EMIT_T: [ocols][orows/16]  (else NULL)    */
  uint8_t* scales_t_sw;  /* swizzled transposed scales (may be NULL)          */
  float amax;            /* out: amax used                                    */
  float s_enc;           /* out: per-tensor encode scale                      */
  float s_dec;           /* out: per-tensor decode scale                      */
} orc_qout;

/* Logical output shape of the quantised operand. */
void orc_out_shape(int mode, int64_t rows, int64_t cols, int64_t* orows, int64_t* ocols);
/* Bytes of a swizzled, padded scale tensor for an operand [orows][ocols]. */
int64_t orc_swizzled_bytes(int64_t orows, int64_t ocols);
int64_t orc_swizzle_offset(int64_t r, int64_t c, int64_t ocols);

/* Returns 0 on success, nonzero on an invalid argument. */
int orc_quantize(const void* x, int in_dtype, int64_t rows, int64_t cols, int64_t ld,
                 int mode, uint32_t flags, uint64_t seed, uint64_t offset,
                 float amax_given, orc_qout* out);

/* orc_quantize of a window of output rows of a larger operand: x holds the
 * window alone, and every element's stochastic-rounding index is its index in
 * the whole operand's output, i.e. its index in the window plus sr_index_base
 * (= first output row of the window * output columns).  Same arithmetic;
 * orc_quantize is this with sr_index_base = 0. */
int orc_quantize_window(const void* x, int in_dtype, int64_t rows, int64_t cols, int64_t ld,
                        int mode, uint32_t flags, uint64_t seed, uint64_t offset,
                        float amax_given, uint64_t sr_index_base, orc_qout* out);

/* Amax of the (optionally RHT'd) operand, as the quantiser computes it. */
float orc_amax(const void* x, int in_dtype, int64_t rows, int64_t cols, int64_t ld,
               int mode, uint32_t flags, uint64_t seed);

/* ---- dequantise and FP64 GEMM ------------------------------------------- */
void orc_dequant(const uint8_t* codes, const uint8_t* scales, float s_dec,
                 int64_t rows, int64_t cols, double* out);
void orc_gemm_fp64(const uint8_t* codes_a, const uint8_t* scales_a, float s_dec_a,
                   const uint8_t* codes_b, const uint8_t* scales_b, float s_dec_b,
                   int64_t M, int64_t N, int64_t K, double* out);
void orc_gemm_fp64_sampled(const uint8_t* codes_a, const uint8_t* scales_a, float s_dec_a,
                           const uint8_t* codes_b, const uint8_t* scales_b, float s_dec_b,
                           int64_t K, const int64_t* m_idx, const int64_t* n_idx,
                           int64_t n_samples, double* out);

/* ---- MX comparison formats (OCP Microscaling): 32-element blocks, E8M0 -- */
enum { ORC_MXFP4 = 0, ORC_MXFP8 = 1 };
enum { ORC_MX_ROW = 0, ORC_MX_COL = 1 };  /* blocks along the output's rows  */
float   orc_e8m0_value(uint8_t b);               /* 2^(b-127); 0xFF is NaN    */
uint8_t orc_e8m0_scale(float amax, int fmt);     /* a block's scale byte      */
void    orc_mx_out_shape(int mode, int64_t rows, int64_t cols, int64_t* orows, int64_t* ocols);
/* codes: MXFP4 [orows][ocols/2] packed like NVFP4, MXFP8 [orows][ocols] E4M3;
 * scales: [orows][ocols/32] E8M0, row-major.  Returns 0, or nonzero on an
 * invalid argument (the blocked dimension must be a multiple of 32). */
int  orc_mx_quantize(const void* x, int in_dtype, int64_t rows, int64_t cols, int64_t ld,
                     int mode, int fmt, uint8_t* codes, uint8_t* scales);
void orc_mx_dequant(const uint8_t* codes, const uint8_t* scales, int fmt, int64_t rows,
                    int64_t cols, double* out);

/* ---- SwiGLU (between the MLP GEMMs) -------------------------------------- */
void orc_swiglu_fwd(const uint16_t* g, const uint16_t* u, int64_t n, uint16_t* h);
void orc_swiglu_bwd(const uint16_t* dh, const uint16_t* g, const uint16_t* u, int64_t n,
                    uint16_t* dg, uint16_t* du);

#ifdef __cplusplus
}
#endif
#endif
