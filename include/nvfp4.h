/*
 * nvfp4.h -- C ABI of libnvfp4.so: NVFP4 quantisers and block-scaled GEMMs
 * for one GB300 (sm_103a), the hot path of an NVFP4 linear / MLP layer.
 *
 * The method is the NVFP4 pretraining recipe of the "NVFP4 pretraining
 * recipe" page (re-post of NVIDIA's blog on NVFP4 in TransformerEngine and
 * MaxText).  Each entry point below cites the passage of that page that
 * defines what it computes.
 *
 * Conventions shared by every entry point
 *  - Pointers named "device" are CUDA device pointers on the current device;
 *    host pointers are marked "host".  The caller owns every buffer, including
 *    workspaces and the per-tensor scalars; the library never allocates,
 *    frees or synchronises on the hot path (nvfp4_check_device_errors is the
 *    one call that synchronises).
 *  - All work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream).  Nothing on the hot path allocates or
 *    synchronises, so a sequence of calls can be captured into a CUDA graph
 *    and replayed (after one uncaptured call of each, which configures the
 *    kernels).  The quantiser, amax and GEMM kernels are launched with
 *    programmatic stream serialization: a kernel may be scheduled while the
 *    previous one on the stream finishes, and waits for it to complete before
 *    it touches global memory, so stream order is kept.
 *  - Argument errors are reported by the return value before anything is
 *    launched; a failed launch returns NVFP4_ERR_CUDA.  Device-side wait
 *    timeouts (a hung pipeline) are recorded in a device error word and
 *    reported by nvfp4_check_device_errors.
 *  - Matrices are row-major.  A "K-major" NVFP4 operand [rows, K] stores the
 *    E2M1 codes of row r in bytes r*K/2 .. r*K/2 + K/2 - 1, element 2i in the
 *    low nibble and element 2i+1 in the high nibble.
 *  - Scale tensors (E4M3, one byte per 16 elements) are stored in the layout
 *    the block-scaled MMA reads: 512-byte atoms of 128 rows x 4 scale
 *    columns, the byte of (row r, scale column c) at
 *        atom(r/128, c/4) * 512 + (r%32)*16 + ((r/32)%4)*4 + c%4,
 *    atoms row-block major, rows padded to 128 and scale columns to 4 with
 *    zero bytes.  Size: pad128(rows) * pad4(cols/16) bytes.
 */
#ifndef NVFP4_H
#define NVFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void* nvfp4_stream; /* a cudaStream_t */

typedef enum {
  NVFP4_OK = 0,
  NVFP4_ERR_INVALID_ARG = 1,    /* null pointer, bad enum or flag combination   */
  NVFP4_ERR_SHAPE = 2,          /* a dimension breaks the rules stated per call */
  NVFP4_ERR_ALIGN = 3,          /* a pointer or leading dimension is misaligned */
  NVFP4_ERR_ARCH = 4,           /* the current device is not sm_103             */
  NVFP4_ERR_WORKSPACE = 5,      /* workspace missing or smaller than required   */
  NVFP4_ERR_CUDA = 6,           /* a CUDA runtime/driver call failed            */
  NVFP4_ERR_DEVICE_TIMEOUT = 7  /* a kernel's bounded wait expired              */
} nvfp4_status;

typedef enum { NVFP4_IN_BF16 = 0, NVFP4_IN_FP32 = 1 } nvfp4_in_dtype;

/* Quantisation geometry ("NVFP4 pretraining recipe", bullets 1 and 4).
 *  ROW_1X16   : 1x16 blocks along the contiguous dim; output [rows, cols].
 *  COL_1X16   : 1x16 blocks along the rows; output is the transpose
 *               [cols, rows] (K-major along the original rows), the form the
 *               WGRAD GEMM consumes.
 *  BLOCK_16X16: one scale per 16x16 tile (weights); output [rows, cols], and
 *               with NVFP4_EMIT_T also the transpose [cols, rows] built from
 *               the same codes (no requantisation). */
typedef enum { NVFP4_ROW_1X16 = 0, NVFP4_COL_1X16 = 1, NVFP4_BLOCK_16X16 = 2 } nvfp4_mode;

enum {
  NVFP4_RHT = 1u,        /* 16-point random Hadamard transform along the blocks (bullet 3) */
  NVFP4_SR = 2u,         /* stochastic rounding of the elements (bullet 5); else RNE       */
  NVFP4_EMIT_T = 4u,     /* BLOCK_16X16 only: also write the transposed operand            */
  NVFP4_AMAX_GIVEN = 8u  /* use *out->amax (device, set by the caller) as the tensor amax   */
};

/* A quantised NVFP4 operand.  The caller fills the pointers; nvfp4_quantize
 * fills rows/cols/mode/flags.  rows x cols is the logical K-major operand
 * (cols = contraction length).
 *   codes    device uint8 [rows][cols/2]
 *   scales   device uint8, MMA layout for [rows, cols]
 *   codes_t  device uint8 [cols][rows/2]     (BLOCK_16X16 + EMIT_T, else NULL)
 *   scales_t device uint8, MMA layout for [cols, rows] (likewise)
 *   amax     device float: tensor amax (output; input with AMAX_GIVEN)
 *   s_dec    device float: per-tensor decode scale 1/s_enc (output)        */
typedef struct nvfp4_tensor {
  void* codes;
  void* scales;
  void* codes_t;
  void* scales_t;
  float* amax;
  float* s_dec;
  int64_t rows;
  int64_t cols;
  int32_t mode;
  uint32_t flags;
} nvfp4_tensor;

/* ---------------------------------------------------------------------- */
/* Status and device                                                       */
/* ---------------------------------------------------------------------- */
const char* nvfp4_status_string(nvfp4_status s);
/* Library version as major*10000 + minor*100 + patch. */
int nvfp4_version(void);
/* NVFP4_OK when `device` is an sm_103 GPU this library's kernels run on. */
nvfp4_status nvfp4_device_check(int device);
/* Synchronises `stream`, then reads and clears the device error word that
 * kernels set when a bounded wait expires.  Returns NVFP4_ERR_DEVICE_TIMEOUT
 * if it was set, NVFP4_ERR_CUDA if the stream reported an error. */
nvfp4_status nvfp4_check_device_errors(nvfp4_stream stream);

/* Failure injection for tests of the bounded waits; the pages have no
 * counterpart (they describe no failure handling).  While a bit of
 * stall_mask is set, the producer of every launch of that kernel family
 * issues no loads, so the consumers' first pipeline wait runs out; nothing is
 * in flight when the kernel gives up, and it returns after recording the
 * timeout (nvfp4_check_device_errors then reports NVFP4_ERR_DEVICE_TIMEOUT):
 *   NVFP4_STALL_QUANTIZE  the quantise passes of nvfp4_quantize
 *   NVFP4_STALL_GEMM      every GEMM kernel (single-SM and CTA-pair tiles;
 *                         on a pair a timeout in either CTA stops both)
 * wait_limit_ns sets how long those kernels' pipeline waits last before they
 * give up (0: the default, 2 s); the waits that drain copies and MMAs
 * already issued keep their own 2 s limit.  Synchronises the device, then
 * applies to later launches until changed; call it with nothing of this
 * library in flight.  Returns NVFP4_ERR_INVALID_ARG for unknown bits,
 * NVFP4_ERR_CUDA if the device cannot be reached. */
enum { NVFP4_STALL_QUANTIZE = 1u, NVFP4_STALL_GEMM = 2u };
nvfp4_status nvfp4_debug_inject(uint32_t stall_mask, uint64_t wait_limit_ns);

/* ---------------------------------------------------------------------- */
/* Quantiser                                                               */
/* ---------------------------------------------------------------------- */
/* Byte sizes for quantising an input x [rows, cols]: the codes (and, with
 * EMIT_T, the same again for codes_t), the MMA-layout scales (scales_t has
 * the size of the transposed operand's scales), and the workspace
 * nvfp4_quantize needs.  Any output pointer may be NULL. */
nvfp4_status nvfp4_quantize_sizes(int64_t rows, int64_t cols, int32_t mode, uint32_t flags,
                                  size_t* codes_bytes, size_t* scales_bytes,
                                  size_t* scales_t_bytes, size_t* workspace_bytes);

/* NVFP4 quantisation of x [rows, cols] (row-major, leading dim ld elements),
 * per "NVFP4 pretraining recipe", bullets 1-5:
 *   amax_T = max |v| over the (RHT-transformed, if NVFP4_RHT) operand v;
 *   s_enc = 6*448 / amax_T (1 if amax_T == 0, FLT_MAX if not finite),
 *   s_dec = 1 / s_enc;
 *   per block b (16 elements, or a 16x16 tile): a_b = max |v|,
 *   S_b = E4M3_rn_satfinite((a_b / 6) * s_enc);
 *   per element: y = v * (S_b == 0 ? 0 : s_enc / S_b), encoded to E2M1 by
 *   round-to-nearest-even with saturation to +-6, or with NVFP4_SR by
 *   stochastic rounding: round |y| up to the next grid value iff
 *   r < floor(frac * 2^32), frac = (|y| - lo) / (hi - lo), where r is word
 *   idx%4 of Philox4x32-10(key = seed, counter = (idx/4 lo, idx/4 hi, 0,
 *   offset lo)) and idx = row*cols + col in the output layout.
 *   NVFP4_RHT (1x16 modes): each block becomes (1/4) H16 diag(s) v, signs s_i
 *   = -1 where bit i of word 0 of Philox(key = seed, counter = (0,0,1,0)) is
 *   set -- one sign vector per seed, so both WGRAD operands quantised with the
 *   same seed share it (bullet 3: RHT on the WGRAD inputs only).
 * Shapes: ROW_1X16 needs cols % 16 == 0; COL_1X16 rows % 16 == 0 and
 * cols % 8 == 0; BLOCK_16X16 rows % 16 == 0, cols % 16 == 0, no NVFP4_RHT.
 * x must be 16-byte aligned and ld * element size a multiple of 16 bytes.
 * The workspace (device, >= the size nvfp4_quantize_sizes gives, 16-byte
 * aligned) holds per-CTA partial maxima; with NVFP4_AMAX_GIVEN it may be NULL.
 * Outputs: out->codes/scales (+ codes_t/scales_t), out->amax, out->s_dec;
 * padding bytes of the scale tensors are written as zero. */
nvfp4_status nvfp4_quantize(const void* x, int32_t in_dtype, int64_t rows, int64_t cols,
                            int64_t ld, int32_t mode, uint32_t flags, uint64_t seed,
                            uint64_t offset, nvfp4_tensor* out, void* workspace,
                            size_t workspace_bytes, nvfp4_stream stream);

/* The per-tensor amax of nvfp4_quantize ("NVFP4 pretraining recipe", bullet
 * 4: amax_T over the operand as quantised) for the two quantisations a
 * training step makes of X and of dY -- the row-wise operand (ROW_1X16, no
 * transform) and the column-wise WGRAD operand (COL_1X16 with NVFP4_RHT) --
 * from one read of x [rows, cols] (leading dim ld, bf16 or fp32):
 *   amax_plain = max |x|                            (if amax_plain != NULL),
 *   amax_rht   = max |(1/4) H16 diag(s) v| over every 16-row block v of every
 *                column, signs s from `seed` as in nvfp4_quantize
 *                                                   (if amax_rht != NULL).
 * Both are device floats; each equals, bit for bit, the amax the matching
 * nvfp4_quantize call computes itself, so passing it with NVFP4_AMAX_GIVEN
 * (out->amax pointing at it) gives identical codes and scales.  At least one
 * output must be non-NULL; amax_rht needs rows % 16 == 0.  x: 16-byte
 * aligned, ld * element size a multiple of 16 bytes, cols % 8 == 0.  The
 * workspace is as for nvfp4_quantize (partial maxima; contents on return
 * unspecified).  Two kernel launches on `stream`; nothing is allocated.
 * Returns NVFP4_ERR_INVALID_ARG, _SHAPE, _ALIGN, _WORKSPACE, _ARCH, _CUDA as
 * nvfp4_quantize does. */
nvfp4_status nvfp4_amax(const void* x, int32_t in_dtype, int64_t rows, int64_t cols, int64_t ld,
                        uint64_t seed, float* amax_plain, float* amax_rht, void* workspace,
                        size_t workspace_bytes, nvfp4_stream stream);

/* Both quantisations a training step makes of one bf16 activation or
 * gradient x [rows, cols] (leading dim ld), from one read of x -- bit for bit
 * what two nvfp4_quantize calls give ("NVFP4 pretraining recipe", bullets
 * 1-5: the FPROP / DGRAD operand is quantised row-wise, the WGRAD operand
 * column-wise with the RHT on the WGRAD inputs only, SR on gradients):
 *   row_out: nvfp4_quantize(x, ROW_1X16, row_flags, seed, row_offset)
 *   col_out: nvfp4_quantize(x, COL_1X16, col_flags, seed, col_offset)
 * row_flags: NVFP4_AMAX_GIVEN, optionally | NVFP4_SR; col_flags:
 * NVFP4_AMAX_GIVEN, optionally | NVFP4_RHT | NVFP4_SR.  Both amaxes are given
 * (*row_out->amax = max |x|, *col_out->amax = the column operand's amax, e.g.
 * both from one nvfp4_amax call), so nothing needs a workspace.  Shapes:
 * rows % 16 == 0, cols % 16 == 0.  x, the codes and scales buffers 16-byte
 * aligned, ld * 2 a multiple of 16; bf16 input only.  One kernel launch on
 * `stream`; nothing is allocated.  Returns NVFP4_ERR_INVALID_ARG (a NULL
 * pointer, fp32 input, a flag outside those above or AMAX_GIVEN missing),
 * _SHAPE, _ALIGN, _ARCH, _CUDA. */
nvfp4_status nvfp4_quantize_rowcol(const void* x, int32_t in_dtype, int64_t rows, int64_t cols,
                                   int64_t ld, uint32_t row_flags, uint32_t col_flags,
                                   uint64_t seed, uint64_t row_offset, uint64_t col_offset,
                                   nvfp4_tensor* row_out, nvfp4_tensor* col_out,
                                   nvfp4_stream stream);

/* nvfp4_quantize without a workspace argument; the pages have no counterpart
 * to this entry point.  It is for callers that cannot provide device scratch
 * memory -- code running during CUDA graph capture (where cudaMalloc is not
 * allowed), plugins given only input and output pointers, or programs whose
 * allocator owns all device memory.  The per-CTA partial maxima of the amax
 * pass go to a fixed 4 KB array (1024 floats) inside the library, held on
 * every GPU that loads the library until the process exits.  The caller still
 * passes x and the output buffers of `out`, exactly as for nvfp4_quantize, and
 * gets the same results.
 * Every call made outside stream capture looks up the array's device address
 * on the current device (after a cudaDeviceReset the array may move); a call
 * made while `stream` is being captured reuses the address the last
 * uncaptured call on that device found, so make the first call on a device
 * before any stream capture.  The call itself allocates and frees nothing.
 * All calls share the one array: calls that can overlap on the GPU
 * (different streams, no ordering between them) race and must not be issued
 * that way.  Each call's amax pass rewrites every partial its quantise pass
 * reads, so nothing needs clearing between calls.  The array holds the
 * partial maxima of the largest amax grid the library launches (1024 CTAs),
 * so every device and shape nvfp4_quantize accepts is accepted; the statuses
 * are those of nvfp4_quantize. */
nvfp4_status nvfp4_quantize_noalloc(const void* x, int32_t in_dtype, int64_t rows, int64_t cols,
                                    int64_t ld, int32_t mode, uint32_t flags, uint64_t seed,
                                    uint64_t offset, nvfp4_tensor* out, nvfp4_stream stream);

/* ---------------------------------------------------------------------- */
/* MX comparison formats                                                   */
/* ---------------------------------------------------------------------- */
/* "NVFP4 pretraining recipe" page, "NVFP4 format and advantages": MXFP4
 * scales 32-element blocks by powers of two (E8M0), against NVFP4's 16-element
 * E4M3 blocks under a per-tensor scale; the same page quotes MXFP8 and MXFP4
 * block-scaled GEMMs on Blackwell.  These quantisers produce those formats
 * for comparison with NVFP4 (error studies), following the OCP Microscaling
 * specification the page links. */
typedef enum { NVFP4_MXFP4 = 0, NVFP4_MXFP8 = 1 } nvfp4_mx_format;
enum {
  NVFP4_MX_ROW = 0,  /* blocks of 32 along the columns; output [rows, cols]            */
  NVFP4_MX_COL = 1   /* blocks of 32 along the rows; output transposed [cols, rows]    */
};

/* Byte sizes of the outputs of nvfp4_mx_quantize for x [rows, cols]:
 * codes = out_rows * out_cols / 2 (MXFP4) or out_rows * out_cols (MXFP8),
 * scales = out_rows * out_cols / 32, scales_sw = the same scales in the MMA
 * layout (512-byte atoms of 128 rows x 4 scale columns, rows padded to 128
 * and scale columns to 4).  Any pointer may be NULL.  Returns
 * NVFP4_ERR_SHAPE unless the blocked dimension is a multiple of 32 (and, for
 * NVFP4_MX_COL, cols a multiple of 8). */
nvfp4_status nvfp4_mx_sizes(int64_t rows, int64_t cols, int32_t mode, int32_t fmt,
                            size_t* codes_bytes, size_t* scales_bytes, size_t* scales_sw_bytes);

/* MXFP4 / MXFP8 quantisation of x [rows, cols] (bf16 or fp32, row-major,
 * leading dim ld elements).  Per block of 32 consecutive output elements:
 *   shared = clamp(floor(log2(amax)) - emax, -127, 127), emax = 2 (E2M1) or
 *            8 (E4M3); scale byte = shared + 127 (E8M0, value 2^shared);
 *            0 when the block is all zero; 0xFF (NaN) when it holds a value
 *            that is not finite, with zero codes;
 *   element = v / 2^shared rounded to nearest-even and saturated to the
 *            element format's largest finite value (6 or 448), sign kept.
 * Outputs (device, caller-owned, sizes from nvfp4_mx_sizes): codes row-major
 * [out_rows][out_cols] -- MXFP4 packed two per byte, element 2i in the low
 * nibble of byte i; MXFP8 one E4M3 byte each -- and scales row-major
 * [out_rows][out_cols / 32], and, if scales_sw is not NULL, the same
 * scale bytes in the MMA layout nvfp4_mx_gemm reads (offset
 * ((r/128) * (padded scale cols / 4) + c/4) * 512 + (r%32)*16 + ((r/32)%4)*4
 * + c%4 for row r, scale column c; padding written as zero).  x and codes
 * must be 16-byte aligned and ld * element size a multiple of 16 bytes.  One
 * kernel launch on `stream` (plus a memset of scales_sw when it has
 * padding); nothing is allocated.  Returns NVFP4_ERR_INVALID_ARG, _SHAPE,
 * _ALIGN, _ARCH, _CUDA. */
nvfp4_status nvfp4_mx_quantize(const void* x, int32_t in_dtype, int64_t rows, int64_t cols,
                               int64_t ld, int32_t mode, int32_t fmt, void* codes, void* scales,
                               void* scales_sw, nvfp4_stream stream);

/* D bf16 [M, N] = A . B^T for MX operands, the comparison GEMMs (the page's
 * quote of MXFP8 and MXFP4 block-scaled GEMMs on Blackwell):
 *   D[m][n] = bf16_rn( sum_k deq(A)[m][k] * deq(B)[n][k] ),
 *   deq = element value * 2^(scale byte - 127) over its 32-element block.
 * A: a_codes [M][K] K-major as nvfp4_mx_quantize writes them (MXFP4: K/2
 * bytes per row, MXFP8: K), a_scales_sw its scales in the MMA layout (the
 * scales_sw output of nvfp4_mx_quantize); B likewise [N][K].  The WGRAD
 * operands are the NVFP4_MX_COL outputs.  Shapes: K % 128 == 0, N % 8 == 0.
 * All pointers device, 16-byte aligned.  One launch (the CTA-pair kernel,
 * tcgen05 kind::mxf4nvf4 scale_vec::2X or kind::mxf8f6f4 scale_vec::1X).
 * Returns NVFP4_ERR_INVALID_ARG, _SHAPE, _ALIGN, _ARCH, _CUDA. */
nvfp4_status nvfp4_mx_gemm(const void* a_codes, const void* a_scales_sw, const void* b_codes,
                           const void* b_scales_sw, int32_t fmt, void* D, int64_t M, int64_t N,
                           int64_t K, nvfp4_stream stream);

/* ---------------------------------------------------------------------- */
/* Block-scaled GEMM                                                       */
/* ---------------------------------------------------------------------- */
/* Output modes of nvfp4_gemm. */
enum {
  NVFP4_D_BF16 = 0,        /* D bf16 [M,N] = bf16(alpha * acc)                            */
  NVFP4_D_F32_ACCUM = 1,   /* D fp32 [M,N] += float(bf16(alpha * acc)) (master gradient)   */
  NVFP4_D_BF16_ADD_C = 2   /* D bf16 [M,N] = bf16(alpha * acc + float(C)), C bf16 [M,N]    */
};

/* D = alpha * A . B^T with A [M, K] and B [N, K] NVFP4 K-major operands and
 * alpha = (*A->s_dec) * (*B->s_dec) read on the device; FP32 accumulation in
 * tensor memory, BF16 output ("NVFP4 pretraining recipe", Figure 1 text:
 * FPROP, DGRAD and WGRAD consume NVFP4 inputs and emit BF16 outputs, later
 * folded into the FP32 master weight -- NVFP4_D_F32_ACCUM).
 * a_view / b_view: 0 reads codes/scales, 1 reads codes_t/scales_t (the
 * transpose written by BLOCK_16X16 + EMIT_T: DGRAD reads W this way, bullet 4).
 * The operand's logical shape must match (rows, cols) = (M, K) / (N, K).
 * Shapes: M, N >= 1, K % 64 == 0, N % 8 == 0.  D (and C) 16-byte aligned.
 * workspace: unused (may be NULL). */
nvfp4_status nvfp4_gemm(const nvfp4_tensor* A, int32_t a_view, const nvfp4_tensor* B,
                        int32_t b_view, void* D, int32_t d_mode, const void* C, int64_t M,
                        int64_t N, int64_t K, void* workspace, size_t workspace_bytes,
                        nvfp4_stream stream);

/* Output-tile configurations of nvfp4_gemm_ex. */
enum {
  NVFP4_TILE_AUTO = 0,          /* 128 x 128 when N <= 128; else the CTA pair when its     *
                                 * 256 x 256 tiles number at least half the SMs (256 x 384 *
                                 * where its rounds of tiles per pair cost less, not with  *
                                 * NVFP4_D_BF16_ADD_C); else 128 x 256 on one SM           */
  NVFP4_TILE_128X128 = 1,       /* one SM per 128 x 128 tile                               */
  NVFP4_TILE_128X256 = 2,       /* one SM per 128 x 256 tile                               */
  NVFP4_TILE_PAIR_256X256 = 3,  /* a cluster of two SMs per 256 x 256 tile (cta_group::2) */
  /* 4 is retired (rejected with NVFP4_ERR_INVALID_ARG)                                    */
  NVFP4_TILE_128X256_K128 = 5,  /* one SM per 128 x 256 tile, 8 stages of K = 128          */
  NVFP4_TILE_PAIR_256X384 = 6   /* a cluster of two SMs per 256 x 384 tile: an N = 256 and *
                                 * an N = 128 MMA per K step, 4 stages; not with           *
                                 * NVFP4_D_BF16_ADD_C (NVFP4_ERR_INVALID_ARG)              */
};

/* As nvfp4_gemm with an explicit output-tile configuration (NVFP4_TILE_*).
 * For tuning and tests; results are identical up to FP32 summation order. */
nvfp4_status nvfp4_gemm_ex(const nvfp4_tensor* A, int32_t a_view, const nvfp4_tensor* B,
                           int32_t b_view, void* D, int32_t d_mode, const void* C, int64_t M,
                           int64_t N, int64_t K, int32_t tile, nvfp4_stream stream);

/* ---------------------------------------------------------------------- */
/* SwiGLU MLP (gate, up, down projections) with NVFP4 GEMMs                */
/* ---------------------------------------------------------------------- */
/* "NVFP4 pretraining recipe", Figure 1 text: the MLP's GEMMs run in NVFP4.
 * Forward: G = X Wg^T, U = X Wu^T, H = silu(G) * U, Y = H Wd^T; backward:
 * dH = dY Wd, dWd += dY^T H, dG/dU from the SwiGLU derivative, dX = dG Wg +
 * dU Wu, dWg += dG^T X, dWu += dU^T X.  Quantisation per operand: X, H and W
 * with RNE (1x16 / 16x16), dY, dG, dU with SR; the WGRAD operands (X^T, H^T,
 * dY^T, dG^T, dU^T) COL_1X16 with the RHT when flags has NVFP4_RHT.
 * Dimensions: M tokens, D hidden, F ffn; Wg, Wu fp32 [F, D], Wd fp32 [D, F]
 * (device, the FP32 master weights, quantised 16x16 every forward).
 * flags: NVFP4_RHT, and NVFP4_AMAX_GIVEN for a forward whose weight amaxes
 * are already in the weight operands' amax slots in `saved`
 * (nvfp4_mlp_operand: Q_WG / Q_WU / Q_WD, .amax), e.g. written there by the
 * previous optimizer step (nvfp4_sgd_step): the three weights are then
 * quantised without their amax passes, with codes and scales identical to a
 * forward that takes the amaxes itself.  The backward ignores
 * NVFP4_AMAX_GIVEN. */
typedef struct nvfp4_mlp_params {
  int64_t M, D, F;
  const float* Wg;
  const float* Wu;
  const float* Wd;
  uint64_t seed;   /* RHT signs and SR key                           */
  uint64_t step;   /* SR counter offsets 8*step + 0..5 (per tensor)  */
  uint32_t flags;  /* NVFP4_RHT | NVFP4_AMAX_GIVEN, or 0             */
} nvfp4_mlp_params;

/* SwiGLU between the gate/up and down projections, with the tensor amaxes of
 * its outputs for the NVFP4 quantisations that follow ("NVFP4 pretraining
 * recipe" page, Figure 1 text and bullets 3-5: each output is quantised
 * row-wise for FPROP / DGRAD and column-wise, with the RHT when enabled, for
 * WGRAD; both need its per-tensor amax).  Computed in FP32 with the CUDA
 * expf, each output rounded once to bf16:
 *   forward   H  = silu(G) * U,               silu(g) = g sigmoid(g)
 *   backward  dU = dH * silu(G),  dG = dH * U * sigmoid(G) (1 + G (1 - sigmoid(G)))
 * All tensors bf16 [rows, cols], contiguous, 16-byte aligned; rows % 16 == 0,
 * cols % 8 == 0.  For each output T the kernel writes two device floats,
 * taken from the bf16 values it stores (no second read of T):
 *   amax_*_row = max |T|, the amax of T's ROW_1X16 quantisation;
 *   amax_*_col = with NVFP4_RHT in flags, max |(1/4) H16 diag(s) v| over every
 *                16-row block v of every column of T, signs s from `seed`
 *                as in nvfp4_quantize; otherwise max |T| again.
 * Each equals, bit for bit, what nvfp4_amax returns for T, so it can be given
 * to nvfp4_quantize with NVFP4_AMAX_GIVEN.  workspace: device scratch of at
 * least nvfp4_swiglu_workspace_bytes(), 16-byte aligned, contents on return
 * unspecified.  Two kernel launches on `stream`; nothing is allocated.
 * Returns NVFP4_ERR_INVALID_ARG (a NULL pointer, unknown flag bits),
 * _SHAPE, _ALIGN, _WORKSPACE, _ARCH, _CUDA. */
size_t nvfp4_swiglu_workspace_bytes(void);
nvfp4_status nvfp4_swiglu_fwd(const void* G, const void* U, void* H, int64_t rows, int64_t cols,
                              uint32_t flags, uint64_t seed, float* amax_h_row,
                              float* amax_h_col, void* workspace, size_t workspace_bytes,
                              nvfp4_stream stream);
nvfp4_status nvfp4_swiglu_bwd(const void* dH, const void* G, const void* U, void* dG, void* dU,
                              int64_t rows, int64_t cols, uint32_t flags, uint64_t seed,
                              float* amax_dg_row, float* amax_dg_col, float* amax_du_row,
                              float* amax_du_col, void* workspace, size_t workspace_bytes,
                              nvfp4_stream stream);

/* Device bytes of the saved-activation buffer (forward -> backward) and of
 * the workspace either call needs. */
nvfp4_status nvfp4_mlp_sizes(int64_t M, int64_t D, int64_t F, size_t* saved_bytes,
                             size_t* workspace_bytes);

/* X bf16 [M, D] -> Y bf16 [M, D]; fills `saved` (device) for the backward.
 * Shapes: M, D, F multiples of 128. */
nvfp4_status nvfp4_mlp_fwd(const nvfp4_mlp_params* p, const void* X, void* Y, void* saved,
                           size_t saved_bytes, void* workspace, size_t workspace_bytes,
                           nvfp4_stream stream);

/* dY bf16 [M, D] -> dX bf16 [M, D]; dWg, dWu fp32 [F, D] and dWd fp32 [D, F]
 * (device) are accumulated: += float(bf16(WGRAD)). */
nvfp4_status nvfp4_mlp_bwd(const nvfp4_mlp_params* p, const void* dY, const void* saved,
                           void* dX, float* dWg, float* dWu, float* dWd, void* workspace,
                           size_t workspace_bytes, nvfp4_stream stream);

/* Where nvfp4_mlp_fwd / nvfp4_mlp_bwd keep the intermediates of one MLP
 * step inside the caller's `saved` and workspace buffers, so a caller can
 * read them after a call (to inspect or check each stage of the step); the
 * same Figure 1 text passage as the MLP calls.  The bf16 tensors (row-major):
 *   G, U       [M, F]  in saved      (gate and up projections, forward)
 *   H          [M, F]  in workspace  (silu(G) * U, forward)
 *   DH, DG, DU [M, F]  in workspace  (backward: dY Wd, the SwiGLU derivative)
 *   DX_GATE    [M, D]  in workspace  (backward: bf16(dG Wg), which the
 *                                     second DGRAD adds to dU Wu)
 * Contents are those the last fwd (G, U, H) or bwd (the others) call wrote.
 */
enum {
  NVFP4_MLP_G = 0, NVFP4_MLP_U = 1, NVFP4_MLP_H = 2, NVFP4_MLP_DH = 3, NVFP4_MLP_DG = 4,
  NVFP4_MLP_DU = 5, NVFP4_MLP_DX_GATE = 6
};
/* *data = device address of tensor `which` inside saved / workspace (the
 * buffer that holds it must not be NULL; the other may be), *rows, *cols its
 * shape.  Returns NVFP4_ERR_SHAPE as nvfp4_mlp_sizes, NVFP4_ERR_INVALID_ARG for
 * an unknown `which` or a NULL pointer.  Nothing is launched. */
nvfp4_status nvfp4_mlp_tensor(int64_t M, int64_t D, int64_t F, const void* saved,
                              const void* workspace, int32_t which, void** data, int64_t* rows,
                              int64_t* cols);

/* The quantised operands of the nine GEMMs (descriptors with rows x cols the
 * logical K-major operand, as nvfp4_quantize fills them):
 *   Q_WG, Q_WU [F, D], Q_WD [D, F]  in saved  16x16 with the transpose
 *                                             (codes_t / scales_t)
 *   Q_XC [D, M], Q_HC [F, M]        in saved  the forward's WGRAD operands
 *   Q_X [M, D], Q_H [M, F]          in workspace (FPROP operands)
 *   Q_DY [M, D], Q_DG, Q_DU [M, F]  in workspace (DGRAD operands, SR)
 *   Q_DYC [D, M], Q_DGC, Q_DUC [F, M] in workspace (WGRAD operands)
 * *out receives the pointers into the buffers; amax and s_dec point at the
 * device floats the quantiser wrote.  Returns as nvfp4_mlp_tensor. */
enum {
  NVFP4_MLP_Q_WG = 16, NVFP4_MLP_Q_WU = 17, NVFP4_MLP_Q_WD = 18, NVFP4_MLP_Q_X = 19,
  NVFP4_MLP_Q_XC = 20, NVFP4_MLP_Q_H = 21, NVFP4_MLP_Q_HC = 22, NVFP4_MLP_Q_DY = 23,
  NVFP4_MLP_Q_DYC = 24, NVFP4_MLP_Q_DG = 25, NVFP4_MLP_Q_DGC = 26, NVFP4_MLP_Q_DU = 27,
  NVFP4_MLP_Q_DUC = 28
};
nvfp4_status nvfp4_mlp_operand(int64_t M, int64_t D, int64_t F, const void* saved,
                               const void* workspace, int32_t which, nvfp4_tensor* out);

/* ---------------------------------------------------------------------- */
/* Optimizer step of an FP32 master weight                                  */
/* ---------------------------------------------------------------------- */
/* "NVFP4 pretraining recipe" page, Figure 1 text: the MLP GEMMs' BF16
 * outputs are folded into FP32 master weights on the optimizer step, and
 * each step quantises the weights 16x16 under a per-tensor FP32 scale taken
 * from the tensor's amax.  This call is that step for one weight, fused with
 * the amax of the updated weight, so the next quantisation needs no amax
 * pass.  The pages name no optimizer: plain SGD on the FP32 master weight W
 * and the FP32 master gradient G (the WGRAD results the GEMM's
 * NVFP4_D_F32_ACCUM mode or nvfp4_mlp_bwd folded into it), elementwise in
 * binary32, the product rounded first:
 *   W[i]  = W[i] - lr * G[i]
 *   G[i]  = 0                  with NVFP4_ZERO_GRAD in flags
 *   *amax = max_i |W[i]|       of the updated W, when amax is not NULL: bit
 *                              for bit what nvfp4_amax returns for W, so it
 *                              can be given to the 16x16 quantiser
 *                              (NVFP4_AMAX_GIVEN), or written straight into
 *                              an MLP weight operand's amax slot for an
 *                              nvfp4_mlp_fwd with NVFP4_AMAX_GIVEN.
 * W, G: device float [n], 16-byte aligned, not overlapping; n > 0, n % 4 == 0;
 * lr finite.  amax: device float, 4-byte aligned, or NULL.  workspace:
 * device scratch of at least the nvfp4_quantize_sizes workspace size
 * (16-byte aligned) when amax is not NULL, else unused (may be NULL);
 * contents on return unspecified.  One read of W and G, one write of W (and
 * of G with NVFP4_ZERO_GRAD); two kernel launches on `stream` (one without
 * amax); nothing is allocated.  Returns NVFP4_ERR_INVALID_ARG (NULL W or G,
 * W and G overlapping, unknown flag bits, lr not finite), _SHAPE, _ALIGN,
 * _WORKSPACE, _ARCH, _CUDA. */
enum { NVFP4_ZERO_GRAD = 16u };
nvfp4_status nvfp4_sgd_step(float* W, float* G, int64_t n, float lr, uint32_t flags, float* amax,
                            void* workspace, size_t workspace_bytes, nvfp4_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4_H */
