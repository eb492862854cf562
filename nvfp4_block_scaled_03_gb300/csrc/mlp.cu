// mlp.cu -- SwiGLU MLP forward / backward with NVFP4 GEMMs: the host-side
// sequence of quantiser, GEMM and SwiGLU launches on one stream, with the
// caller's saved-activation buffer and workspace carved into the operands
// ("NVFP4 pretraining recipe" page, Figure 1 text: the three MLP GEMMs of
// each projection consume NVFP4 inputs and emit BF16; BF16 weight gradients
// are folded into the FP32 master gradient).
//
// Per-operand recipe (bullets 3-5): X, H row-wise RNE for FPROP; W 16x16 RNE
// with its transpose for DGRAD; dY, dG, dU row-wise SR for DGRAD; the WGRAD
// operands X^T, H^T, dY^T, dG^T, dU^T column-wise, with the RHT (one sign
// vector per seed, shared by every WGRAD pair) when flags has NVFP4_RHT, RNE
// for activations and SR for gradients.  SR offsets: 8*step + 0..5 for
// dY row/col, dG row/col, dU row/col.
#include "internal.h"

namespace nvfp4 {
namespace {

struct Carver {
  uint8_t* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<uint8_t*>(b)) {}
  void* take(size_t bytes) {
    off = (off + 255) & ~size_t(255);
    void* p = base ? base + off : nullptr;
    off += bytes;
    return p;
  }
};

// One quantised operand carved from a buffer.
void carve_q(Carver& c, nvfp4_tensor* t, int64_t rows, int64_t cols, int32_t mode, bool emit_t) {
  size_t codes = 0, sc = 0, sct = 0;
  nvfp4_quantize_sizes(rows, cols, mode, emit_t ? NVFP4_EMIT_T : 0u, &codes, &sc, &sct, nullptr);
  t->codes = c.take(codes);
  t->scales = c.take(sc);
  t->codes_t = emit_t ? c.take(codes) : nullptr;
  t->scales_t = emit_t ? c.take(sct) : nullptr;
  t->amax = static_cast<float*>(c.take(sizeof(float)));
  t->s_dec = static_cast<float*>(c.take(sizeof(float)));
  t->rows = t->cols = 0;
  t->mode = mode;
  t->flags = 0;
}

struct Saved {
  nvfp4_tensor qWg, qWu, qWd, qXc, qHc;
  void* G;
  void* U;
};
struct Work {
  void* partials;
  void* sw_partials;  // the SwiGLU kernels' amax partial maxima
  nvfp4_tensor qX, qH, qdY, qdYc, qdG, qdGc, qdU, qdUc;
  void* H;
  void* dH;
  void* dG;
  void* dU;
  void* dXg;
};

void carve_saved(void* base, int64_t M, int64_t D, int64_t F, Saved* s, size_t* bytes) {
  Carver c(base);
  carve_q(c, &s->qWg, F, D, NVFP4_BLOCK_16X16, true);
  carve_q(c, &s->qWu, F, D, NVFP4_BLOCK_16X16, true);
  carve_q(c, &s->qWd, D, F, NVFP4_BLOCK_16X16, true);
  carve_q(c, &s->qXc, M, D, NVFP4_COL_1X16, false);
  carve_q(c, &s->qHc, M, F, NVFP4_COL_1X16, false);
  s->G = c.take((size_t)(M * F * 2));
  s->U = c.take((size_t)(M * F * 2));
  *bytes = c.off;
}

void carve_work(void* base, int64_t M, int64_t D, int64_t F, Work* w, size_t* bytes) {
  Carver c(base);
  w->partials = c.take(kQuantWorkspaceBytes);
  w->sw_partials = c.take(kSwigluPartialsBytes);
  carve_q(c, &w->qX, M, D, NVFP4_ROW_1X16, false);
  carve_q(c, &w->qH, M, F, NVFP4_ROW_1X16, false);
  carve_q(c, &w->qdY, M, D, NVFP4_ROW_1X16, false);
  carve_q(c, &w->qdYc, M, D, NVFP4_COL_1X16, false);
  carve_q(c, &w->qdG, M, F, NVFP4_ROW_1X16, false);
  carve_q(c, &w->qdGc, M, F, NVFP4_COL_1X16, false);
  carve_q(c, &w->qdU, M, F, NVFP4_ROW_1X16, false);
  carve_q(c, &w->qdUc, M, F, NVFP4_COL_1X16, false);
  w->H = c.take((size_t)(M * F * 2));
  w->dH = c.take((size_t)(M * F * 2));
  w->dG = c.take((size_t)(M * F * 2));
  w->dU = c.take((size_t)(M * F * 2));
  w->dXg = c.take((size_t)(M * D * 2));
  *bytes = c.off;
}

bool dims_ok(int64_t M, int64_t D, int64_t F) {
  return M > 0 && D > 0 && F > 0 && M % 128 == 0 && D % 128 == 0 && F % 128 == 0;
}

#define NVFP4_TRY(expr)                     \
  do {                                      \
    nvfp4_status _s = (expr);               \
    if (_s != NVFP4_OK) return _s;          \
  } while (0)

// A bf16 operand [rows, cols] quantised twice -- row-wise (FPROP / DGRAD
// operand) and column-wise (WGRAD operand).  With amax_given, row->amax and
// col->amax already hold the tensor amaxes (written by the kernel that
// produced x); otherwise both are taken from one read of x first.  Both
// operands then come from one more read of x.
nvfp4_status quantize_pair(const void* x, int64_t rows, int64_t cols, uint32_t row_flags,
                           uint32_t col_flags, uint64_t seed, uint64_t row_offset,
                           uint64_t col_offset, nvfp4_tensor* row, nvfp4_tensor* col,
                           bool amax_given, void* ws, size_t wsb, cudaStream_t st) {
  if (!amax_given) {
    const bool rht = col_flags & NVFP4_RHT;
    NVFP4_TRY(amax_impl(x, NVFP4_IN_BF16, rows, cols, cols, seed, row->amax,
                        rht ? col->amax : nullptr, ws, wsb, st));
    if (!rht &&
        cudaMemcpyAsync(col->amax, row->amax, sizeof(float), cudaMemcpyDeviceToDevice, st) !=
            cudaSuccess)
      return NVFP4_ERR_CUDA;
  }
  return quantize_rowcol_impl(x, NVFP4_IN_BF16, rows, cols, cols, row_flags | NVFP4_AMAX_GIVEN,
                              col_flags | NVFP4_AMAX_GIVEN, seed, row_offset, col_offset, row, col,
                              st);
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

nvfp4_status nvfp4_mlp_sizes(int64_t M, int64_t D, int64_t F, size_t* saved_bytes,
                             size_t* workspace_bytes) {
  if (!dims_ok(M, D, F)) return NVFP4_ERR_SHAPE;
  Saved s;
  Work w;
  size_t sb = 0, wb = 0;
  carve_saved(nullptr, M, D, F, &s, &sb);
  carve_work(nullptr, M, D, F, &w, &wb);
  if (saved_bytes) *saved_bytes = sb;
  if (workspace_bytes) *workspace_bytes = wb;
  return NVFP4_OK;
}

nvfp4_status nvfp4_mlp_fwd(const nvfp4_mlp_params* p, const void* X, void* Y, void* saved,
                           size_t saved_bytes, void* workspace, size_t workspace_bytes,
                           nvfp4_stream stream) {
  if (!p || !X || !Y || !saved || !workspace || !p->Wg || !p->Wu || !p->Wd)
    return NVFP4_ERR_INVALID_ARG;
  if (p->flags & ~(uint32_t)(NVFP4_RHT | NVFP4_AMAX_GIVEN)) return NVFP4_ERR_INVALID_ARG;
  const int64_t M = p->M, D = p->D, F = p->F;
  if (!dims_ok(M, D, F)) return NVFP4_ERR_SHAPE;
  Saved s;
  Work w;
  size_t sb = 0, wb = 0;
  carve_saved(saved, M, D, F, &s, &sb);
  carve_work(workspace, M, D, F, &w, &wb);
  if (saved_bytes < sb || workspace_bytes < wb) return NVFP4_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const uint32_t rht = p->flags & NVFP4_RHT;
  void* ws = w.partials;
  const size_t wsb = kQuantWorkspaceBytes;

  // the weights' amaxes either taken here or already in their operand slots
  // (the optimizer step's fused amax, nvfp4_sgd_step)
  const uint32_t wf = NVFP4_EMIT_T | (p->flags & NVFP4_AMAX_GIVEN);
  NVFP4_TRY(quantize_impl(p->Wg, NVFP4_IN_FP32, F, D, D, NVFP4_BLOCK_16X16, wf, 0, 0, &s.qWg, ws,
                          wsb, st));
  NVFP4_TRY(quantize_impl(p->Wu, NVFP4_IN_FP32, F, D, D, NVFP4_BLOCK_16X16, wf, 0, 0, &s.qWu, ws,
                          wsb, st));
  NVFP4_TRY(quantize_impl(p->Wd, NVFP4_IN_FP32, D, F, F, NVFP4_BLOCK_16X16, wf, 0, 0, &s.qWd, ws,
                          wsb, st));
  NVFP4_TRY(quantize_pair(X, M, D, 0, rht, p->seed, 0, 0, &w.qX, &s.qXc, false, ws, wsb, st));
  NVFP4_TRY(gemm_impl(&w.qX, 0, &s.qWg, 0, s.G, NVFP4_D_BF16, nullptr, M, F, D, 0, st));
  NVFP4_TRY(gemm_impl(&w.qX, 0, &s.qWu, 0, s.U, NVFP4_D_BF16, nullptr, M, F, D, 0, st));
  NVFP4_TRY(swiglu_fwd_impl(s.G, s.U, w.H, M, F, p->seed, rht, w.qH.amax, s.qHc.amax,
                            w.sw_partials, kSwigluPartialsBytes, st));
  NVFP4_TRY(quantize_pair(w.H, M, F, 0, rht, p->seed, 0, 0, &w.qH, &s.qHc, true, ws, wsb, st));
  NVFP4_TRY(gemm_impl(&w.qH, 0, &s.qWd, 0, Y, NVFP4_D_BF16, nullptr, M, D, F, 0, st));
  return NVFP4_OK;
}

nvfp4_status nvfp4_mlp_bwd(const nvfp4_mlp_params* p, const void* dY, const void* saved,
                           void* dX, float* dWg, float* dWu, float* dWd, void* workspace,
                           size_t workspace_bytes, nvfp4_stream stream) {
  if (!p || !dY || !saved || !dX || !dWg || !dWu || !dWd || !workspace)
    return NVFP4_ERR_INVALID_ARG;
  if (p->flags & ~(uint32_t)(NVFP4_RHT | NVFP4_AMAX_GIVEN)) return NVFP4_ERR_INVALID_ARG;
  const int64_t M = p->M, D = p->D, F = p->F;
  if (!dims_ok(M, D, F)) return NVFP4_ERR_SHAPE;
  Saved s;
  Work w;
  size_t sb = 0, wb = 0;
  carve_saved(const_cast<void*>(saved), M, D, F, &s, &sb);
  carve_work(workspace, M, D, F, &w, &wb);
  if (workspace_bytes < wb) return NVFP4_ERR_WORKSPACE;
  // the saved operands' shapes (written by the forward's quantiser calls)
  s.qWg.rows = F; s.qWg.cols = D;
  s.qWu.rows = F; s.qWu.cols = D;
  s.qWd.rows = D; s.qWd.cols = F;
  s.qXc.rows = D; s.qXc.cols = M;
  s.qHc.rows = F; s.qHc.cols = M;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const uint32_t rht = p->flags & NVFP4_RHT;
  const uint64_t o = 8 * p->step;
  void* ws = w.partials;
  const size_t wsb = kQuantWorkspaceBytes;

  NVFP4_TRY(quantize_pair(dY, M, D, NVFP4_SR, rht | NVFP4_SR, p->seed, o + 0, o + 1, &w.qdY,
                          &w.qdYc, false, ws, wsb, st));
  // DGRAD of the down projection: dH = dY . Wd  (Wd read through its transpose)
  NVFP4_TRY(gemm_impl(&w.qdY, 0, &s.qWd, 1, w.dH, NVFP4_D_BF16, nullptr, M, F, D, 0, st));
  // WGRAD of the down projection: dWd += dY^T . H
  NVFP4_TRY(gemm_impl(&w.qdYc, 0, &s.qHc, 0, dWd, NVFP4_D_F32_ACCUM, nullptr, D, F, M, 0, st));
  NVFP4_TRY(swiglu_bwd_impl(w.dH, s.G, s.U, w.dG, w.dU, M, F, p->seed, rht, w.qdG.amax,
                            w.qdGc.amax, w.qdU.amax, w.qdUc.amax, w.sw_partials,
                            kSwigluPartialsBytes, st));
  NVFP4_TRY(quantize_pair(w.dG, M, F, NVFP4_SR, rht | NVFP4_SR, p->seed, o + 2, o + 3, &w.qdG,
                          &w.qdGc, true, ws, wsb, st));
  NVFP4_TRY(quantize_pair(w.dU, M, F, NVFP4_SR, rht | NVFP4_SR, p->seed, o + 4, o + 5, &w.qdU,
                          &w.qdUc, true, ws, wsb, st));
  // DGRAD of gate and up: dX = dG . Wg + dU . Wu (second GEMM adds the first)
  NVFP4_TRY(gemm_impl(&w.qdG, 0, &s.qWg, 1, w.dXg, NVFP4_D_BF16, nullptr, M, D, F, 0, st));
  NVFP4_TRY(gemm_impl(&w.qdU, 0, &s.qWu, 1, dX, NVFP4_D_BF16_ADD_C, w.dXg, M, D, F, 0, st));
  // WGRAD of gate and up: dWg += dG^T . X, dWu += dU^T . X
  NVFP4_TRY(gemm_impl(&w.qdGc, 0, &s.qXc, 0, dWg, NVFP4_D_F32_ACCUM, nullptr, F, D, M, 0, st));
  NVFP4_TRY(gemm_impl(&w.qdUc, 0, &s.qXc, 0, dWu, NVFP4_D_F32_ACCUM, nullptr, F, D, M, 0, st));
  return NVFP4_OK;
}

nvfp4_status nvfp4_mlp_tensor(int64_t M, int64_t D, int64_t F, const void* saved,
                              const void* workspace, int32_t which, void** data, int64_t* rows,
                              int64_t* cols) {
  if (!dims_ok(M, D, F)) return NVFP4_ERR_SHAPE;
  if (!data || !rows || !cols) return NVFP4_ERR_INVALID_ARG;
  Saved s;
  Work w;
  size_t sb = 0, wb = 0;
  carve_saved(const_cast<void*>(saved), M, D, F, &s, &sb);
  carve_work(const_cast<void*>(workspace), M, D, F, &w, &wb);
  void* p = nullptr;
  int64_t r = M, c = F;
  switch (which) {
    case NVFP4_MLP_G: p = s.G; break;
    case NVFP4_MLP_U: p = s.U; break;
    case NVFP4_MLP_H: p = w.H; break;
    case NVFP4_MLP_DH: p = w.dH; break;
    case NVFP4_MLP_DG: p = w.dG; break;
    case NVFP4_MLP_DU: p = w.dU; break;
    case NVFP4_MLP_DX_GATE: p = w.dXg; c = D; break;
    default: return NVFP4_ERR_INVALID_ARG;
  }
  const bool in_saved = which == NVFP4_MLP_G || which == NVFP4_MLP_U;
  if (!(in_saved ? saved : workspace)) return NVFP4_ERR_INVALID_ARG;
  *data = p;
  *rows = r;
  *cols = c;
  return NVFP4_OK;
}

nvfp4_status nvfp4_mlp_operand(int64_t M, int64_t D, int64_t F, const void* saved,
                               const void* workspace, int32_t which, nvfp4_tensor* out) {
  if (!dims_ok(M, D, F)) return NVFP4_ERR_SHAPE;
  if (!out) return NVFP4_ERR_INVALID_ARG;
  Saved s;
  Work w;
  size_t sb = 0, wb = 0;
  carve_saved(const_cast<void*>(saved), M, D, F, &s, &sb);
  carve_work(const_cast<void*>(workspace), M, D, F, &w, &wb);
  const nvfp4_tensor* t = nullptr;
  int64_t r = 0, c = 0;  // the operand's logical (K-major) shape
  bool in_saved = true;
  switch (which) {
    case NVFP4_MLP_Q_WG: t = &s.qWg; r = F; c = D; break;
    case NVFP4_MLP_Q_WU: t = &s.qWu; r = F; c = D; break;
    case NVFP4_MLP_Q_WD: t = &s.qWd; r = D; c = F; break;
    case NVFP4_MLP_Q_XC: t = &s.qXc; r = D; c = M; break;
    case NVFP4_MLP_Q_HC: t = &s.qHc; r = F; c = M; break;
    default: in_saved = false; break;
  }
  if (!in_saved) {
    switch (which) {
      case NVFP4_MLP_Q_X: t = &w.qX; r = M; c = D; break;
      case NVFP4_MLP_Q_H: t = &w.qH; r = M; c = F; break;
      case NVFP4_MLP_Q_DY: t = &w.qdY; r = M; c = D; break;
      case NVFP4_MLP_Q_DYC: t = &w.qdYc; r = D; c = M; break;
      case NVFP4_MLP_Q_DG: t = &w.qdG; r = M; c = F; break;
      case NVFP4_MLP_Q_DGC: t = &w.qdGc; r = F; c = M; break;
      case NVFP4_MLP_Q_DU: t = &w.qdU; r = M; c = F; break;
      case NVFP4_MLP_Q_DUC: t = &w.qdUc; r = F; c = M; break;
      default: return NVFP4_ERR_INVALID_ARG;
    }
  }
  if (!(in_saved ? saved : workspace)) return NVFP4_ERR_INVALID_ARG;
  *out = *t;
  out->rows = r;
  out->cols = c;
  out->flags = t->codes_t ? (uint32_t)NVFP4_EMIT_T : 0u;
  return NVFP4_OK;
}

}  // extern "C"
