"""The layer step captured as one CUDA graph and replayed writes exactly what
the same calls write when launched one by one.

The step is the hot path of one NVFP4 linear layer ("NVFP4 pretraining
recipe" page, Figure 1 text and recipe bullets 1-5): X's and dY's amaxes
(one read each), X's row-wise and column-wise RHT operands, W's 16x16
operand with its transposed codes, dY's row-wise SR and column-wise RHT + SR
operands, then FPROP, DGRAD and WGRAD.  Every entry point takes a stream and
caller-owned buffers and makes no host synchronisation, so the step can be
captured; the shapes below send FPROP and WGRAD to the 256 x 384 CTA-pair
tile and DGRAD to the 256 x 256 one.  Outputs are compared bit for bit
(same kernels, same inputs, deterministic SR).
"""
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nv():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from nvfp4_block_scaled_03_gb300 import binding
    return binding


def _operands(nv, M, K, N):
    import torch
    g = torch.Generator(device="cuda").manual_seed(7)
    X = torch.randn(M, K, generator=g, device="cuda").to(torch.bfloat16)
    W = (0.02 * torch.randn(N, K, generator=g, device="cuda")).to(torch.bfloat16)
    dY = (1e-3 * torch.randn(M, N, generator=g, device="cuda")).to(torch.bfloat16)
    q = {
        "X": nv.alloc_qtensor(M, K, nv.ROW_1X16, device=X.device),
        "Xc": nv.alloc_qtensor(M, K, nv.COL_1X16, device=X.device),
        "W": nv.alloc_qtensor(N, K, nv.BLOCK_16X16, nv.EMIT_T, device=X.device),
        "dY": nv.alloc_qtensor(M, N, nv.ROW_1X16, device=X.device),
        "dYc": nv.alloc_qtensor(M, N, nv.COL_1X16, device=X.device),
    }
    out = {"Y": torch.empty(M, N, dtype=torch.bfloat16, device="cuda"),
           "dX": torch.empty(M, K, dtype=torch.bfloat16, device="cuda"),
           "dW": torch.empty(N, K, dtype=torch.bfloat16, device="cuda")}
    ws = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    return X, W, dY, q, out, ws


def _step(nv, X, W, dY, q, out, ws):
    nv.nvfp4_amax(X, q["X"].amax, q["Xc"].amax, seed=0, workspace=ws)
    nv.nvfp4_quantize_rowcol(X, 0, nv.RHT, seed=0, row_out=q["X"], col_out=q["Xc"])
    nv.nvfp4_quantize(W, nv.BLOCK_16X16, nv.EMIT_T, out=q["W"], workspace=ws)
    nv.nvfp4_amax(dY, q["dY"].amax, q["dYc"].amax, seed=0, workspace=ws)
    nv.nvfp4_quantize_rowcol(dY, nv.SR, nv.RHT | nv.SR, seed=0, row_offset=0, col_offset=1,
                             row_out=q["dY"], col_out=q["dYc"])
    nv.nvfp4_gemm(q["X"], q["W"], out=out["Y"])
    nv.nvfp4_gemm(q["dY"], q["W"], b_view=1, out=out["dX"])
    nv.nvfp4_gemm(q["dYc"], q["Xc"], out=out["dW"])


def _snapshot(q, out):
    snap = {k: v.clone() for k, v in out.items()}
    for name, t in q.items():
        for f in ("codes", "scales", "amax", "s_dec", "codes_t", "scales_t"):
            v = getattr(t, f, None)
            if v is not None:
                snap[f"{name}.{f}"] = v.clone()
    return snap


def _clear(q, out):
    for v in out.values():
        v.fill_(0)
    for t in q.values():
        for f in ("codes", "scales", "amax", "s_dec", "codes_t", "scales_t"):
            v = getattr(t, f, None)
            if v is not None:
                v.fill_(0)


def test_layer_step_graph_replay_equals_eager(nv):
    import torch
    M, K, N = 2048, 4096, 14336
    X, W, dY, q, out, ws = _operands(nv, M, K, N)
    _step(nv, X, W, dY, q, out, ws)
    nv.check_device_errors()
    eager = _snapshot(q, out)

    _clear(q, out)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _step(nv, X, W, dY, q, out, ws)
    for replay in range(2):
        _clear(q, out)
        graph.replay()
        torch.cuda.synchronize()
        nv.check_device_errors()
        now = _snapshot(q, out)
        for k, v in eager.items():
            assert torch.equal(v.view(torch.uint8), now[k].view(torch.uint8)), \
                f"replay {replay}: {k} differs from the eager step"


def test_mlp_step_graph_replay_equals_eager(nv):
    """The SwiGLU MLP forward + backward (nine GEMMs, the SwiGLU kernels,
    every quantisation of the recipe, WGRAD folded into FP32 master
    gradients) captured as one graph: a replay writes Y, dX and the folded
    gradients exactly as the eager calls do."""
    import torch
    M, D, F = 512, 512, 1024
    g = torch.Generator(device="cuda").manual_seed(11)
    X = torch.randn(M, D, generator=g, device="cuda").to(torch.bfloat16)
    dY = (1e-3 * torch.randn(M, D, generator=g, device="cuda")).to(torch.bfloat16)
    Wg, Wu = (0.02 * torch.randn(F, D, generator=g, device="cuda") for _ in range(2))
    Wd = 0.02 * torch.randn(D, F, generator=g, device="cuda")
    sb, wb = nv.mlp_sizes(M, D, F)
    saved = torch.empty(sb, dtype=torch.uint8, device="cuda")
    ws = torch.empty(wb, dtype=torch.uint8, device="cuda")
    Y = torch.empty(M, D, dtype=torch.bfloat16, device="cuda")
    dX = torch.empty_like(Y)
    grads = [torch.zeros_like(w) for w in (Wg, Wu, Wd)]
    p = nv.mlp_params(M, D, F, Wg, Wu, Wd, seed=5, step=3, rht=True)

    def step():
        for t in grads:
            t.zero_()
        nv.nvfp4_mlp_fwd(p, X, Y, saved, ws)
        nv.nvfp4_mlp_bwd(p, dY, saved, dX, *grads, ws)

    step()
    nv.check_device_errors()
    eager = [t.clone() for t in (Y, dX, *grads)]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for t in (Y, dX, *grads):
        t.fill_(0)
    graph.replay()
    torch.cuda.synchronize()
    nv.check_device_errors()
    for name, a, b in zip(("Y", "dX", "dWg", "dWu", "dWd"), eager, (Y, dX, *grads)):
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), f"{name} differs"
