"""Failure detection on the GPU without a fault: the bounded waits.

Every pipeline wait of the quantise passes and of the GEMM kernels is
bounded; on expiry a kernel records a code in its device error word, stops
its other roles at their next wait, drains what it issued and frees its
tensor memory, so the context stays usable and nvfp4_check_device_errors
reports NVFP4_ERR_DEVICE_TIMEOUT.  These tests make a wait run out (the
injected stall: the producer issues no loads, so nothing the consumers wait
for ever arrives) under a 1 ms limit, read the status, then run the same call
normally and check it bit for bit (quantiser) or within the GEMM tolerance --
which also shows the error word was cleared and tensor memory freed (a leaked
allocation would block the next GEMM's allocation)."""
import numpy as np
import pytest

import gpu_helpers as H
from nvfp4_block_scaled_03_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu
LIMIT_NS = 1_000_000


@pytest.fixture(scope="module")
def nv():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from nvfp4_block_scaled_03_gb300 import binding
    return binding


@pytest.mark.parametrize("mode,flags", [(0, 2), (1, 3), (2, 4)])
def test_quantize_wait_expires_then_recovers(nv, orc, mode, flags):
    x = syn.activations((128, 256), seed=1)
    xt = H.dev_bf16(x)
    nv.check_device_errors()
    nv.debug_inject(nv.STALL_QUANTIZE, LIMIT_NS)
    try:
        nv.nvfp4_quantize(xt, mode, flags, seed=3, offset=1)
        with pytest.raises(nv.NVFP4Error) as e:
            nv.check_device_errors()
        assert e.value.status == nv.ERR_DEVICE_TIMEOUT
    finally:
        nv.debug_inject(0, 0)
    nv.check_device_errors()                       # the error word was cleared
    q = nv.nvfp4_quantize(xt, mode, flags, seed=3, offset=1)
    nv.check_device_errors()
    H.assert_quant_equal(q, orc.quantize(x, mode, flags, seed=3, offset=1), "after recovery")


@pytest.mark.parametrize("tile", [1, 2, 5, 3, 6])  # single-SM tiles, then the CTA pairs
def test_gemm_wait_expires_then_recovers(nv, orc, tile):
    X, W = syn.activations((128, 512), seed=1), syn.weights((256, 512), seed=2)
    a, b = orc.quantize(X, orc.ROW_1X16), orc.quantize(W, orc.BLOCK_16X16)
    A, B = H.upload(nv, a), H.upload(nv, b)
    nv.check_device_errors()
    nv.debug_inject(nv.STALL_GEMM, LIMIT_NS)
    try:
        nv.nvfp4_gemm(A, B, tile=tile)
        with pytest.raises(nv.NVFP4Error) as e:
            nv.check_device_errors()
        assert e.value.status == nv.ERR_DEVICE_TIMEOUT
    finally:
        nv.debug_inject(0, 0)
    nv.check_device_errors()
    for _ in range(2):                             # tensor memory is allocatable again
        D = nv.nvfp4_gemm(A, B, tile=tile)
        nv.check_device_errors()
        H.assert_gemm_close(H.host_f64(D), orc.gemm_fp64(a, b), f"tile {tile} after recovery")


def test_debug_inject_rejects_unknown_bits(nv):
    with pytest.raises(nv.NVFP4Error) as e:
        nv.debug_inject(8, 0)
    assert e.value.status == nv.ERR_INVALID_ARG
    nv.debug_inject(0, 0)
