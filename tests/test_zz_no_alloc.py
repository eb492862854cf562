"""The quantiser entry point that allocates nothing (nvfp4_quantize_noalloc).

It exists for callers that cannot give the library device scratch memory --
for example code running under CUDA graph capture, where cudaMalloc is not
allowed, or a plugin that is handed only its input and output buffers.  Its
scratch (the amax pass's partial maxima) is a fixed array inside the library.
This test calls it through the C ABI twice in a row -- a large tensor with
large values, then a smaller one with small values, so a stale partial from
the first call would corrupt the second call's amax -- and checks every
output byte against the workspace-taking nvfp4_quantize on the same inputs
(the quantiser tolerance is bit-exact).  This file is collected last so that a
run that stops at the first failure has run every other test before it.
"""
import ctypes as C

import numpy as np
import pytest

from nvfp4_block_scaled_03_gb300 import synthetic as syn

pytestmark = pytest.mark.gpu


def _dev(bits):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def test_noalloc_entry_point_matches_nvfp4_quantize_twice():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from nvfp4_block_scaled_03_gb300 import binding as nv
    f = nv.lib.nvfp4_quantize_noalloc
    calls = [
        (syn.f32_to_bf16_bits(syn.bf16_bits_to_f32(syn.activations((1024, 2048), seed=41)) * 1000),
         nv.COL_1X16, nv.RHT | nv.SR, 5, 2),
        (syn.gradients((256, 512), seed=42), nv.ROW_1X16, nv.SR, 6, 3),
    ]
    stream = torch.cuda.current_stream().cuda_stream
    for bits, mode, flags, seed, offset in calls:
        x = _dev(bits)
        rows, cols = x.shape
        ref = nv.nvfp4_quantize(x, mode, flags, seed=seed, offset=offset)
        out = nv.alloc_qtensor(rows, cols, mode, flags)
        st = f(C.c_void_p(x.data_ptr()), nv.IN_BF16, rows, cols, cols, mode, flags, seed, offset,
               C.byref(out.desc), C.c_void_p(stream))
        assert st == nv.OK, nv.status_string(st)
        torch.cuda.synchronize()
        for name in ("codes", "scales", "amax", "s_dec"):
            assert torch.equal(getattr(out, name), getattr(ref, name)), name
        assert (out.rows, out.cols) == (ref.rows, ref.cols)
    nv.check_device_errors()
