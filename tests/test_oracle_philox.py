"""Pins of the oracle's Philox4x32-10 generator -- CPU only.

The external pin is Triton's own Philox4x32-10 (``tl.randint4x``), *run* in
Triton's CPU interpreter in a subprocess: an implementation written by another
project from the same SC'11 definition.  Its mapping is key = (seed low, seed
high) and counter = (offset, 0, 0, 0).
"""
import json
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest

_TRITON_SCRIPT = textwrap.dedent("""
    import json, os, sys
    os.environ["TRITON_INTERPRET"] = "1"
    import torch, triton, triton.language as tl

    @triton.jit
    def k(out_ptr, seed, base, N: tl.constexpr):
        offs = tl.arange(0, N) + base
        a, b, c, d = tl.randint4x(seed, offs)
        i = tl.arange(0, N)
        tl.store(out_ptr + i * 4 + 0, a)
        tl.store(out_ptr + i * 4 + 1, b)
        tl.store(out_ptr + i * 4 + 2, c)
        tl.store(out_ptr + i * 4 + 3, d)

    res = {}
    for seed, base in json.loads(sys.argv[1]):
        out = torch.zeros(64 * 4, dtype=torch.int32)
        k[(1,)](out, seed, base, 64)
        res[f"{seed},{base}"] = [v & 0xffffffff for v in out.tolist()]
    print(json.dumps(res))
""")


def _triton_available():
    try:
        import triton  # noqa: F401
        import torch  # noqa: F401
        return True
    except Exception:
        return False


@pytest.mark.skipif(not _triton_available(), reason="triton not importable")
def test_philox_matches_triton_interpreter(orc):
    cases = [(0, 0), (1, 0), (12345, 1000), (0x7FFFFFFF, 77), (987654321, 1 << 20)]
    env = dict(os.environ, TRITON_INTERPRET="1")
    out = subprocess.check_output([sys.executable, "-c", _TRITON_SCRIPT, json.dumps(cases)],
                                  env=env, text=True, timeout=600)
    ref = json.loads(out.strip().splitlines()[-1])
    for seed, base in cases:
        words = ref[f"{seed},{base}"]
        for i in range(64):
            got = orc.philox([base + i, 0, 0, 0], [seed & 0xFFFFFFFF, seed >> 32])
            assert got == words[4 * i:4 * i + 4], (seed, base, i)


def test_philox_inputs_all_matter_and_bits_balance(orc):
    base = orc.philox([1, 2, 3, 4], [5, 6])
    for j in range(4):
        c = [1, 2, 3, 4]
        c[j] ^= 1
        assert orc.philox(c, [5, 6]) != base
    for j in range(2):
        k = [5, 6]
        k[j] ^= 1
        assert orc.philox([1, 2, 3, 4], k) != base
    words = np.array([orc.sr_word(3, 9, i) for i in range(4096)], dtype=np.uint64)
    bits = ((words[:, None] >> np.arange(32, dtype=np.uint64)) & 1).mean(axis=0)
    assert np.all(np.abs(bits - 0.5) < 5 * 0.5 / np.sqrt(4096))


def test_sr_word_layout(orc):
    # idx -> counter (idx/4, stream 0, offset), word idx%4
    for idx in (0, 1, 2, 3, 4, 4095, (1 << 33) + 5):
        g = idx // 4
        w = orc.philox([g & 0xFFFFFFFF, g >> 32, 0, 17], [42, 0])
        assert orc.sr_word(42, 17, idx) == w[idx % 4]


def test_rht_signs(orc):
    signs = [orc.rht_signs(s) for s in range(256)]
    for s in signs:
        assert set(np.unique(s)).issubset({-1.0, 1.0})
    allv = np.stack(signs)
    assert abs((allv < 0).mean() - 0.5) < 0.05
    assert len({tuple(s) for s in signs}) == 256
