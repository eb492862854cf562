"""GB300-native NVFP4 linear-layer kernels (quantisers + tcgen05 block-scaled
GEMMs) behind a C-ABI library, ``libnvfp4.so``.

The Python side is a thin ctypes binding (:mod:`.binding`) with the C-ABI's
names; it is imported lazily so that :mod:`.synthetic` (the seeded input
generators) can be used without the CUDA library.
"""
__all__ = ["binding", "synthetic"]


def __getattr__(name):
    if name == "binding":
        from . import binding
        return binding
    raise AttributeError(name)
