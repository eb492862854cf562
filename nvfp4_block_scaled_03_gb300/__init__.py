"""GB300-native NVFP4 linear-layer kernels (quantisers + tcgen05 block-scaled
GEMMs) behind a C-ABI library, ``libnvfp4.so``.

Import :mod:`nvfp4_block_scaled_03_gb300.binding` for the ctypes binding with
the C ABI's names (it loads the CUDA library and fails if it is not built);
:mod:`.synthetic` holds the seeded input generators and needs no GPU.
"""
