"""Kitty 2-bit paged KV cache with Dynamic Channel-wise Precision Boost, on GB300.

The compute path lives in the CUDA library ``libkitty.so`` (C ABI declared in
``include/kitty.h``); :mod:`mixed_precision_bit_gb300.kitty` is its thin ctypes
binding.  :mod:`mixed_precision_bit_gb300.synth` holds seeded input generators.
"""
