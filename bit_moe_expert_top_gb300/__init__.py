"""GB300-native low-bit routed-expert FFN (2-bit codebook / MXFP4 / FP8 workspace).

The compute lives in ``libmoe.so`` (hand-written CUDA for sm_103a, C ABI in
``include/moe.h``).  ``_lib`` is its ctypes binding (same names as the C entry
points), ``layer.MoELayer`` chains the calls of one layer step, ``synth`` holds
the seeded input recipes.  Importing the package loads nothing; the library
is loaded on first use and its absence is an error.
"""
__all__ = ["synth", "_lib", "layer", "build"]
