"""Blockwise-FP8 and MXFP8 linear-layer training kernels for GB300 (sm_103a).

The compute lives in ``libfp8bw.so`` (hand-written CUDA behind a C ABI, see
``include/fp8bw.h``); ``binding`` marshals torch tensors into its calls.
Importing this package does not load the library: ``binding.lib()`` does, and
raises if it has not been built.
"""
