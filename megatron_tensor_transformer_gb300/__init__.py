"""Megatron-style tensor-parallel linear layers of a Llama block on one GB300.

The compute lives in libtpx.so (CUDA for sm_103a, C ABI in include/tpx.h);
``tpx`` is its ctypes binding and ``inputs`` draws the seeded synthetic tensors.
"""
