"""Vocab-wide logprobs, entropy and KL (and fused linear logp) on GB300.

The compute runs in ``libvp.so`` (hand-written CUDA for sm_103a behind a C-ABI,
declared in ``include/vp.h``). This package is a thin ctypes binding: it turns
torch tensors into pointers, sizes and strides and calls the C functions of the
same names. There is no CPU fallback: every call raises if the library is
missing or no CUDA device is present.
"""
__all__ = ["workloads"]
