"""GB300-native batched GQA attention over a paged bf16 KV cache.

The compute path is the C-ABI library ``libpkv.so`` (CUDA kernels for sm_103a, see
``csrc/``); ``binding`` wraps it with ctypes.  Importing this package loads nothing:
``binding.load()`` opens the library and raises if it is missing.
"""
__all__ = ["binding", "workloads"]
