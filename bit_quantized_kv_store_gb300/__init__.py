"""Attention over a sub-byte quantized KV cache, native to GB300 (sm_103a).

The compute lives in ``libkvq.so`` (CUDA kernels behind the C ABI of
``include/kvq.h``); ``_lib`` is its ctypes binding and ``synth`` holds the
seeded synthetic input recipes.  Importing the package does not load the
library; the first call into ``_lib`` does, and raises if it is not built.
"""
from . import _lib as kvq  # noqa: F401

__all__ = ["kvq"]
