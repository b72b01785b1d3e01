"""Fused Swin (shifted-)window multi-head attention for GB300 (sm_103a).

The compute path is a C-ABI shared library (``libswin_wattn.so``, declared in
``include/swin_wattn.h``) built from the CUDA sources in ``csrc/``; ``capi`` is its thin
ctypes binding. Importing the package does not load CUDA; ``capi.load()`` does, and fails
loudly when the library has not been built.
"""
from . import inputs  # noqa: F401

__all__ = ["inputs"]
