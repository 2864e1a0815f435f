"""Ownership-aware sharded gradient reduction + clip + AdamW on GB300.

The compute path is libgrs.so (hand-written sm_103a CUDA kernels behind the
C ABI in include/grs.h); `grs` is its thin ctypes binding with the same
names.  Importing this package fails if the library has not been built.
"""
from . import grs  # noqa: F401  (fails loudly when libgrs.so is missing)
from .grs import *  # noqa: F401,F403
