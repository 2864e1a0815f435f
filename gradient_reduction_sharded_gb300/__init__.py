"""Ownership-aware sharded gradient reduction + clip + AdamW on GB300.

The compute path is libgrs.so (hand-written sm_103a CUDA kernels behind the
C ABI in include/grs.h); `grs` is its thin ctypes binding with the same
names.  Importing `grs` (or any of its names from this package) fails if
the library has not been built: there is no fallback.
"""
import importlib


def __getattr__(name):
    if name.startswith("_"):
        raise AttributeError(name)  # private names and submodules such as _build
    mod = importlib.import_module(__name__ + ".grs")
    if name == "grs":
        return mod
    return getattr(mod, name)
