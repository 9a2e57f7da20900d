"""GB300 (sm_103a) tiled GEMM / Linear-layer library.

The compute path is the C-ABI shared library built from ``csrc/`` (see
``include/gemm.h``); ``gemm`` is its thin ctypes binding.  Importing the
package does not load the library; the first call into ``gemm`` does, and
raises if it has not been built.
"""
__all__ = ["gemm", "inputs", "roofline"]


def __getattr__(name):
    if name == "gemm":
        from . import gemm as _g
        return _g
    raise AttributeError(name)
