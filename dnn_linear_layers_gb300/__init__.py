"""GB300 (sm_103a) tiled GEMM / Linear-layer library.

The compute path is the C-ABI shared library built from ``csrc/`` (declared
in ``include/gemm.h``); ``dnn_linear_layers_gb300.gemm`` is its thin ctypes
binding.  The library is loaded on the first call into the binding, which
raises if it has not been built.
"""
__all__ = ["gemm", "inputs", "roofline", "build"]
