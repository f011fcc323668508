"""Averis mean-residual split NVFP4 linear layer for B300 (sm_103a).

The compute path is the C-ABI library ``libaveris.so`` (hand-written CUDA:
fused mean-split quantize pass, rank-one GEMV, tcgen05 block-scaled FP4 GEMM
with the Averis epilogue).  ``capi`` binds it through ctypes; ``layout``
describes its NVFP4 storage; ``build`` compiles it in-tree.
"""

from . import layout  # noqa: F401

__all__ = ["capi", "layout", "build"]
