"""tgemm: a tiled dense GEMM (C = A*B) for one NVIDIA GB300, sm_103a.

The compute path is the C-ABI library ``_build/libtgemm.so`` (hand-written
tcgen05/TMA kernels); ``tgemm`` is its Python binding and ``inputs`` the
seeded synthetic operand generator.
"""
from . import inputs  # noqa: F401

__all__ = ["inputs", "tgemm", "build"]
