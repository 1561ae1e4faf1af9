"""GB300-native dense GEMM / GEMV / expert-ID matmul.

The product is the C-ABI library ``libgbmm.so`` (include/gbmm.h), built
in-tree by ``gemv_moe_expert_gb300.build.build()`` for sm_103a.
``binding`` is its ctypes binding (same function names, argument marshalling
only); ``synth`` draws the seeded synthetic inputs.
"""

from . import binding  # noqa: F401  (loads libgbmm.so lazily, on first call)

__all__ = ["binding"]
