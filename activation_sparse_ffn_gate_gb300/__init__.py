"""GB300-native (sm_103a) activation-sparse gated FFN with the tile-wise ELL (TwELL) format.

The compute path is libtwell_gb300.so (hand-written CUDA, C ABI in include/twell.h); this package
holds its build script, a thin ctypes binding with the C names, and seeded synthetic layers.
"""
from . import synthetic  # noqa: F401  (pure input construction; no CUDA needed)

__all__ = ["binding", "build", "synthetic"]
