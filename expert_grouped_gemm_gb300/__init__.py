"""GB300-native MoE expert block: forward, retention select, backward.

The compute lives in libmoe_gb300.so (hand-written sm_103a CUDA behind the C
ABI of include/moe.h); this package holds the thin ctypes binding (``_lib``),
the layer wrapper (``layer``), the build step (``build``) and the seeded
synthetic input generator (``inputs``).
"""
from . import inputs  # noqa: F401

__all__ = ["inputs"]
