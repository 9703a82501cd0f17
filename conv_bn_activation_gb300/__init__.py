"""Fused convolution + BatchNorm + activation for one GB300 GPU (sm_103a).

``binding`` is the thin ctypes layer over the C ABI (include/cb.h) and loads
libcb.so on first use; ``nets`` builds layers and network chains from those
calls; ``synthetic`` draws the seeded inputs; ``workloads`` holds the
algorithmic byte / FLOP counts used for roofline fractions.
"""
from . import binding  # noqa: F401  (loads libcb.so lazily)

__all__ = ["binding"]
