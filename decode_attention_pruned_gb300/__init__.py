"""Decode attention over a LeanK-pruned KV cache, native to GB300 (sm_103a).

The compute path is the C-ABI library ``_build/libleank.so`` (CUDA kernels,
declared in ``include/leank.h``); ``binding`` is its thin ctypes wrapper and
``synth`` draws seeded inputs.  Nothing here computes attention on the CPU.
"""
from .binding import Cache, LeankError, Plan, load  # noqa: F401

__all__ = ["Cache", "LeankError", "Plan", "load"]
