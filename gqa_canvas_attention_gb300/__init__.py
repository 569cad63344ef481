"""GB300-native (sm_103a) DiffusionGemma canvas-forward attention block.

The compute lives in ``libdgattn.so`` (C ABI: ``include/dg_attn.h``); ``binding`` is its ctypes
binding and ``workloads`` the seeded synthetic inputs.  Importing the package loads nothing; the
library is loaded on first use and its absence is an error, never a fallback.
"""
__all__ = ["binding", "workloads", "build"]
