"""GB300-native fused multi-head attention forward (sm_103a).

The compute path is the CUDA library ``libfmha.so`` built from ``csrc/``;
``binding`` is a thin ctypes layer over its C ABI (``include/fmha.h``).
``workloads`` holds the seeded synthetic inputs.  Importing this package does
not load the CUDA library; ``binding.lib()`` does, and raises if the library
is missing -- there is no CPU fallback.
"""
__all__ = ["binding", "workloads", "build"]
