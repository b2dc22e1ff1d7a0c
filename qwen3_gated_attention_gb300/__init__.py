"""GB300-native (sm_103a) gated full-attention decoder layer: decode and
speculative-verify steps through a C-ABI CUDA library (``libgattn.so``).

``gattn``   ctypes binding of include/gattn.h (same names, marshalling only)
``device``  torch-owned device buffers around one layer handle
``synth``   seeded synthetic inputs
``build``   nvcc build of the library
"""
from . import synth  # noqa: F401

__all__ = ["synth", "gattn", "device", "build"]
