"""GB300-native Medusa verify step: a C-ABI CUDA library (libmedusa) and its thin binding.

Submodules:
  binding  ctypes marshalling of the entry points declared in include/medusa.h
  step     device buffers and the ordered five-call step
  configs  the synthetic workloads (sizes only)
  synth    seeded input generators (Philox4x32-10 uniforms, normal draws)
  _build   in-tree nvcc build of libmedusa.so for sm_103a
"""
from . import configs  # noqa: F401
