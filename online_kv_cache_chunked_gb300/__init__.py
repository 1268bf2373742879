"""GB300-native online KV-cache clustering: Chunked Soft Matching compression and
degree-aware decode attention, behind the C ABI in include/csmkv.h.

Modules:
  binding  -- ctypes binding of the C ABI (same names as the C functions)
  pipeline -- host driver of the inference pipeline (budget, trigger, schedule)
  synth    -- seeded synthetic workloads (inputs only, none of the method)
  _build   -- nvcc build of libcsmkv.so for sm_103a
"""
from . import binding  # noqa: F401
from ._build import build  # noqa: F401
