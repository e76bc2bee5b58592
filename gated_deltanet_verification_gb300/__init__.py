"""Closed-form Gated DeltaNet tree verification for GB300 (sm_103a).

Modules:
  bole    -- ctypes binding of the C ABI in include/bole.h (libbole.so)
  device  -- device copies of a packed forest and one verify + commit round
  inputs  -- seeded synthetic workloads (trees, operands); no method arithmetic
  build   -- nvcc build of the in-tree library
"""
__all__ = ["bole", "device", "inputs", "build"]
