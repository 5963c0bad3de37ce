"""int4 grouped-GEMM sparse MoE layer for one GB300 (sm_103a).

The compute path is the CUDA library ``libmoe_gb300.so`` (C ABI in
``include/moe.h``); this package holds its ctypes binding (``_lib``), thin
device-resident helpers (``moe``), the nvcc build step (``build``) and the
seeded synthetic-input generators (``synthetic``).
"""
__all__ = ["_lib", "moe", "synthetic", "build"]
