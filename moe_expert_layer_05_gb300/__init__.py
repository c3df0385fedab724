"""GB300-native Megatron-Core-style MoE expert layer.

The compute lives in libmoe_gb300.so (C ABI, include/moe_gb300.h), hand-written
CUDA for sm_103a; ``api`` is its ctypes binding and ``inputs`` the seeded
synthetic workloads.  Importing the package loads nothing; the library is
loaded on first use.
"""
__all__ = ["api", "inputs", "build"]
