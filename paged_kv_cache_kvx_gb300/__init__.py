"""GB300-native paged KV-cache block transfer: run encoding, dense-group
planning, arithmetic rebuild and pack/unpack as sm_103a CUDA kernels behind
a C ABI (include/kvx.h, libkvx.so).  ``kvx`` is the ctypes binding,
``workloads`` the seeded synthetic inputs, ``build`` the in-tree build."""

__all__ = ["build", "kvx", "workloads"]
