"""fp4_kv_cache_kvq_gb300 -- FP4 (E2M1 + E4M3 per 16 channels) KV cache and
split-K decode attention for GB300 (sm_103a).

The compute lives in libkvq.so (C ABI, include/kvq.h); ``kvq`` is its thin
ctypes binding, ``workloads`` the seeded synthetic inputs, ``build`` the nvcc
build step.  Importing the package does not load the CUDA library.
"""
from . import workloads  # noqa: F401

__all__ = ["kvq", "workloads", "build"]
