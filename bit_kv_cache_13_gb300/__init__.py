"""Rotated low-bit KV-cache quantisation and fused packed-cache decode
attention for GB300 (sm_103a).

The compute path is libkvq.so (include/kvq.h); `_lib` binds it with ctypes,
`inputs` draws seeded synthetic workloads and `workload` sets up paged
caches on the device through the library's own append calls.
"""
from . import inputs  # noqa: F401
