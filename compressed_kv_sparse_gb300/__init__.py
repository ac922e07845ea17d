"""GB300 (sm_103a) compressed-KV sparse attention layer.

The layer's steps run in libds4a.so (CUDA kernels behind a C ABI, declared in
include/ds4a.h); ``lib`` is the ctypes binding with the same call names.
"""
from . import lib  # noqa: F401
