"""Batched speculative-decoding verify-and-sample epilogue for one GB300 (sm_103a).

The computation lives in libdspark.so (hand-written CUDA, C ABI in include/dspark.h);
this package builds it in-tree and binds it with ctypes.  Importing the binding raises if
the library is missing: there is no CPU or PyTorch fallback.
"""
from .build import build, LIB  # noqa: F401
from .binding import (  # noqa: F401
    dspark_host_workspace_bytes,
    dspark_launches_per_call,
    dspark_status_string,
    dspark_verify_sample,
    dspark_verify_sample_host,
    dspark_workspace_bytes,
    load_library,
)
