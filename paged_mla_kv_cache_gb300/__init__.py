"""GB300-native paged MLA KV-cache gather.

The compute lives in ``csrc/pmg_gather.cu`` (hand-written sm_103a kernels
behind a C ABI, declared in ``include/pmg.h``); ``binding`` loads that shared
library with ctypes and marshals torch tensors into its plain-pointer calls.
Importing this package does not load the library; the first call does, and it
raises if the library is missing.
"""
from .binding import (  # noqa: F401
    PmgError, gather, debug_plan, select_path, status_string, library_path, load_library,
)

__all__ = ["PmgError", "gather", "debug_plan", "select_path", "status_string", "library_path", "load_library"]
