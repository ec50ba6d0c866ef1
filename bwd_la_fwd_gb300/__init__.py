"""GB300-native (sm_103a) normalised linear attention: forward and backward of one LA head batch.

The compute lives in ``csrc/`` (hand-written CUDA, C ABI in ``include/la.h``); ``la.py`` is a thin
ctypes binding over that ABI.  The library is loaded on first use and a missing or stale build raises
an error: there is no CPU fallback.
"""
from .la import (LA_BF16, LA_F32, LAError, la_backward, la_forward, la_get_status, la_launch_count, la_status_string,
                 la_workspace_bytes, library_path, load_library)

__all__ = ["LA_BF16", "LA_F32", "LAError", "la_backward", "la_forward", "la_get_status", "la_launch_count", "la_status_string",
           "la_workspace_bytes", "library_path", "load_library"]
