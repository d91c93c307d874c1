"""GB300-native (sm_103a) chunked forward pass of Kimi Delta Attention (KDA).

The compute lives in libkda.so (C ABI declared in include/kda.h); the Python
names below are a thin ctypes binding with the same names.
"""
from .kda import (KdaError, kda_chunk_bwd, kda_chunk_fwd, kda_chunk_fwd_segmented,  # noqa: F401
                  kda_decode_step, kda_device_status, kda_segmented_workspace_size,
                  kda_select_path, load, library_path)

__all__ = ["kda_chunk_fwd", "kda_chunk_bwd", "kda_chunk_fwd_segmented", "kda_segmented_workspace_size",
           "kda_decode_step", "kda_device_status", "kda_select_path", "KdaError", "load",
           "library_path"]
