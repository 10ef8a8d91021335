"""KDA (Kimi Delta Attention) forward for GB300 (sm_103a).

The compute path is the C-ABI library ``libkda.so`` built from ``csrc/``
(``python -m linear_attention_recurrence_fwd_gb300.build``); the functions
exported here are thin ctypes bindings with the same names as the C entry
points in ``include/kda.h``.  There is no CPU fallback: a missing library
raises on first use.
"""
from .binding import (KDAError, kda_chunk_fwd, kda_chunk_fwd_noalloc, kda_decode_step,
                      kda_last_device_status, kda_status_string, kda_varlen_fwd, kda_version)

__all__ = ["KDAError", "kda_chunk_fwd", "kda_chunk_fwd_noalloc", "kda_varlen_fwd",
           "kda_decode_step",
           "kda_last_device_status", "kda_status_string", "kda_version"]
