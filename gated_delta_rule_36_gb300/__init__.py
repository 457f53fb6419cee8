"""GB300 (sm_103a) Kimi Delta Attention chunked prefill forward.

Public API (thin ctypes binding of ``include/kda.h``):
  kda_fwd, kda_workspace_size, kda_read_device_status, fwd, kda_fwd_no_alloc,
  kda_fwd_host (host buffers), kda_fwd_host_device_bytes, kda_decode (one token per sequence),
  kda_fwd_schedule (the launch schedule for a unit count), kda_fwd_set_trace (chain trace)
"""
from .binding import (KDAError, fwd, kda_decode, kda_fwd, kda_fwd_host, kda_fwd_host_device_bytes,  # noqa: F401
                      kda_fwd_host_workspace_offset, kda_fwd_no_alloc, kda_fwd_schedule, kda_fwd_set_trace, kda_read_device_status,
                      kda_workspace_size, load, library_path)

__all__ = ["KDAError", "fwd", "kda_decode", "kda_fwd", "kda_fwd_host", "kda_fwd_host_device_bytes", "kda_fwd_host_workspace_offset",
           "kda_fwd_no_alloc", "kda_fwd_schedule", "kda_fwd_set_trace", "kda_read_device_status", "kda_workspace_size", "load", "library_path"]
