"""SWA(w,s) -- sliding-window softmax attention with attention sinks on GB300.

Public calls (all run in the package's CUDA library, on the current torch
stream): ``prefill``, ``prefill_chunk`` (a prompt continued from a cache),
``Cache`` (with ``Cache.append``), ``decode``, ``device_error``.  ``W_INF``
selects the infinite window (full causal).
"""
from .swa import (W_INF, Cache, SwaError, decode, decode_workspace_bytes, device_error, lib,
                  prefill, prefill_chunk, prefill_chunk_workspace_bytes, status_string,
                  workspace_for)

__all__ = ["W_INF", "Cache", "SwaError", "decode", "decode_workspace_bytes", "device_error",
           "lib", "prefill", "prefill_chunk", "prefill_chunk_workspace_bytes", "status_string",
           "workspace_for"]
