"""SWA(w,s) -- sliding-window softmax attention with attention sinks on GB300.

Public calls (all run in the package's CUDA library, on the current torch
stream): ``prefill``, ``prefill_varlen`` (a ragged batch packed along the
first dimension), ``prefill_chunk`` (a prompt continued from a cache),
``Cache`` (with ``Cache.append``), ``decode``, ``append_decode`` (append
and decode of one token in one kernel), ``device_error``, and the
hybrid window + linear mode (``LinearState``, ``hybrid_append``,
``hybrid_decode``).  ``W_INF``
selects the infinite window (full causal).  bf16 and fp16 tensors are
accepted (one type per call).
"""
from .swa import (W_INF, Cache, LinearState, SwaError, append_decode, decode, decode_workspace_bytes,
                  device_error, hybrid_append, hybrid_decode, lib, prefill, prefill_chunk,
                  prefill_chunk_workspace_bytes, prefill_varlen, prefill_varlen_workspace_bytes,
                  status_string, workspace_for)

__all__ = ["W_INF", "Cache", "LinearState", "SwaError", "append_decode", "decode",
           "decode_workspace_bytes",
           "device_error", "hybrid_append", "hybrid_decode", "lib", "prefill", "prefill_chunk",
           "prefill_chunk_workspace_bytes", "prefill_varlen", "prefill_varlen_workspace_bytes",
           "status_string", "workspace_for"]
