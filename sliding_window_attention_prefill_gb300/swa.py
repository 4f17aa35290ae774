"""Python binding of libswa: argument marshalling over the C ABI in include/swa.h.

Every step of the computation runs in the library's CUDA kernels; this module
only checks tensor properties, passes raw device pointers and sizes, and uses
the current torch stream.  If the library has not been built, every call
raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

from . import build as _build

W_INF = -1

# swa_dtype codes of the 16-bit element types
DTYPE_CODES = {torch.bfloat16: 0, torch.float16: 1}

_c_int = ctypes.c_int
_c_i32 = ctypes.c_int32
_c_i64 = ctypes.c_int64
_c_size = ctypes.c_size_t
_c_p = ctypes.c_void_p


class SwaCacheStruct(ctypes.Structure):
    """Mirror of ``swa_cache``."""
    _fields_ = [("k", _c_p), ("v", _c_p), ("B", _c_i32), ("Hkv", _c_i32), ("d", _c_i32),
                ("cap", _c_i32), ("w", _c_i32), ("s", _c_i32), ("dtype", _c_i32)]


class SwaLinearStateStruct(ctypes.Structure):
    """Mirror of ``swa_linear_state``."""
    _fields_ = [("S", _c_p), ("z", _c_p), ("W", _c_p), ("B", _c_i32), ("Hkv", _c_i32), ("d", _c_i32),
                ("df", _c_i32)]


STATUS = {0: "SWA_OK", -1: "SWA_ERR_INVALID_ARG", -2: "SWA_ERR_UNSUPPORTED",
          -3: "SWA_ERR_ALIGNMENT", -4: "SWA_ERR_WORKSPACE", -5: "SWA_ERR_CUDA",
          -6: "SWA_ERR_TIMEOUT", -7: "SWA_ERR_BOUNDS"}


def status_string(status: int) -> str:
    return STATUS.get(int(status), f"SWA_ERR_UNKNOWN({status})")


class SwaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lib = None


def library_path() -> str:
    return _build.LIB


def _declare(L) -> None:
    P = ctypes.POINTER
    L.swa_prefill.argtypes = [_c_p, _c_p, _c_p, _c_p, _c_p] + [_c_int] * 7 + [_c_p]
    L.swa_prefill.restype = _c_int
    L.swa_prefill_ex.argtypes = [_c_p, _c_p, _c_p, _c_p, _c_p] + [_c_int] * 8 + [_c_p]
    L.swa_prefill_ex.restype = _c_int
    L.swa_cache_append.argtypes = [P(SwaCacheStruct), _c_p, _c_p, _c_int, _c_i64, _c_p]
    L.swa_cache_append.restype = _c_int
    L.swa_decode_workspace_bytes.argtypes = [_c_int] * 6
    L.swa_decode_workspace_bytes.restype = _c_size
    L.swa_decode.argtypes = [_c_p, P(SwaCacheStruct), _c_p, _c_int, _c_int, _c_int, _c_p, _c_p,
                             _c_size, _c_p]
    L.swa_decode.restype = _c_int
    L.swa_append_decode.argtypes = [_c_p, _c_p, _c_p, P(SwaCacheStruct), _c_p, _c_int, _c_int,
                                    _c_int, _c_p, _c_p, _c_size, _c_p]
    L.swa_append_decode.restype = _c_int
    L.swa_status_string.argtypes = [_c_int]
    L.swa_status_string.restype = ctypes.c_char_p
    L.swa_get_device_error.argtypes = [_c_p]
    L.swa_get_device_error.restype = _c_int
    L.swa_check_prefill.argtypes = [_c_p, _c_p, _c_p, _c_p, _c_p] + [_c_int] * 7
    L.swa_check_prefill.restype = _c_int
    L.swa_check_append.argtypes = [P(SwaCacheStruct), _c_p, _c_p, _c_int, _c_i64]
    L.swa_check_append.restype = _c_int
    L.swa_check_decode.argtypes = [_c_p, P(SwaCacheStruct), _c_p, _c_int, _c_int, _c_int, _c_p,
                                   _c_p, _c_size, _c_size]
    L.swa_check_decode.restype = _c_int
    L.swa_cache_slot.argtypes = [_c_i64, _c_int, _c_int]
    L.swa_cache_slot.restype = _c_i64
    L.swa_version.argtypes = []
    L.swa_version.restype = ctypes.c_char_p
    L.swa_last_cuda_error.argtypes = []
    L.swa_last_cuda_error.restype = ctypes.c_char_p
    L.swa_debug_bounds_checked.argtypes = []
    L.swa_debug_bounds_checked.restype = _c_int
    L.swa_debug_bounds_index.argtypes = [_c_p]
    L.swa_debug_bounds_index.restype = _c_i64
    L.swa_debug_set_extent_margin.argtypes = [_c_i64]
    L.swa_debug_set_extent_margin.restype = _c_int
    L.swa_selftest_wait_timeout.argtypes = [_c_p]
    L.swa_selftest_wait_timeout.restype = _c_int
    L.swa_prefill_chunk_workspace_bytes.argtypes = [_c_int, _c_int, _c_int, _c_int, _c_int, _c_i64]
    L.swa_prefill_chunk_workspace_bytes.restype = _c_size
    L.swa_prefill_chunk.argtypes = [_c_p, _c_p, _c_p, _c_p, _c_p, P(SwaCacheStruct), _c_int, _c_i64,
                                    _c_int, _c_p, _c_size, _c_p]
    L.swa_prefill_chunk.restype = _c_int
    L.swa_check_prefill_chunk.argtypes = [_c_p, _c_p, _c_p, _c_p, _c_p, P(SwaCacheStruct), _c_int,
                                          _c_i64, _c_int, _c_p, _c_size]
    L.swa_check_prefill_chunk.restype = _c_int
    L.swa_hybrid_append.argtypes = [P(SwaCacheStruct), P(SwaLinearStateStruct), _c_p, _c_p, _c_int,
                                    _c_i64, _c_p]
    L.swa_hybrid_append.restype = _c_int
    L.swa_hybrid_decode_workspace_bytes.argtypes = [_c_int] * 6
    L.swa_hybrid_decode_workspace_bytes.restype = _c_size
    L.swa_hybrid_decode.argtypes = [_c_p, P(SwaCacheStruct), P(SwaLinearStateStruct), _c_p, _c_int,
                                    _c_int, _c_int, _c_p, _c_p, _c_size, _c_p]
    L.swa_hybrid_decode.restype = _c_int
    L.swa_prefill_varlen_workspace_bytes.argtypes = [_c_int] * 4
    L.swa_prefill_varlen_workspace_bytes.restype = _c_size
    L.swa_prefill_varlen.argtypes = ([_c_p] * 6 + [_c_int] * 9 + [_c_p, _c_size, _c_p])
    L.swa_prefill_varlen.restype = _c_int
    L.swa_check_prefill_varlen.argtypes = ([_c_p] * 6 + [_c_int] * 9 + [_c_p, _c_size])
    L.swa_check_prefill_varlen.restype = _c_int


def lib():
    """The loaded library (loaded once; raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"the CUDA library is not built ({path} missing): run "
                "`python -m sliding_window_attention_prefill_gb300.build`")
        L = ctypes.CDLL(path)
        _declare(L)
        _lib = L
    return _lib


def load_checked():
    """The bounds-checked debug build of the library (built on first use),
    loaded beside the normal one and declared the same way.  To run the
    package's calls on it, assign it to ``swa._lib``."""
    path = _build.build_checked()
    L = ctypes.CDLL(path)
    _declare(L)
    return L


def declared_functions() -> list[str]:
    """Names of the functions include/swa.h declares."""
    text = open(os.path.join(_build.INCLUDE, "swa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(swa_[a-z_0-9]+)\s*\(", text)))


def _check(status: int, what: str) -> None:
    if status != 0:
        if status == -5:
            what = f"{what} [{lib().swa_last_cuda_error().decode(errors='replace')}]"
        raise SwaError(status, what)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dtype_code(dtype) -> int:
    if dtype not in DTYPE_CODES:
        raise TypeError(f"element type must be torch.bfloat16 or torch.float16, got {dtype}")
    return DTYPE_CODES[dtype]


def _need(t: torch.Tensor, name: str, dtype=torch.bfloat16) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _out(out, q: torch.Tensor, dtype) -> torch.Tensor:
    """The output tensor: a new one like q, or `out` checked to have q's shape
    (the kernels write that many elements through a plain pointer) and the
    type, device and layout every call needs."""
    if out is None:
        return torch.empty_like(q)
    if not isinstance(out, torch.Tensor):
        raise TypeError("out must be a torch.Tensor")
    if out.shape != q.shape:
        raise ValueError(f"out must have the shape of q {tuple(q.shape)}, got {tuple(out.shape)}")
    _need(out, "out", dtype)
    return out


# ----------------------------------------------------------------------------- prefill
def prefill(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, w: int, s: int,
            out: torch.Tensor | None = None, return_lse: bool = False):
    """SWA(w,s) attention of every prompt position.

    q [B, L, Hq, d], k/v [B, L, Hkv, d] CUDA tensors, all bf16 or all fp16;
    returns o [B, L, Hq, d] of the same type (and lse [B, Hq, L] fp32 if
    ``return_lse``).  ``w = W_INF`` is full causal.
    """
    if not isinstance(q, torch.Tensor):
        raise TypeError("q must be a torch.Tensor")
    dt = _dtype_code(q.dtype)
    _need(q, "q", q.dtype), _need(k, "k", q.dtype), _need(v, "v", q.dtype)
    B, L, Hq, d = q.shape
    if k.shape[:2] != (B, L) or k.shape[3] != d or v.shape != k.shape:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)}, k {tuple(k.shape)}, v {tuple(v.shape)}")
    Hkv = k.shape[2]
    o = _out(out, q, q.dtype)
    lse = torch.empty(B, Hq, L, dtype=torch.float32, device=q.device) if return_lse else None
    st = lib().swa_prefill_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, L, Hq, Hkv, d,
                              int(w), int(s), dt, _stream(q.device))
    _check(st, "swa_prefill_ex")
    return (o, lse) if return_lse else o


# ----------------------------------------------------------------------------- varlen prefill
_varlen_workspaces: dict = {}


def prefill_varlen_workspace_bytes(B: int, total: int, Hq: int, Hkv: int) -> int:
    return int(lib().swa_prefill_varlen_workspace_bytes(B, total, Hq, Hkv))


def prefill_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens: torch.Tensor,
                   w: int, s: int, max_len: int | None = None, out: torch.Tensor | None = None,
                   return_lse: bool = False, workspace: torch.Tensor | None = None):
    """SWA(w,s) prefill of a ragged batch packed along the first dimension.

    q [total, Hq, d], k/v [total, Hkv, d] CUDA tensors (bf16 or fp16);
    cu_seqlens int32 CUDA tensor [B+1] (sequence b is rows cu_seqlens[b] ..
    cu_seqlens[b+1]-1).  Returns o [total, Hq, d] (and lse [Hq, total] fp32
    if ``return_lse``).  ``max_len`` bounds the sequence lengths (default:
    total); it only picks the key tile width for w = W_INF.
    """
    if not isinstance(q, torch.Tensor):
        raise TypeError("q must be a torch.Tensor")
    dt = _dtype_code(q.dtype)
    _need(q, "q", q.dtype), _need(k, "k", q.dtype), _need(v, "v", q.dtype)
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    if q.dim() != 3 or k.dim() != 3 or k.shape != v.shape or k.shape[0] != q.shape[0] or k.shape[2] != q.shape[2]:
        raise ValueError(f"q must be [total, Hq, d] and k, v [total, Hkv, d]: {tuple(q.shape)}, {tuple(k.shape)}")
    total, Hq, d = q.shape
    Hkv = k.shape[1]
    B = cu_seqlens.numel() - 1
    if B < 1:
        raise ValueError("cu_seqlens needs at least two entries")
    o = _out(out, q, q.dtype)
    lse = torch.empty(Hq, total, dtype=torch.float32, device=q.device) if return_lse else None
    nbytes = prefill_varlen_workspace_bytes(B, total, Hq, Hkv)
    ws = workspace
    if ws is None:
        key = q.device
        ws = _varlen_workspaces.get(key)
        if ws is None or ws.numel() < nbytes:
            ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
            _varlen_workspaces[key] = ws
    st = lib().swa_prefill_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens), B,
                                  total, int(max_len if max_len is not None else total), Hq, Hkv, d,
                                  int(w), int(s), dt, _ptr(ws), ws.numel(), _stream(q.device))
    _check(st, "swa_prefill_varlen")
    return (o, lse) if return_lse else o


# ----------------------------------------------------------------------------- cache
class Cache:
    """One layer's fixed SWA(w,s) cache: k, v [B, Hkv, cap, d] (torch-owned),
    bf16 or fp16 (``dtype``; queries and outputs of the calls on the cache
    have the same type).

    cap = w for a finite window (s sink slots + a (w-s)-slot ring), or
    ``max_len`` for ``w = W_INF``.
    """

    def __init__(self, B: int, Hkv: int, d: int, w: int, s: int, max_len: int | None = None,
                 device="cuda", dtype=torch.bfloat16):
        _dtype_code(dtype)
        if w == W_INF:
            if not max_len:
                raise ValueError("an infinite window needs max_len")
            cap = int(max_len)
        else:
            cap = int(w)
        self.B, self.Hkv, self.d, self.w, self.s, self.cap = B, Hkv, d, int(w), int(s), cap
        self.dtype = dtype
        self.k = torch.zeros(B, Hkv, cap, d, dtype=dtype, device=device)
        self.v = torch.zeros(B, Hkv, cap, d, dtype=dtype, device=device)

    @classmethod
    def from_tensors(cls, k: torch.Tensor, v: torch.Tensor, w: int, s: int) -> "Cache":
        _dtype_code(k.dtype)
        _need(k, "cache k", k.dtype), _need(v, "cache v", k.dtype)
        obj = cls.__new__(cls)
        obj.dtype = k.dtype
        obj.B, obj.Hkv, obj.cap, obj.d = k.shape
        obj.w, obj.s, obj.k, obj.v = int(w), int(s), k, v
        return obj

    def struct(self) -> SwaCacheStruct:
        return SwaCacheStruct(self.k.data_ptr(), self.v.data_ptr(), self.B, self.Hkv, self.d,
                              self.cap, self.w, self.s, DTYPE_CODES[self.dtype])

    def append(self, k_new: torch.Tensor, v_new: torch.Tensor, pos0: int) -> None:
        """Write positions pos0 .. pos0+n-1 from k_new/v_new [B, n, Hkv, d]."""
        _need(k_new, "k_new", self.dtype), _need(v_new, "v_new", self.dtype)
        if (k_new.shape != v_new.shape or k_new.shape[0] != self.B
                or tuple(k_new.shape[2:]) != (self.Hkv, self.d)):
            raise ValueError(f"k_new/v_new must be [B, n, Hkv, d], got {tuple(k_new.shape)}")
        c = self.struct()
        st = lib().swa_cache_append(ctypes.byref(c), _ptr(k_new), _ptr(v_new), k_new.shape[1],
                                    int(pos0), _stream(self.k.device))
        _check(st, "swa_cache_append")


# ----------------------------------------------------------------------------- chunked prefill
_chunk_workspaces: dict = {}


def prefill_chunk_workspace_bytes(B: int, n: int, Hkv: int, d: int, w: int, pos0: int) -> int:
    return int(lib().swa_prefill_chunk_workspace_bytes(B, n, Hkv, d, int(w), int(pos0)))


def prefill_chunk(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cache: "Cache", pos0: int,
                  out: torch.Tensor | None = None, return_lse: bool = False,
                  workspace: torch.Tensor | None = None):
    """Prefill positions pos0 .. pos0+n-1 of a prompt against what ``cache``
    holds of the earlier positions, then append them to the cache.

    q [B, n, Hq, d], k/v [B, n, Hkv, d] CUDA tensors of the cache's type;
    returns o [B, n, Hq, d] (and lse [B, Hq, n] fp32 if ``return_lse``).
    Chunk by chunk this equals one prefill of the whole prompt.
    """
    _need(q, "q", cache.dtype), _need(k, "k", cache.dtype), _need(v, "v", cache.dtype)
    B, n, Hq, d = q.shape
    if (B, d) != (cache.B, cache.d) or k.shape != (B, n, cache.Hkv, d) or v.shape != k.shape:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)}, k {tuple(k.shape)}, cache "
                         f"B={cache.B} Hkv={cache.Hkv} d={cache.d}")
    o = _out(out, q, cache.dtype)
    lse = torch.empty(B, Hq, n, dtype=torch.float32, device=q.device) if return_lse else None
    nbytes = prefill_chunk_workspace_bytes(B, n, cache.Hkv, d, cache.w, pos0)
    ws = workspace
    if ws is None and nbytes > 0:
        key = q.device
        ws = _chunk_workspaces.get(key)
        if ws is None or ws.numel() < nbytes:
            ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
            _chunk_workspaces[key] = ws
    wbytes = 0 if ws is None else ws.numel() * ws.element_size()
    c = cache.struct()
    st = lib().swa_prefill_chunk(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), ctypes.byref(c), n,
                                 int(pos0), Hq, _ptr(ws), wbytes, _stream(q.device))
    _check(st, "swa_prefill_chunk")
    return (o, lse) if return_lse else o


# ----------------------------------------------------------------------------- decode
_workspaces: dict = {}


def decode_workspace_bytes(B: int, Hq: int, Hkv: int, d: int, cap: int, w: int) -> int:
    return int(lib().swa_decode_workspace_bytes(B, Hq, Hkv, d, cap, w))


def workspace_for(cache: "Cache", Hq: int) -> torch.Tensor | None:
    """A (reused) device workspace large enough for decoding with this cache."""
    n = decode_workspace_bytes(cache.B, Hq, cache.Hkv, cache.d, cache.cap, cache.w)
    if n == 0:
        return None
    key = (cache.k.device, n)
    ws = _workspaces.get(key)
    if ws is None:
        ws = torch.empty(n, dtype=torch.uint8, device=cache.k.device)
        _workspaces[key] = ws
    return ws


def decode(q: torch.Tensor, cache: Cache, pos: torch.Tensor, out: torch.Tensor | None = None,
           workspace: torch.Tensor | None = None) -> torch.Tensor:
    """One token per sequence: q [B, Hq, d] (the cache's type) at positions
    pos [B] (int32, device)."""
    _need(q, "q", cache.dtype)
    _need(pos, "pos", torch.int32)
    B, Hq, d = q.shape
    if B != cache.B or d != cache.d or pos.numel() != B:
        raise ValueError("q / pos do not match the cache")
    o = _out(out, q, cache.dtype)
    ws = workspace if workspace is not None else workspace_for(cache, Hq)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    c = cache.struct()
    st = lib().swa_decode(_ptr(q), ctypes.byref(c), _ptr(pos), Hq, cache.w, cache.s, _ptr(o),
                          _ptr(ws), nbytes, _stream(q.device))
    _check(st, "swa_decode")
    return o


def append_decode(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor, cache: Cache,
                  pos: torch.Tensor, out: torch.Tensor | None = None,
                  workspace: torch.Tensor | None = None) -> torch.Tensor:
    """One decode step in one kernel: the new token of each sequence (k_new,
    v_new [B, 1, Hkv, d] or [B, Hkv, d]) goes to its cache slot at position
    pos [B] (int32, device), and q [B, Hq, d] at that position attends to the
    cache -- the same as ``cache.append`` then ``decode``."""
    _need(q, "q", cache.dtype)
    _need(k_new, "k_new", cache.dtype), _need(v_new, "v_new", cache.dtype)
    _need(pos, "pos", torch.int32)
    B, Hq, d = q.shape
    if B != cache.B or d != cache.d or pos.numel() != B:
        raise ValueError("q / pos do not match the cache")
    for t, n in ((k_new, "k_new"), (v_new, "v_new")):
        if t.numel() != B * cache.Hkv * d or t.shape[0] != B or t.shape[-1] != d:
            raise ValueError(f"{n} must be [B, 1, Hkv, d] or [B, Hkv, d], got {tuple(t.shape)}")
    o = _out(out, q, cache.dtype)
    ws = workspace if workspace is not None else workspace_for(cache, Hq)
    nbytes = 0 if ws is None else ws.numel() * ws.element_size()
    c = cache.struct()
    st = lib().swa_append_decode(_ptr(q), _ptr(k_new), _ptr(v_new), ctypes.byref(c), _ptr(pos), Hq,
                                 cache.w, cache.s, _ptr(o), _ptr(ws), nbytes, _stream(q.device))
    _check(st, "swa_append_decode")
    return o


# ----------------------------------------------------------------------------- hybrid
class LinearState:
    """The linear-attention state of a hybrid window + linear layer: S fp32
    [B, Hkv, 2 df, d], z fp32 [B, Hkv, 2 df] (zero: nothing evicted yet) and
    the feature weights W fp32 [Hkv, d, df] of phi(x) = (exp(xW), exp(-xW))."""

    def __init__(self, cache: "Cache", W: torch.Tensor):
        _need(W, "W", torch.float32)
        if W.dim() != 3 or W.shape[0] != cache.Hkv or W.shape[1] != cache.d:
            raise ValueError(f"W must be [Hkv, d, df], got {tuple(W.shape)}")
        self.df = int(W.shape[2])
        self.W = W
        F = 2 * self.df
        self.S = torch.zeros(cache.B, cache.Hkv, F, cache.d, dtype=torch.float32, device=W.device)
        self.z = torch.zeros(cache.B, cache.Hkv, F, dtype=torch.float32, device=W.device)
        self.B, self.Hkv, self.d = cache.B, cache.Hkv, cache.d

    def struct(self) -> SwaLinearStateStruct:
        return SwaLinearStateStruct(self.S.data_ptr(), self.z.data_ptr(), self.W.data_ptr(), self.B,
                                    self.Hkv, self.d, self.df)


def hybrid_append(cache: "Cache", state: LinearState, k_new: torch.Tensor, v_new: torch.Tensor,
                  pos0: int) -> None:
    """Cache.append that first folds the positions it evicts into ``state``."""
    _need(k_new, "k_new", cache.dtype), _need(v_new, "v_new", cache.dtype)
    if (k_new.shape != v_new.shape or k_new.shape[0] != cache.B
            or tuple(k_new.shape[2:]) != (cache.Hkv, cache.d)):
        raise ValueError(f"k_new/v_new must be [B, n, Hkv, d], got {tuple(k_new.shape)}")
    c, st = cache.struct(), state.struct()
    _check(lib().swa_hybrid_append(ctypes.byref(c), ctypes.byref(st), _ptr(k_new), _ptr(v_new),
                                   k_new.shape[1], int(pos0), _stream(cache.k.device)),
           "swa_hybrid_append")


_hybrid_workspaces: dict = {}


def hybrid_decode(q: torch.Tensor, cache: "Cache", state: LinearState, pos: torch.Tensor,
                  out: torch.Tensor | None = None, workspace: torch.Tensor | None = None):
    """decode with the linear part of the evicted positions mixed in."""
    _need(q, "q", cache.dtype)
    _need(pos, "pos", torch.int32)
    B, Hq, d = q.shape
    if B != cache.B or d != cache.d or pos.numel() != B:
        raise ValueError("q / pos do not match the cache")
    o = _out(out, q, cache.dtype)
    n = int(lib().swa_hybrid_decode_workspace_bytes(B, Hq, cache.Hkv, d, cache.cap, cache.w))
    ws = workspace
    if ws is None:
        key = (q.device, n)
        ws = _hybrid_workspaces.get(key)
        if ws is None:
            ws = torch.empty(max(n, 16), dtype=torch.uint8, device=q.device)
            _hybrid_workspaces[key] = ws
    c, st = cache.struct(), state.struct()
    _check(lib().swa_hybrid_decode(_ptr(q), ctypes.byref(c), ctypes.byref(st), _ptr(pos), Hq, cache.w,
                                   cache.s, _ptr(o), _ptr(ws), ws.numel() * ws.element_size(),
                                   _stream(q.device)), "swa_hybrid_decode")
    return o


def selftest_wait_timeout(device=None) -> None:
    """Enqueue the kernel whose bounded wait runs out on purpose (see
    swa_selftest_wait_timeout in include/swa.h); read the result with
    device_error()."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    _check(lib().swa_selftest_wait_timeout(_stream(dev)), "swa_selftest_wait_timeout")


def device_error(device=None) -> int:
    """Synchronise the current stream and read/clear the library's device error word."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    return int(lib().swa_get_device_error(_stream(dev)))
