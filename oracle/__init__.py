"""fp64 CPU oracle for SWA(w,s) -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never links, loads or
calls it, and this package imports nothing from the CUDA side.

The arithmetic lives in ``swa_oracle.c`` (plain C, fp64, OpenMP over output
rows); this module compiles it with gcc and wraps it with ctypes.  Inputs are
16-bit floating-point bit patterns (``numpy.uint16``), bf16 or IEEE fp16:
torch tensors say which by their dtype, bare bit arrays are bf16 unless
``dtype="f16"`` is passed.  Outputs are float64.  ``W_INF`` (-1) stands for
an infinite window (full causal attention).

Definition followed: "Sliding-window beats linear attention" (paper summary
page), section "Prerequisites / Sliding-window attention SWA(w, s)": the window
equation for x_t and the SWA(w,s) notation (first s tokens plus the latest w-s
tokens, softmax normalised only over them, scale 1/sqrt(d)).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "swa_oracle.c")
DEFAULT_LIB = os.path.join(_HERE, "_build", "liboracle_swa.so")

W_INF = -1

# element types (the C source's ORACLE_BF16, ORACLE_F16)
DTYPES = {"bf16": 0, "f16": 1}

_i64 = ctypes.c_int64
_int = ctypes.c_int
_p = ctypes.c_void_p


def compile_source(src_path: str, out_path: str) -> str:
    """Compile an oracle source file to a shared library (gcc, -O2, OpenMP)."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", src_path, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Build the default oracle library if it is missing or older than its source."""
    if (force or not os.path.exists(DEFAULT_LIB)
            or os.path.getmtime(DEFAULT_LIB) < os.path.getmtime(SOURCE)):
        compile_source(SOURCE, DEFAULT_LIB)
    return DEFAULT_LIB


def bits16(x) -> np.ndarray:
    """Bit patterns of a torch bf16 or fp16 tensor (or pass a uint16 array through)."""
    if isinstance(x, np.ndarray):
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x)
    import torch
    assert x.dtype in (torch.bfloat16, torch.float16)
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def bf16_bits(x) -> np.ndarray:
    """bf16 bit patterns of a torch bf16 tensor (or pass a uint16 array through)."""
    if not isinstance(x, np.ndarray):
        import torch
        assert x.dtype == torch.bfloat16
    return bits16(x)


def dtype_code(x, dtype: str | None = None) -> int:
    """Element-type code of an input: ``dtype`` if given, else the tensor's
    dtype (bare uint16 arrays are bf16)."""
    if dtype is not None:
        return DTYPES[dtype]
    if isinstance(x, np.ndarray):
        return DTYPES["bf16"]
    import torch
    return DTYPES["f16"] if x.dtype == torch.float16 else DTYPES["bf16"]


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_p)


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, lib_path: str | None = None):
        self.path = lib_path or build()
        L = ctypes.CDLL(self.path)
        L.oracle_in_window.argtypes = [_i64, _i64, _i64, _i64]
        L.oracle_in_window.restype = _int
        L.oracle_cache_slot.argtypes = [_i64, _i64, _i64]
        L.oracle_cache_slot.restype = _i64
        L.oracle_set_threads.argtypes = [_int]
        L.oracle_get_threads.restype = _int
        L.oracle_swa_prefill.argtypes = [_p, _p, _p, _p, _p] + [_i64] * 7 + [_p, _p, _int, _int]
        L.oracle_swa_prefill.restype = _int
        L.oracle_swa_prefill_rows.argtypes = ([_p, _p, _p, _p, _i64, _p, _p] + [_i64] * 7
                                              + [_p, _p, _int, _int])
        L.oracle_swa_prefill_rows.restype = _int
        L.oracle_swa_decode.argtypes = [_p, _p, _p, _p, _p] + [_i64] * 7 + [_p, _p, _int, _int]
        L.oracle_swa_decode.restype = _int
        L.oracle_cache_append.argtypes = [_p, _p, _p, _p] + [_i64] * 8
        L.oracle_cache_append.restype = _int
        L.oracle_swa_decode_cache.argtypes = ([_p, _p, _p, _p, _p] + [_i64] * 7
                                              + [_p, _p, _int, _int])
        L.oracle_swa_decode_cache.restype = _int
        L.oracle_hybrid_decode.argtypes = ([_p, _p, _p, _p, _p, _p] + [_i64] * 8
                                           + [_p, _p, _int, _int])
        L.oracle_hybrid_decode.restype = _int
        L.oracle_hybrid_state.argtypes = [_p, _p, _p, _p, _p] + [_i64] * 7 + [_p, _int, _int]
        L.oracle_hybrid_state.restype = _int
        self.lib = L

    # -- set and slot definitions -------------------------------------------------
    def in_window(self, t: int, i: int, w: int, s: int) -> bool:
        return bool(self.lib.oracle_in_window(t, i, w, s))

    def window(self, t: int, w: int, s: int) -> list[int]:
        return [i for i in range(t + 1) if self.in_window(t, i, w, s)]

    def cache_slot(self, p: int, w: int, s: int) -> int:
        return int(self.lib.oracle_cache_slot(p, w, s))

    # -- attention ----------------------------------------------------------------
    def threads(self, n: int | None) -> int:
        return n if n and n > 0 else max(1, int(self.lib.oracle_get_threads()))

    def prefill(self, q, k, v, w: int, s: int, threads: int | None = None,
                dtype: str | None = None):
        """All rows.  q [B,L,Hq,d], k/v [B,L,Hkv,d] 16-bit -> (o [B,L,Hq,d], lse [B,Hq,L])."""
        dt = dtype_code(q, dtype)
        q, k, v = bits16(q), bits16(k), bits16(v)
        B, L, Hq, d = q.shape
        Hkv = k.shape[2]
        nt = self.threads(threads)
        o = np.empty((B, L, Hq, d), np.float64)
        lse = np.empty((B, Hq, L), np.float64)
        wi = np.empty(nt * max(L, 1), np.int64)
        ws = np.empty(nt * max(L, 1), np.float64)
        rc = self.lib.oracle_swa_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                         B, L, Hq, Hkv, d, w, s, _ptr(wi), _ptr(ws), nt, dt)
        if rc != 0:
            raise ValueError("oracle_swa_prefill rejected its arguments")
        return o, lse

    def prefill_rows(self, q, k, v, rows, w: int, s: int, threads: int | None = None,
                     dtype: str | None = None):
        """Selected rows: rows is an (n, 3) int array of (b, t, h) -> (o [n,d], lse [n])."""
        dt = dtype_code(q, dtype)
        q, k, v = bits16(q), bits16(k), bits16(v)
        B, L, Hq, d = q.shape
        Hkv = k.shape[2]
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
        n = rows.shape[0]
        nt = self.threads(threads)
        o = np.empty((n, d), np.float64)
        lse = np.empty(n, np.float64)
        wi = np.empty(nt * max(L, 1), np.int64)
        ws = np.empty(nt * max(L, 1), np.float64)
        rc = self.lib.oracle_swa_prefill_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(rows), n, _ptr(o),
                                              _ptr(lse), B, L, Hq, Hkv, d, w, s, _ptr(wi),
                                              _ptr(ws), nt, dt)
        if rc != 0:
            raise ValueError("oracle_swa_prefill_rows rejected its arguments")
        return o, lse

    def decode(self, q, k_hist, v_hist, pos, w: int, s: int, threads: int | None = None,
               dtype: str | None = None):
        """q [B,Hq,d] at positions pos [B] over history k/v [B,P,Hkv,d] -> o [B,Hq,d]."""
        dt = dtype_code(q, dtype)
        q, k_hist, v_hist = bits16(q), bits16(k_hist), bits16(v_hist)
        B, Hq, d = q.shape
        P, Hkv = k_hist.shape[1], k_hist.shape[2]
        pos = np.ascontiguousarray(np.asarray(pos, dtype=np.int64).reshape(B))
        nt = self.threads(threads)
        o = np.empty((B, Hq, d), np.float64)
        wi = np.empty(nt * max(P, 1), np.int64)
        ws = np.empty(nt * max(P, 1), np.float64)
        rc = self.lib.oracle_swa_decode(_ptr(q), _ptr(k_hist), _ptr(v_hist), _ptr(pos), _ptr(o),
                                        B, P, Hq, Hkv, d, w, s, _ptr(wi), _ptr(ws), nt, dt)
        if rc != 0:
            raise ValueError("oracle_swa_decode rejected its arguments")
        return o

    # -- cache --------------------------------------------------------------------
    def cache_append(self, cache_k: np.ndarray, cache_v: np.ndarray, k_new, v_new,
                     pos0: int, w: int, s: int) -> None:
        """In place: cache [B,Hkv,cap,d] uint16, k_new/v_new [B,n,Hkv,d] 16-bit patterns
        (copied bit for bit, whatever their type)."""
        k_new, v_new = bits16(k_new), bits16(v_new)
        assert cache_k.dtype == np.uint16 and cache_k.flags.c_contiguous
        assert cache_v.dtype == np.uint16 and cache_v.flags.c_contiguous
        B, Hkv, cap, d = cache_k.shape
        n = k_new.shape[1]
        rc = self.lib.oracle_cache_append(_ptr(cache_k), _ptr(cache_v), _ptr(k_new), _ptr(v_new),
                                          B, Hkv, d, cap, w, s, n, pos0)
        if rc != 0:
            raise ValueError("oracle_cache_append: a slot falls outside the cache")

    def decode_cache(self, q, cache_k, cache_v, pos, w: int, s: int, threads: int | None = None,
                     dtype: str | None = None):
        """q [B,Hq,d] over the filled slots of cache [B,Hkv,cap,d] -> o [B,Hq,d]."""
        dt = dtype_code(q, dtype)
        q, cache_k, cache_v = bits16(q), bits16(cache_k), bits16(cache_v)
        B, Hq, d = q.shape
        Hkv, cap = cache_k.shape[1], cache_k.shape[2]
        pos = np.ascontiguousarray(np.asarray(pos, dtype=np.int64).reshape(B))
        nt = self.threads(threads)
        o = np.empty((B, Hq, d), np.float64)
        wi = np.empty(nt * max(cap, 1), np.int64)
        ws = np.empty(nt * max(cap, 1), np.float64)
        rc = self.lib.oracle_swa_decode_cache(_ptr(q), _ptr(cache_k), _ptr(cache_v), _ptr(pos),
                                              _ptr(o), B, Hq, Hkv, d, cap, w, s, _ptr(wi),
                                              _ptr(ws), nt, dt)
        if rc != 0:
            raise ValueError("oracle_swa_decode_cache rejected its arguments")
        return o


    # -- hybrid window + linear attention -----------------------------------------
    def hybrid_decode(self, q, k_hist, v_hist, W, pos, w: int, s: int,
                      threads: int | None = None, dtype: str | None = None):
        """q [B,Hq,d] at positions pos [B] over history k/v [B,P,Hkv,d] with the
        feature weights W [Hkv,d,df] -> o [B,Hq,d] (softmax over A(t) plus the
        linear part over the earlier positions outside it)."""
        dt = dtype_code(q, dtype)
        q, k_hist, v_hist = bits16(q), bits16(k_hist), bits16(v_hist)
        W = np.ascontiguousarray(np.asarray(W, np.float64))
        B, Hq, d = q.shape
        P, Hkv = k_hist.shape[1], k_hist.shape[2]
        df = W.shape[2]
        pos = np.ascontiguousarray(np.asarray(pos, dtype=np.int64).reshape(B))
        nt = self.threads(threads)
        o = np.empty((B, Hq, d), np.float64)
        wi = np.empty(nt * max(P, 1), np.int64)
        ws = np.empty(nt * (max(P, 1) + 4 * df), np.float64)
        rc = self.lib.oracle_hybrid_decode(_ptr(q), _ptr(k_hist), _ptr(v_hist), _ptr(W), _ptr(pos),
                                           _ptr(o), B, P, Hq, Hkv, d, df, w, s, _ptr(wi), _ptr(ws),
                                           nt, dt)
        if rc != 0:
            raise ValueError("oracle_hybrid_decode rejected its arguments")
        return o

    def hybrid_state(self, k_hist, v_hist, W, w: int, s: int, threads: int | None = None,
                     dtype: str | None = None):
        """Linear state after positions 0..P-1 of k/v [B,P,Hkv,d] were appended:
        S [B,Hkv,2df,d] and z [B,Hkv,2df] (sums over the evicted positions)."""
        dt = dtype_code(k_hist, dtype)
        k_hist, v_hist = bits16(k_hist), bits16(v_hist)
        W = np.ascontiguousarray(np.asarray(W, np.float64))
        B, P, Hkv, d = k_hist.shape
        df = W.shape[2]
        nt = self.threads(threads)
        S = np.empty((B, Hkv, 2 * df, d), np.float64)
        z = np.empty((B, Hkv, 2 * df), np.float64)
        ws = np.empty(nt * 2 * df, np.float64)
        rc = self.lib.oracle_hybrid_state(_ptr(k_hist), _ptr(v_hist), _ptr(W), _ptr(S), _ptr(z), B, P,
                                          Hkv, d, df, w, s, _ptr(ws), nt, dt)
        if rc != 0:
            raise ValueError("oracle_hybrid_state rejected its arguments")
        return S, z


_default: Oracle | None = None


def get() -> Oracle:
    """The oracle built from this directory's source (built on first use)."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default
