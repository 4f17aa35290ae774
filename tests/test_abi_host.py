"""Host-side checks of the C ABI (no GPU): the library loads, exports every
function include/swa.h declares, and rejects bad arguments before touching
the device."""
import ctypes

import pytest
import torch

import oracle
from sliding_window_attention_prefill_gb300 import build as swa_build
from sliding_window_attention_prefill_gb300 import swa

OK, INVALID, UNSUPPORTED, ALIGN, WORKSPACE = 0, -1, -2, -3, -4
INF = swa.W_INF


@pytest.fixture(scope="module")
def L():
    swa_build.build()
    return swa.lib()


def test_exports_every_declared_symbol(L):
    names = swa.declared_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/swa.h but not exported"


def test_version_and_status_strings(L):
    assert L.swa_version().decode().count(".") == 2
    for code, name in swa.STATUS.items():
        assert L.swa_status_string(code).decode() == name
    assert L.swa_status_string(-99).decode() == "SWA_ERR_UNKNOWN"


FAKE = 0x10000  # an aligned, never dereferenced address


def _p(off=0):
    return ctypes.c_void_p(FAKE * (1 + off))


def test_check_prefill(L):
    q, k, v, o = _p(0), _p(1000), _p(2000), _p(3000)
    c = L.swa_check_prefill
    assert c(q, k, v, o, None, 1, 256, 4, 1, 64, 64, 4) == OK
    assert c(q, k, v, o, None, 2, 4096, 32, 8, 128, INF, 0) == OK
    assert c(None, None, None, None, None, 0, 10, 4, 1, 64, 64, 4) == OK      # empty batch
    assert c(q, k, v, o, None, 1, 0, 4, 1, 64, 64, 4) == OK                   # empty prompt
    assert c(q, k, v, o, None, 1, 256, 4, 1, 64, 4, 4) == INVALID             # w <= s
    assert c(q, k, v, o, None, 1, 256, 4, 1, 64, 8, -1) == INVALID
    assert c(q, k, v, o, None, 1, 256, 4, 1, 64, 0, 0) == INVALID
    assert c(q, k, v, o, None, 1, 256, 4, 1, 64, -2, 0) == INVALID
    assert c(q, k, v, o, None, 1, 256, 6, 4, 64, 64, 4) == INVALID            # Hq % Hkv
    assert c(q, k, v, o, None, 1, 256, 6, 2, 64, 64, 4) == UNSUPPORTED        # G = 3
    assert c(q, k, v, o, None, 1, 256, 4, 1, 96, 64, 4) == UNSUPPORTED        # d
    assert c(q, k, v, o, None, 1, 256, 4, 1, 64, 128, 65) == UNSUPPORTED      # s > max sinks
    assert c(None, k, v, o, None, 1, 256, 4, 1, 64, 64, 4) == INVALID
    assert c(ctypes.c_void_p(FAKE + 8), k, v, o, None, 1, 256, 4, 1, 64, 64, 4) == ALIGN
    assert c(q, k, v, q, None, 1, 256, 4, 1, 64, 64, 4) == INVALID           # o aliases q
    assert c(q, k, v, o, ctypes.c_void_p(FAKE * 5000 + 2), 1, 256, 4, 1, 64, 64, 4) == ALIGN


def _cache(B=2, Hkv=2, d=128, cap=64, w=64, s=4, k=None, v=None, dtype=0):
    return swa.SwaCacheStruct(k if k is not None else FAKE * 10, v if v is not None else FAKE * 900,
                              B, Hkv, d, cap, w, s, dtype)


def test_element_types(L):
    """bf16 (0) and fp16 (1) are the element types; anything else is rejected
    on the host before any launch."""
    q, k, v, o = _p(1000), _p(2000), _p(3000), _p(4000)
    for bad in (2, -1, 7):
        assert L.swa_prefill_ex(q, k, v, o, None, 1, 256, 4, 1, 64, 64, 4, bad, None) == INVALID
    kn, vn = _p(5000), _p(6000)
    assert L.swa_check_append(ctypes.byref(_cache(dtype=1)), kn, vn, 1, 0) == OK
    assert L.swa_check_append(ctypes.byref(_cache(dtype=2)), kn, vn, 1, 0) == INVALID
    qd, pos, od = _p(7000), _p(7100), _p(7200)
    assert L.swa_check_decode(qd, ctypes.byref(_cache(dtype=1)), pos, 8, 64, 4, od, None, 0, 0) == OK
    assert L.swa_check_decode(qd, ctypes.byref(_cache(dtype=3)), pos, 8, 64, 4, od, None, 0,
                              0) == INVALID
    assert swa.DTYPE_CODES == {torch.bfloat16: 0, torch.float16: 1}


def test_check_append(L):
    c = L.swa_check_append
    kn, vn = _p(5000), _p(6000)
    assert c(ctypes.byref(_cache()), kn, vn, 1, 4096) == OK
    assert c(ctypes.byref(_cache()), kn, vn, 4096, 0) == OK                  # bulk prompt
    assert c(ctypes.byref(_cache()), kn, vn, 0, 0) == OK
    assert c(ctypes.byref(_cache()), kn, vn, -1, 0) == INVALID
    assert c(ctypes.byref(_cache()), kn, vn, 1, -1) == INVALID
    assert c(ctypes.byref(_cache(cap=65)), kn, vn, 1, 0) == INVALID          # cap != w
    assert c(ctypes.byref(_cache(w=INF, s=0, cap=100)), kn, vn, 100, 0) == OK
    assert c(ctypes.byref(_cache(w=INF, s=0, cap=100)), kn, vn, 1, 100) == INVALID  # past cap
    assert c(ctypes.byref(_cache(d=80)), kn, vn, 1, 0) == UNSUPPORTED
    assert c(ctypes.byref(_cache(k=FAKE * 10 + 4)), kn, vn, 1, 0) == ALIGN
    assert c(None, kn, vn, 1, 0) == INVALID
    assert c(ctypes.byref(_cache()), kn, ctypes.c_void_p(FAKE * 10), 1, 0) == INVALID  # aliases cache


def test_check_decode(L):
    c = L.swa_check_decode
    q, pos, o, ws = _p(7000), _p(7100), _p(7200), _p(7300)
    cache = _cache(B=2, Hkv=2, d=128, cap=64, w=64, s=4)
    assert c(q, ctypes.byref(cache), pos, 8, 64, 4, o, None, 0, 0) == OK
    assert c(q, ctypes.byref(cache), pos, 8, 64, 4, o, ws, 1024, 1024) == OK
    assert c(q, ctypes.byref(cache), pos, 8, 64, 4, o, ws, 512, 1024) == WORKSPACE
    assert c(q, ctypes.byref(cache), pos, 8, 64, 4, o, None, 0, 1024) == WORKSPACE
    assert c(q, ctypes.byref(cache), pos, 8, 128, 4, o, None, 0, 0) == INVALID   # w differs
    assert c(q, ctypes.byref(cache), pos, 8, 64, 3, o, None, 0, 0) == INVALID    # s differs
    assert c(q, ctypes.byref(cache), pos, 7, 64, 4, o, None, 0, 0) == INVALID    # Hq % Hkv
    assert c(q, ctypes.byref(cache), pos, 32, 64, 4, o, None, 0, 0) == UNSUPPORTED  # G = 16
    big = _cache(B=1 << 12, Hkv=8, d=128, cap=1 << 16, w=INF, s=0, k=1 << 44, v=1 << 46)
    assert c(q, ctypes.byref(big), pos, 32, INF, 0, o, None, 0, 0) == UNSUPPORTED  # 2^31 rows
    assert c(q, ctypes.byref(cache), ctypes.c_void_p(FAKE * 7100 + 2), 8, 64, 4, o, None, 0, 0) == ALIGN
    assert c(q, ctypes.byref(cache), None, 8, 64, 4, o, None, 0, 0) == INVALID


def test_check_prefill_chunk(L):
    c, wb = L.swa_check_prefill_chunk, L.swa_prefill_chunk_workspace_bytes
    q, kn, vn, o, ws = _p(7000), _p(7400), _p(7500), _p(7600), _p(20000)
    cache = _cache(B=2, Hkv=2, d=128, cap=64, w=64, s=4)
    # finite window: the gathered keys are the cache (min(pos0, w) rows) + the chunk
    assert wb(2, 100, 2, 128, 64, 10) == 2 * 2 * (10 + 100) * 2 * 128 * 2
    assert wb(2, 100, 2, 128, 64, 5000) == 2 * 2 * (64 + 100) * 2 * 128 * 2
    assert wb(2, 100, 2, 128, INF, 5000) == 0                # read in place
    need = wb(2, 100, 2, 128, 64, 5000)
    assert c(q, kn, vn, o, None, ctypes.byref(cache), 100, 5000, 8, ws, need) == OK
    assert c(q, kn, vn, o, None, ctypes.byref(cache), 100, 5000, 8, ws, need - 16) == WORKSPACE
    assert c(q, kn, vn, o, None, ctypes.byref(cache), 100, 5000, 8, None, 0) == WORKSPACE
    assert c(q, kn, vn, o, None, ctypes.byref(cache), 0, 5000, 8, None, 0) == OK     # empty chunk
    assert c(q, kn, vn, o, None, ctypes.byref(cache), -1, 0, 8, ws, need) == INVALID
    assert c(q, kn, vn, o, None, ctypes.byref(cache), 100, -1, 8, ws, need) == INVALID
    assert c(q, kn, vn, o, None, ctypes.byref(cache), 100, 5000, 7, ws, need) == INVALID  # Hq % Hkv
    assert c(q, kn, vn, o, None, ctypes.byref(cache), 100, 5000, 6, ws, need) == UNSUPPORTED  # G=3
    assert c(q, kn, vn, q, None, ctypes.byref(cache), 100, 5000, 8, ws, need) == INVALID  # o aliases q
    assert c(q, kn, vn, o, None, ctypes.byref(cache), 100, 5000, 8, _p(7600), need) == INVALID
    assert c(q, kn, vn, o, None, ctypes.byref(cache), 100, 5000, 8,
             ctypes.c_void_p(FAKE * 20000 + 8), need) == ALIGN
    inf = _cache(B=2, Hkv=2, d=128, cap=300, w=INF, s=0)
    assert c(q, kn, vn, o, None, ctypes.byref(inf), 100, 200, 8, None, 0) == OK
    assert c(q, kn, vn, o, None, ctypes.byref(inf), 100, 201, 8, None, 0) == INVALID  # past cap


def test_slot_map_matches_oracle(L):
    orc = oracle.get()
    for w, s in [(64, 4), (512, 4), (9, 0), (5, 4), (INF, 0), (128, 64)]:
        for p in range(0, 3 * (w if w > 0 else 50)):
            assert L.swa_cache_slot(p, w, s) == orc.cache_slot(p, w, s), (w, s, p)
    assert L.swa_cache_slot(-1, 64, 4) == -1
    assert L.swa_cache_slot(3, 4, 4) == -1


def test_check_prefill_varlen(L):
    c, wb = L.swa_check_prefill_varlen, L.swa_prefill_varlen_workspace_bytes
    q, k, v, o, cu, ws = _p(1000), _p(2000), _p(3000), _p(4000), _p(5000), _p(20000)
    # B=3 sequences, 1000 rows, Hq=32, Hkv=8 (G=4: 32 positions per tile)
    need = wb(3, 1000, 32, 8)
    assert need == 16 + 16 * (3 + (1000 + 31) // 32)
    assert wb(0, 1000, 32, 8) == 0 and wb(3, 1000, 30, 8) == 0
    args = (3, 1000, 600, 32, 8, 128, 64, 4, 0)
    assert c(q, k, v, o, None, cu, *args, ws, need) == OK
    assert c(q, k, v, o, None, cu, *args, ws, need - 16) == WORKSPACE
    assert c(q, k, v, o, None, cu, *args, None, 0) == WORKSPACE
    assert c(q, k, v, o, None, None, *args, ws, need) == INVALID
    assert c(q, k, v, o, None, ctypes.c_void_p(FAKE * 5000 + 2), *args, ws, need) == ALIGN
    assert c(q, k, v, o, None, cu, 0, 1000, 600, 32, 8, 128, 64, 4, 0, ws, need) == INVALID  # B
    assert c(q, k, v, o, None, cu, 3, 1000, 600, 32, 8, 128, 64, 4, 2, ws, need) == INVALID  # dtype
    assert c(q, k, v, o, None, cu, 3, 1000, 600, 32, 8, 96, 64, 4, 0, ws, need) == UNSUPPORTED  # d
    assert c(q, k, v, o, None, cu, 3, 1000, 600, 32, 8, 128, 4, 4, 0, ws, need) == INVALID  # w <= s
    assert c(q, k, v, q, None, cu, *args, ws, need) == INVALID                # o aliases q
    assert c(q, k, v, o, None, cu, *args, _p(1000), need) == INVALID          # workspace aliases q


def test_normal_build_has_no_bounds_checks(L):
    """The normal library reports no checks, refuses the test margin and has
    no refused index to report (the record is only read on a GPU)."""
    assert L.swa_debug_bounds_checked() == 0
    assert L.swa_debug_set_extent_margin(16) == UNSUPPORTED


def test_checked_build_compiles_and_reports_itself():
    """The bounds-checked debug library (SWA_CHECK_BOUNDS=1) cross-compiles
    for sm_103a, exports the same functions, reports itself as checked and
    takes a test margin (no GPU is touched)."""
    C = swa.load_checked()
    for n in swa.declared_functions():
        assert hasattr(C, n), n
    assert C.swa_debug_bounds_checked() == 1
    assert C.swa_debug_set_extent_margin(-1) == INVALID
    assert C.swa_debug_set_extent_margin(64) == OK
    assert C.swa_debug_set_extent_margin(0) == OK
