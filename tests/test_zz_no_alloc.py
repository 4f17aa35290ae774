"""swa_decode_noalloc, the decode entry point for callers that cannot allocate.

Some callers of this library may not allocate device memory at all -- a
plugin whose host framework owns every device buffer and hands it only inputs
and outputs, or a latency-critical serving loop that must not risk an
allocation's synchronisation or failure.  They cannot supply the workspace
swa_decode needs, so swa_decode_noalloc keeps its split partials in scratch
built into the library.  This file checks it through the C ABI against
swa_decode on the same inputs, on two calls in a row (the second call finds
whatever the first left in the shared scratch).  It is collected last on
purpose and works when run on its own.
"""
import ctypes

import pytest
import torch

from sliding_window_attention_prefill_gb300 import W_INF, Cache, build, decode, device_error, inputs
from sliding_window_attention_prefill_gb300 import swa as binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def noalloc():
    build.build()
    L = binding.lib()
    fn = L.swa_decode_noalloc
    fn.argtypes = [ctypes.c_void_p, ctypes.POINTER(binding.SwaCacheStruct), ctypes.c_void_p,
                   ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    return fn


def _call(fn, q, cache, pos):
    o = torch.empty_like(q)
    c = cache.struct()
    st = fn(ctypes.c_void_p(q.data_ptr()), ctypes.byref(c), ctypes.c_void_p(pos.data_ptr()),
            q.shape[1], cache.w, cache.s, ctypes.c_void_p(o.data_ptr()),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, binding.status_string(st)
    return o


@pytest.mark.parametrize("B,w,s,prompt,cap", [(1, W_INF, 0, 15000, 20000), (16, 512, 4, 4096, None)])
def test_noalloc_matches_decode_twice(noalloc, B, w, s, prompt, cap):
    Hq, Hkv, d = 32, 8, 128
    cache = Cache(B, Hkv, d, w, s, max_len=cap)
    assert binding.decode_workspace_bytes(B, Hq, Hkv, d, cache.cap, w) > 0  # scratch is used
    kp, vp, _, _, qs = inputs.decode_stream(B, Hq, Hkv, d, prompt, 2, seed=31)
    cache.append(kp.cuda(), vp.cuda(), 0)
    for call, p in enumerate([prompt - 1, prompt // 2]):
        q = qs[call].cuda()
        pos = torch.full((B,), p, dtype=torch.int32, device="cuda")
        ref = decode(q, cache, pos)
        got = _call(noalloc, q, cache, pos)
        torch.cuda.synchronize()
        # the same kernels on the same plan and inputs: equal bit for bit
        assert torch.equal(got, ref), f"call {call + 1} (pos {p})"
    assert device_error() == 0
