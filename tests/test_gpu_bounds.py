"""The bounds-checked debug build on the GPU.

Built with SWA_CHECK_BOUNDS=1, every kernel tests each global index it
computes against the extent of its buffer; an out-of-range index is skipped
and recorded (SWA_ERR_BOUNDS and the index), never trapped.  These tests run
the package's calls on that library:
- on shapes where stores run closest to the ends of their buffers it writes
  the same bits as the normal build and refuses nothing;
- told that the buffers it writes are shorter than they are (the test
  margin, which involves no access outside any real buffer), it refuses
  exactly the writes past the declared end, records them, leaves those
  elements untouched, and writes everything before them as usual.
"""
import numpy as np
import pytest
import torch

from sliding_window_attention_prefill_gb300 import (W_INF, Cache, append_decode, build, decode,
                                                    device_error, inputs, prefill, prefill_varlen)
from sliding_window_attention_prefill_gb300 import swa as binding

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def checked():
    build.build()
    normal = binding.lib()
    C = binding.load_checked()
    assert C.swa_debug_bounds_checked() == 1
    yield normal, C
    binding._lib = normal
    C.swa_debug_set_extent_margin(0)


def _run(lib, fn):
    binding._lib = lib
    try:
        out = fn()
        torch.cuda.synchronize()
        return out
    finally:
        binding._lib = None


def _index(lib):
    return int(lib.swa_debug_bounds_index(binding._stream(torch.device("cuda"))))


def _prefill_cases():
    yield (1, 333, 32, 8, 128, 64, 4, torch.bfloat16)
    yield (2, 200, 16, 16, 64, 512, 4, torch.float16)
    yield (1, 700, 32, 8, 128, W_INF, 0, torch.bfloat16)


@pytest.mark.parametrize("case", list(_prefill_cases()), ids=lambda c: "L{}d{}w{}".format(c[1], c[4], c[5]))
def test_checked_prefill_matches_and_refuses_nothing(checked, case):
    normal, C = checked
    B, L, Hq, Hkv, d, w, s, dt = case
    q, k, v = inputs.prefill_inputs(B, L, Hq, Hkv, d, seed=81, dtype=dt)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    ref, ref_l = _run(normal, lambda: prefill(q, k, v, w, s, return_lse=True))
    got, got_l = _run(C, lambda: prefill(q, k, v, w, s, return_lse=True))
    binding._lib = C
    assert device_error() == 0 and _index(C) == -1
    binding._lib = None
    assert torch.equal(got, ref) and torch.equal(got_l, ref_l)


def test_checked_decode_paths_match(checked):
    """append, decode with split partials, append_decode and varlen on the
    checked library: the normal build's bits, nothing refused."""
    normal, C = checked
    g = inputs.generator(82)
    B, Hq, Hkv, d = 2, 32, 8, 128
    kp = inputs.normal_bf16((B, 900, Hkv, d), g).cuda()
    vp = inputs.normal_bf16((B, 900, Hkv, d), g).cuda()
    q = inputs.normal_bf16((B, Hq, d), g).cuda()
    k1 = inputs.normal_bf16((B, 1, Hkv, d), g).cuda()
    v1 = inputs.normal_bf16((B, 1, Hkv, d), g).cuda()
    pos = torch.full((B,), 900, dtype=torch.int32, device="cuda")
    outs = []
    for lib in (normal, C):
        def calls():
            c = Cache(B, Hkv, d, 512, 4)
            c.append(kp, vp, 0)
            o1 = decode(q, c, pos - 1)
            o2 = append_decode(q, k1, v1, c, pos)
            ci = Cache(B, Hkv, d, W_INF, 0, max_len=1000)
            ci.append(kp, vp, 0)
            o3 = decode(q, ci, pos - 1)  # many splits
            lens = [1, 33, 200, 5]
            qq, kk, vv = inputs.prefill_inputs(1, sum(lens), Hq, Hkv, d, seed=83)
            cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
            o4 = prefill_varlen(qq[0].cuda(), kk[0].cuda(), vv[0].cuda(), cu, 64, 4)
            return o1, o2, o3, o4, c.k.clone(), c.v.clone()
        outs.append(_run(lib, calls))
    binding._lib = C
    assert device_error() == 0 and _index(C) == -1
    binding._lib = None
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_checked_build_refuses_writes_past_a_declared_end(checked):
    """With the margin set, the cache append refuses the last elements of
    the cache, records SWA_ERR_BOUNDS and the first refused vector index,
    and leaves those elements as they were; the rest matches the normal
    build.  The same for a decode's output."""
    normal, C = checked
    g = inputs.generator(84)
    B, Hq, Hkv, d, w, s = 2, 8, 2, 64, 64, 4
    kp = inputs.normal_bf16((B, 300, Hkv, d), g).cuda()
    vp = inputs.normal_bf16((B, 300, Hkv, d), g).cuda()
    q = inputs.normal_bf16((B, Hq, d), g).cuda()
    ref = _run(normal, lambda: Cache(B, Hkv, d, w, s))
    _run(normal, lambda: ref.append(kp, vp, 0))
    ref_o = _run(normal, lambda: decode(q, ref, torch.full((B,), 299, dtype=torch.int32, device="cuda")))
    margin = 3 * d  # the last three slots of the last kv head's ring
    n = B * Hkv * w * d
    try:
        assert C.swa_debug_set_extent_margin(margin) == 0
        c = _run(C, lambda: Cache(B, Hkv, d, w, s))
        c.k.fill_(7.0), c.v.fill_(7.0)
        _run(C, lambda: c.append(kp, vp, 0))
        binding._lib = C
        assert device_error() == -7
        first = _index(C)
        binding._lib = None
        assert first >= (n - margin) // 8, first  # a vector index past the declared end
        kf, rf = c.k.reshape(-1), ref.k.reshape(-1)
        assert torch.equal(kf[:n - margin], rf[:n - margin])
        assert torch.all(kf[n - margin:] == 7.0)
        # the output of a decode: its last `margin` elements are refused
        o = torch.full((B, Hq, d), 5.0, dtype=torch.bfloat16, device="cuda")
        c2 = _run(C, lambda: Cache(B, Hkv, d, w, s))
        c2.k.copy_(ref.k), c2.v.copy_(ref.v)
        pos = torch.full((B,), 299, dtype=torch.int32, device="cuda")
        _run(C, lambda: decode(q, c2, pos, out=o))
        binding._lib = C
        assert device_error() == -7 and _index(C) >= 0
        binding._lib = None
        of, rof = o.reshape(-1), ref_o.reshape(-1)
        m = of.numel()
        assert torch.equal(of[:m - margin], rof[:m - margin])
        assert torch.all(of[m - margin:] == 5.0)
    finally:
        C.swa_debug_set_extent_margin(0)
        binding._lib = None
