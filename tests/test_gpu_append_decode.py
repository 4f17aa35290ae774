"""append_decode (one decode step in one kernel) on the GPU.

It must give exactly what ``Cache.append`` of the token followed by
``decode`` gives: the same output bits and the same cache bytes, on a ring
that has wrapped, a cache still filling, sink positions, the infinite window
and the split-K path; and the fp64 oracle's output for a token stream.
"""
import pytest
import torch

import oracle
from gpu_helpers import assert_close, bits
from sliding_window_attention_prefill_gb300 import (W_INF, Cache, append_decode, build, decode,
                                                    device_error, inputs)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


CASES = [
    # B, Hq, Hkv, d, w, s, prompt, steps, max_len, dtype
    (4, 32, 8, 128, 64, 4, 300, 3, None, torch.bfloat16),      # ring wrapped, G = 4
    (2, 8, 2, 128, 512, 4, 100, 3, None, torch.bfloat16),      # cache still filling
    (3, 8, 8, 64, 16, 12, 5, 12, None, torch.bfloat16),        # sink positions, tiny ring, G = 1
    (2, 16, 2, 64, W_INF, 0, 300, 2, 400, torch.bfloat16),     # infinite window, G = 8
    (64, 32, 8, 128, 512, 4, 4096, 2, None, torch.bfloat16),   # one split per sequence and head
    (1, 32, 8, 128, 512, 4, 1000, 2, None, torch.bfloat16),    # several splits (merge kernel)
    (1, 16, 16, 64, 64, 4, 4096, 2, None, torch.float16),      # the pages' shape, fp16
    (2, 32, 8, 128, 128, 4, 129, 3, None, torch.bfloat16),     # two-chunk items, new slot in the first
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}Hq{}Hkv{}d{}w{}s{}P{}".format(*c[:7]))
def test_equals_append_then_decode(case):
    B, Hq, Hkv, d, w, s, prompt, steps, max_len, dtype = case
    kp, vp, ks, vs, qs = inputs.decode_stream(B, Hq, Hkv, d, prompt, steps, seed=21, dtype=dtype)
    a = Cache(B, Hkv, d, w, s, max_len=max_len, dtype=dtype)
    f = Cache(B, Hkv, d, w, s, max_len=max_len, dtype=dtype)
    a.append(kp.cuda(), vp.cuda(), 0)
    f.append(kp.cuda(), vp.cuda(), 0)
    pos = torch.empty(B, dtype=torch.int32, device="cuda")
    for j in range(steps):
        p = prompt + j
        pos.fill_(p)
        k1, v1, q1 = ks[j].cuda(), vs[j].cuda(), qs[j].cuda()
        a.append(k1, v1, p)
        o_ref = decode(q1, a, pos)
        o = append_decode(q1, k1, v1, f, pos)
        torch.cuda.synchronize()
        assert device_error() == 0
        assert torch.equal(o, o_ref), f"step {j}: output differs from append + decode"
        assert torch.equal(f.k, a.k) and torch.equal(f.v, a.v), f"step {j}: cache differs"


def test_token_stream_against_oracle():
    """Llama shape, SWA(64,4): a prompt, then 4 tokens decoded with
    append_decode, each against the oracle's decode over the full history."""
    B, Hq, Hkv, d, w, s, prompt, steps = 2, 32, 8, 128, 64, 4, 200, 4
    kp, vp, ks, vs, qs = inputs.decode_stream(B, Hq, Hkv, d, prompt, steps, seed=22)
    c = Cache(B, Hkv, d, w, s)
    c.append(kp.cuda(), vp.cuda(), 0)
    pos = torch.empty(B, dtype=torch.int32, device="cuda")
    hk, hv = [kp], [vp]
    orc = oracle.get()
    for j in range(steps):
        p = prompt + j
        pos.fill_(p)
        o = append_decode(qs[j].cuda(), ks[j].cuda(), vs[j].cuda(), c, pos).cpu()
        torch.cuda.synchronize()
        assert device_error() == 0
        hk.append(ks[j])
        hv.append(vs[j])
        ref = orc.decode(bits(qs[j]), bits(torch.cat(hk, 1)), bits(torch.cat(hv, 1)), [p] * B, w, s)
        assert_close(o, ref, f"step {j}")


def test_position_outside_cache_changes_nothing():
    """Infinite window, pos[1] = cap: SWA_ERR_BOUNDS on the device; that
    sequence's slot and output are untouched, the other is decoded."""
    B, Hq, Hkv, d, cap = 2, 8, 2, 64, 128
    kp, vp, ks, vs, qs = inputs.decode_stream(B, Hq, Hkv, d, 100, 1, seed=23)
    c = Cache(B, Hkv, d, W_INF, 0, max_len=cap)
    c.append(kp.cuda(), vp.cuda(), 0)
    k_before, v_before = c.k.clone(), c.v.clone()
    pos = torch.tensor([100, cap], dtype=torch.int32, device="cuda")
    out = torch.full((B, Hq, d), 3.0, dtype=torch.bfloat16, device="cuda")
    append_decode(qs[0].cuda(), ks[0].cuda(), vs[0].cuda(), c, pos, out=out)
    torch.cuda.synchronize()
    assert device_error() == -7
    assert torch.all(out[1] == 3.0)
    assert torch.equal(c.k[1], k_before[1]) and torch.equal(c.v[1], v_before[1])
    assert not torch.equal(c.k[0], k_before[0])  # sequence 0's token was written
