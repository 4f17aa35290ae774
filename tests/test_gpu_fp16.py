"""fp16 element type (GPU) against the fp64 oracle: prefill, cache append,
decode and chunked prefill.

fp16 is the precision of the pages' own system measurements ("Sliding-window
beats linear attention", paper summary page, section "Method steps", step
five): a 4-layer model with D = 1024 and 16 heads of 64 (multi-head, G = 1),
batch 1.  The inputs are the same N(0,1) draws as the bf16 tests, rounded to
fp16; the oracle widens the same fp16 bits exactly.  The bf16 tolerance is
kept (fp16 rounds 8 times finer, so it holds with room).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, bits
from sliding_window_attention_prefill_gb300 import (W_INF, Cache, build, decode, device_error, inputs,
                                                    prefill, prefill_chunk)

pytestmark = pytest.mark.gpu

F16 = torch.float16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


PREFILL_CASES = [
    # B, L, Hq, Hkv, d, w, s
    (1, 2048, 16, 16, 64, 64, 4),      # the pages' attention shape, SWA(64,4)
    (1, 1500, 16, 16, 64, 512, 4),     # same shape, SWA(512,4), ragged tail
    (1, 1000, 16, 16, 64, W_INF, 0),   # same shape, full causal
    (2, 300, 8, 2, 128, 64, 4),        # d = 128, G = 4, two sequences
    (1, 1600, 4, 1, 128, 1400, 4),     # 256-column key tiles at d = 128
    (1, 700, 8, 8, 64, 900, 4),        # 256-column key tiles at d = 64
    (1, 90, 4, 1, 128, 16, 12),        # 12 sinks, tiny ring
]


@pytest.mark.parametrize("case", PREFILL_CASES, ids=lambda c: "B{}L{}Hq{}Hkv{}d{}w{}s{}".format(*c))
def test_prefill_f16(case):
    B, L, Hq, Hkv, d, w, s = case
    q, k, v = inputs.prefill_inputs(B, L, Hq, Hkv, d, seed=3, sink_rows=4, dtype=F16)
    o, lse = prefill(q.cuda(), k.cuda(), v.cuda(), w, s, return_lse=True)
    torch.cuda.synchronize()
    assert o.dtype == F16
    assert device_error() == 0
    ref_o, ref_l = oracle.get().prefill(bits(q), bits(k), bits(v), w, s, dtype="f16")
    assert_close(o, ref_o, f"o {case}")
    assert_close(lse, ref_l, f"lse {case}", max_abs=4e-3, mean_rel=1e-3)


def test_prefill_f16_differs_from_bf16_reading():
    """The same bits read as bf16 give another result: the kernel really
    computes in fp16 (a bf16 MMA on fp16 bits would fail the parity above,
    and this checks the oracle side of that argument)."""
    q, k, v = inputs.prefill_inputs(1, 64, 2, 2, 64, seed=4, dtype=F16)
    a, _ = oracle.get().prefill(bits(q), bits(k), bits(v), 16, 4, dtype="f16")
    b, _ = oracle.get().prefill(bits(q), bits(k), bits(v), 16, 4, dtype="bf16")
    assert np.abs(a - b).max() > 1.0


@pytest.mark.parametrize("B,Hq,Hkv,d,w,s,prompt,steps,max_len", [
    (1, 16, 16, 64, 64, 4, 4096, 4, None),        # the pages' shape, SWA(64,4)
    (1, 16, 16, 64, 512, 4, 4096, 4, None),       # the pages' shape, SWA(512,4)
    (1, 16, 16, 64, W_INF, 0, 6000, 3, 6100),     # the pages' shape, full causal (split merge)
    (8, 32, 8, 128, 512, 4, 1000, 3, None),       # d = 128, G = 4
    (2, 8, 4, 64, 100, 4, 60, 3, None),           # cache still filling, G = 2
])
def test_decode_f16(B, Hq, Hkv, d, w, s, prompt, steps, max_len):
    kp, vp, ks, vs, qs = inputs.decode_stream(B, Hq, Hkv, d, prompt, steps, seed=6, dtype=F16)
    c = Cache(B, Hkv, d, w, s, max_len=max_len, dtype=F16)
    c.append(kp.cuda(), vp.cuda(), 0)
    pos_t = torch.empty(B, dtype=torch.int32, device="cuda")
    outs = []
    for j in range(steps):
        c.append(ks[j].cuda(), vs[j].cuda(), prompt + j)
        pos_t.fill_(prompt + j)
        outs.append(decode(qs[j].cuda(), c, pos_t).cpu())
    torch.cuda.synchronize()
    assert device_error() == 0
    hk = bits(torch.cat([kp] + [ks[j] for j in range(steps)], dim=1))
    hv = bits(torch.cat([vp] + [vs[j] for j in range(steps)], dim=1))
    orc = oracle.get()
    for j, o in enumerate(outs):
        assert o.dtype == F16
        ref = orc.decode(bits(qs[j]), hk, hv, [prompt + j] * B, w, s, dtype="f16")
        assert_close(o, ref, f"decode step {j} SWA({w},{s}) B={B} d={d}")
    # the cache holds the fp16 bits the oracle's append simulation writes
    ck = np.zeros((B, Hkv, c.cap, d), np.uint16)
    cv = np.zeros_like(ck)
    orc.cache_append(ck, cv, hk, hv, 0, w, s)
    assert np.array_equal(bits(c.k), ck) and np.array_equal(bits(c.v), cv)


@pytest.mark.parametrize("w,s,chunks", [(64, 4, [700, 1, 300]), (W_INF, 0, [256, 300])])
def test_prefill_chunk_f16(w, s, chunks):
    """The pages' shape prefilled chunk by chunk from an fp16 cache equals the
    oracle's prefill of the whole prompt."""
    B, Hq, Hkv, d = 1, 16, 16, 64
    L = sum(chunks)
    q, k, v = inputs.prefill_inputs(B, L, Hq, Hkv, d, seed=8, dtype=F16)
    ref_o, _ = oracle.get().prefill(bits(q), bits(k), bits(v), w, s, dtype="f16")
    cache = Cache(B, Hkv, d, w, s, max_len=(L if w == W_INF else None), dtype=F16)
    pos0 = 0
    for n in chunks:
        sl = slice(pos0, pos0 + n)
        o = prefill_chunk(q[:, sl].contiguous().cuda(), k[:, sl].contiguous().cuda(),
                          v[:, sl].contiguous().cuda(), cache, pos0)
        torch.cuda.synchronize()
        assert device_error() == 0
        assert_close(o, ref_o[:, sl], f"chunk at {pos0} (n={n})")
        pos0 += n


def test_mixed_types_are_rejected():
    """q of one type with k, v or the cache of the other fails in the binding."""
    q, k, v = inputs.prefill_inputs(1, 32, 2, 2, 64, seed=9, dtype=F16)
    with pytest.raises(TypeError):
        prefill(q.cuda(), k.to(torch.bfloat16).cuda(), v.cuda(), 16, 4)
    c = Cache(1, 2, 64, 16, 4, dtype=F16)
    with pytest.raises(TypeError):
        c.append(k.to(torch.bfloat16).cuda(), v.to(torch.bfloat16).cuda(), 0)
    pos = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(TypeError):
        decode(torch.zeros(1, 2, 64, dtype=torch.bfloat16, device="cuda"), c, pos)


def test_prefill_many_units_per_cta_keeps_its_waits():
    """Many two-tile units per CTA (the pages' shape, L = 32768, SWA(512,4)):
    repeated launches record no wait timeout, and sampled rows match the
    oracle.  (An mbarrier waited by one parity bit must not complete twice
    before it is waited; a fast softmax finishing two tiles before the MMA
    warp looked at the first would otherwise stall the kernel.)"""
    B, L, Hq, Hkv, d, w, s = 1, 32768, 16, 16, 64, 512, 4
    q, k, v = inputs.prefill_inputs(B, L, Hq, Hkv, d, seed=12, dtype=F16)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    for _ in range(3):
        o = prefill(qd, kd, vd, w, s)
        torch.cuda.synchronize()
        assert device_error() == 0
    rng = np.random.default_rng(5)
    rows = np.stack([np.zeros(64, np.int64), rng.integers(0, L, 64), rng.integers(0, Hq, 64)], 1)
    ref, _ = oracle.get().prefill_rows(bits(q), bits(k), bits(v), rows, w, s, dtype="f16")
    got = o.cpu()[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert_close(got, ref, "sampled rows")
