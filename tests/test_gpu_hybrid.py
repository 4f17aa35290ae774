"""Hybrid window + linear decode (GPU) against the fp64 oracle.

The cache keeps the SWA(w,s) attended set; the tokens it evicts are folded
into the linear state S, z (hybrid_append), and decode mixes both
(hybrid_decode).  The state is compared with the oracle's sums over the
evicted positions, the outputs with the oracle's direct definition.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, bits
from sliding_window_attention_prefill_gb300 import (W_INF, Cache, LinearState, build, decode,
                                                    device_error, hybrid_append, hybrid_decode,
                                                    inputs)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def _weights(Hkv, d, df, seed):
    g = inputs.generator(seed)
    return (torch.randn(Hkv, d, df, generator=g, dtype=torch.float32) * (0.3 / d ** 0.5))


def _assert_state(state, k_hist, v_hist, W, w, s, dt, what):
    S_ref, z_ref = oracle.get().hybrid_state(bits(k_hist), bits(v_hist), W.double().numpy(), w, s,
                                             dtype=dt)
    S, z = state.S.cpu().double().numpy(), state.z.cpu().double().numpy()
    for got, ref, name in ((S, S_ref, "S"), (z, z_ref, "z")):
        err = np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30)
        assert err < 1e-4, f"{what}: {name} relative error {err:.2e}"


CASES = [
    # B, Hq, Hkv, d, df, w, s, prompt, steps, dtype
    (2, 32, 8, 128, 64, 64, 4, 300, 3, torch.bfloat16),     # Llama shape, SWA(64,4) + linear
    (1, 16, 16, 64, 32, 64, 4, 500, 3, torch.float16),      # the pages' shape, fp16
    (2, 8, 2, 128, 32, 96, 0, 130, 4, torch.bfloat16),      # no sinks, G = 4
    (3, 8, 4, 64, 64, 16, 12, 70, 3, torch.bfloat16),       # 12 sinks, ring of 4 slots
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}Hq{}Hkv{}d{}df{}w{}s{}".format(*c[:7]))
def test_hybrid_state_and_decode(case):
    B, Hq, Hkv, d, df, w, s, prompt, steps, dtype = case
    dt = "f16" if dtype == torch.float16 else "bf16"
    kp, vp, ks, vs, qs = inputs.decode_stream(B, Hq, Hkv, d, prompt, steps, seed=13, dtype=dtype)
    W = _weights(Hkv, d, df, seed=14)
    cache = Cache(B, Hkv, d, w, s, dtype=dtype)
    state = LinearState(cache, W.cuda())
    hybrid_append(cache, state, kp.cuda(), vp.cuda(), 0)   # the prompt in one bulk append
    torch.cuda.synchronize()
    assert device_error() == 0
    _assert_state(state, kp, vp, W, w, s, dt, "after the prompt")
    pos = torch.empty(B, dtype=torch.int32, device="cuda")
    hist_k, hist_v = [kp], [vp]
    orc = oracle.get()
    for j in range(steps):
        p = prompt + j
        hybrid_append(cache, state, ks[j].cuda(), vs[j].cuda(), p)
        pos.fill_(p)
        o = hybrid_decode(qs[j].cuda(), cache, state, pos).cpu()
        torch.cuda.synchronize()
        assert device_error() == 0
        hist_k.append(ks[j])
        hist_v.append(vs[j])
        hk, hv = torch.cat(hist_k, dim=1), torch.cat(hist_v, dim=1)
        ref = orc.hybrid_decode(bits(qs[j]), bits(hk), bits(hv), W.double().numpy(), [p] * B, w, s,
                                dtype=dt)
        assert_close(o, ref, f"hybrid decode step {j}")
    _assert_state(state, hk, hv, W, w, s, dt, "after the steps")


def test_hybrid_bulk_append_after_wrap():
    """Two bulk appends, the second starting after the ring has wrapped and
    evicting both ring entries and its own first tokens."""
    B, Hq, Hkv, d, df, w, s = 2, 8, 2, 128, 64, 64, 4
    kp, vp, _, _, _ = inputs.decode_stream(B, Hq, Hkv, d, 400, 0, seed=15)
    W = _weights(Hkv, d, df, seed=16)
    cache = Cache(B, Hkv, d, w, s)
    state = LinearState(cache, W.cuda())
    hybrid_append(cache, state, kp[:, :150].contiguous().cuda(), vp[:, :150].contiguous().cuda(), 0)
    hybrid_append(cache, state, kp[:, 150:].contiguous().cuda(), vp[:, 150:].contiguous().cuda(), 150)
    torch.cuda.synchronize()
    assert device_error() == 0
    _assert_state(state, kp, vp, W, w, s, "bf16", "two bulk appends")


def test_hybrid_without_eviction_is_swa_decode():
    """Before the cache is full (and for w = infinity) nothing is evicted: the
    hybrid decode is the SWA decode."""
    B, Hq, Hkv, d, df = 2, 8, 2, 128, 64
    for w, s, prompt, max_len in [(64, 4, 40, None), (W_INF, 0, 300, 400)]:
        kp, vp, _, _, qs = inputs.decode_stream(B, Hq, Hkv, d, prompt, 1, seed=17)
        cache = Cache(B, Hkv, d, w, s, max_len=max_len)
        state = LinearState(cache, _weights(Hkv, d, df, seed=18).cuda())
        hybrid_append(cache, state, kp.cuda(), vp.cuda(), 0)
        pos = torch.full((B,), prompt - 1, dtype=torch.int32, device="cuda")
        a = hybrid_decode(qs[0].cuda(), cache, state, pos)
        b = decode(qs[0].cuda(), cache, pos)
        torch.cuda.synchronize()
        assert device_error() == 0
        assert not state.S.any() and not state.z.any()
        assert (a.float() - b.float()).abs().max().item() <= 2e-3, w
