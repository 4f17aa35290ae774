"""Parity at the decode workloads' full footprints (GPU).

The fixed cache holds the first s tokens and the latest w - s, and stops
growing once it holds w ("No post-training, just 4 more tokens", news page,
section "Research method"; "Microsoft SWA paper overturns linear attention",
blog page, section "What they tested").  These cases run the library where
its integer work is widest:
- a full-causal cache of 256 sequences x 8 kv heads x 32769 slots, more than
  2^32 elements per tensor (the 64-bit offsets of the append and of the fused
  append + decode, and the row coordinates of the decode's tensor maps);
- one sequence decoded at position 262143, the end of the context sweep, for
  w = 64, 512 and infinity;
- 256 sequences at position 262143 (ring offsets far from slot 0);
- the B = 64 decode workload's whole stream: a 4096-token prompt, then 1024
  steps that each append one token and decode it.
Every output is compared with the oracle element by element and every cache
byte of the compared sequences with the oracle's host simulation.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, bits
from sliding_window_attention_prefill_gb300 import (W_INF, Cache, append_decode, build, decode,
                                                    device_error, inputs)

pytestmark = pytest.mark.gpu

HQ, HKV, D = 32, 8, 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    yield
    torch.cuda.empty_cache()


def _zeros_like_cache(B, cap):
    return (np.zeros((B, HKV, cap, D), np.uint16), np.zeros((B, HKV, cap, D), np.uint16))


def test_full_causal_cache_beyond_2_32_elements():
    """B=256, w=inf, 32768 positions appended in bulk chunks of 1024, then one
    append_decode of position 32768; sequences 0, 127 and 255 are compared."""
    B, P, n = 256, 32768, 1024
    cap = P + 1
    checked = [0, 127, 255]
    c = Cache(B, HKV, D, W_INF, 0, max_len=cap)
    assert c.k.numel() > (1 << 32)
    gen = inputs.device_generator(41)
    hist_k = np.empty((len(checked), cap, HKV, D), np.uint16)
    hist_v = np.empty_like(hist_k)
    sim_k, sim_v = _zeros_like_cache(len(checked), cap)
    orc = oracle.get()
    for p0 in range(0, P, n):
        kn = inputs.normal16_on((B, n, HKV, D), gen)
        vn = inputs.normal16_on((B, n, HKV, D), gen)
        c.append(kn, vn, p0)
        hk, hv = bits(kn[checked]), bits(vn[checked])
        hist_k[:, p0:p0 + n], hist_v[:, p0:p0 + n] = hk, hv
        orc.cache_append(sim_k, sim_v, hk, hv, p0, W_INF, 0)
        del kn, vn
    q = inputs.normal16_on((B, HQ, D), gen)
    k1 = inputs.normal16_on((B, 1, HKV, D), gen)
    v1 = inputs.normal16_on((B, 1, HKV, D), gen)
    pos = torch.full((B,), P, dtype=torch.int32, device="cuda")
    o_fused = append_decode(q, k1, v1, c, pos)
    o_plain = decode(q, c, pos)
    torch.cuda.synchronize()
    assert device_error() == 0
    hk1, hv1 = bits(k1[checked]), bits(v1[checked])
    hist_k[:, P:P + 1], hist_v[:, P:P + 1] = hk1, hv1
    orc.cache_append(sim_k, sim_v, hk1, hv1, P, W_INF, 0)
    assert np.array_equal(bits(c.k[checked]), sim_k), "K slots of the checked sequences"
    assert np.array_equal(bits(c.v[checked]), sim_v), "V slots of the checked sequences"
    ref = orc.decode(bits(q[checked]), hist_k, hist_v, [P] * len(checked), W_INF, 0)
    assert_close(o_fused[checked], ref, "append_decode, w=inf, 32768 positions, B=256")
    assert_close(o_plain[checked], ref, "decode, w=inf, 32768 positions, B=256")
    del c
    torch.cuda.empty_cache()


@pytest.fixture(scope="module")
def long_history():
    """One sequence of 262144 positions (k, v [1, 262144, Hkv, d]) and the
    query of the last position, on the device and as host bit patterns."""
    gen = inputs.device_generator(43)
    k = inputs.normal16_on((1, 1 << 18, HKV, D), gen)
    v = inputs.normal16_on((1, 1 << 18, HKV, D), gen)
    q = inputs.normal16_on((1, HQ, D), gen)
    yield k, v, q, bits(k), bits(v), bits(q)


@pytest.mark.parametrize("w,s", [(64, 4), (512, 4), (W_INF, 0)])
def test_single_sequence_at_position_262143(long_history, w, s):
    """Positions 0 .. 262142 appended in one bulk call (only the survivors are
    written for a finite window), then append_decode of position 262143."""
    k, v, q, hk, hv, hq = long_history
    P = (1 << 18) - 1
    c = Cache(1, HKV, D, w, s, max_len=(P + 1 if w == W_INF else None))
    c.append(k[:, :P], v[:, :P], 0)
    pos = torch.full((1,), P, dtype=torch.int32, device="cuda")
    o_fused = append_decode(q, k[:, P:], v[:, P:], c, pos)
    o_plain = decode(q, c, pos)
    torch.cuda.synchronize()
    assert device_error() == 0
    orc = oracle.get()
    sim_k, sim_v = _zeros_like_cache(1, c.cap)
    orc.cache_append(sim_k, sim_v, hk[:, :P], hv[:, :P], 0, w, s)
    orc.cache_append(sim_k, sim_v, hk[:, P:], hv[:, P:], P, w, s)
    assert np.array_equal(bits(c.k), sim_k), f"K, SWA({w},{s})"
    assert np.array_equal(bits(c.v), sim_v), f"V, SWA({w},{s})"
    ref = orc.decode(hq, hk, hv, [P], w, s)
    assert_close(o_fused, ref, f"append_decode SWA({w},{s}) at {P}")
    assert_close(o_plain, ref, f"decode SWA({w},{s}) at {P}")
    del c
    torch.cuda.empty_cache()


@pytest.mark.parametrize("w", [64, 512])
def test_batch256_at_position_262143(w):
    """B=256, SWA(w,4) at position 262143.  The cache receives the sinks
    (positions 0-3) and the positions 262143-(w-4)+1 .. 262142 as two bulk
    appends, then the token 262143 through append_decode: exactly the set the
    query attends to.  The oracle simulates the same appends on the host and
    decodes over its own cache (its decode over the ring is pinned to its
    decode over the history)."""
    B, s = 256, 4
    P = (1 << 18) - 1
    gen = inputs.device_generator(47 + w)
    ks = inputs.normal16_on((B, s, HKV, D), gen)
    vs = inputs.normal16_on((B, s, HKV, D), gen)
    nb = w - s - 1
    kb = inputs.normal16_on((B, nb, HKV, D), gen)
    vb = inputs.normal16_on((B, nb, HKV, D), gen)
    k1 = inputs.normal16_on((B, 1, HKV, D), gen)
    v1 = inputs.normal16_on((B, 1, HKV, D), gen)
    q = inputs.normal16_on((B, HQ, D), gen)
    c = Cache(B, HKV, D, w, s)
    c.append(ks, vs, 0)
    c.append(kb, vb, P - nb)
    pos = torch.full((B,), P, dtype=torch.int32, device="cuda")
    o = append_decode(q, k1, v1, c, pos)
    torch.cuda.synchronize()
    assert device_error() == 0
    orc = oracle.get()
    sim_k, sim_v = _zeros_like_cache(B, w)
    orc.cache_append(sim_k, sim_v, bits(ks), bits(vs), 0, w, s)
    orc.cache_append(sim_k, sim_v, bits(kb), bits(vb), P - nb, w, s)
    orc.cache_append(sim_k, sim_v, bits(k1), bits(v1), P, w, s)
    assert np.array_equal(bits(c.k), sim_k), f"K, SWA({w},4)"
    assert np.array_equal(bits(c.v), sim_v), f"V, SWA({w},4)"
    ref = orc.decode_cache(bits(q), sim_k, sim_v, [P] * B, w, s)
    assert_close(o, ref, f"B=256 SWA({w},4) at {P}")


@pytest.fixture(scope="module")
def llama_stream():
    """The B=64 decode workload's inputs: a 4096-token N(0,1) prompt, then 1024
    steps of one token (k, v) and one query each (CPU generator, seed 0)."""
    return inputs.decode_stream(64, HQ, HKV, D, 4096, 1024, seed=0)


STREAM_CHECKS = sorted({0, 1, 2, 59, 60, 61, 127, 255, 383, 508, 509, 511, 512, 640, 767, 895,
                        1000, 1022, 1023})


@pytest.mark.parametrize("w", [64, 512])
def test_batch64_stream_of_1024_steps(llama_stream, w):
    """B=64, SWA(w,4): the prompt bulk-appended, then all 1024 append_decode
    steps; 19 steps spread over the stream (the ring's wrap points included,
    and the last) are compared with the oracle's decode over the whole
    history, and the final cache with its host simulation, byte for byte."""
    B, s, prompt, steps = 64, 4, 4096, 1024
    kp, vp, ks, vs, qs = llama_stream
    c = Cache(B, HKV, D, w, s)
    c.append(kp.cuda(), vp.cuda(), 0)
    ks_d, vs_d, qs_d = ks.cuda(), vs.cuda(), qs.cuda()
    pos = torch.empty(B, dtype=torch.int32, device="cuda")
    outs = {}
    for j in range(steps):
        pos.fill_(prompt + j)
        o = append_decode(qs_d[j], ks_d[j], vs_d[j], c, pos)
        if j in STREAM_CHECKS:
            outs[j] = o.cpu()
    torch.cuda.synchronize()
    assert device_error() == 0
    orc = oracle.get()
    hk = bits(torch.cat([kp, ks.transpose(0, 1).reshape(B, steps, HKV, D)], dim=1))
    hv = bits(torch.cat([vp, vs.transpose(0, 1).reshape(B, steps, HKV, D)], dim=1))
    for j, o in outs.items():
        ref = orc.decode(bits(qs[j]), hk, hv, [prompt + j] * B, w, s)
        assert_close(o, ref, f"SWA({w},4) B=64 step {j}")
    sim_k, sim_v = _zeros_like_cache(B, w)
    orc.cache_append(sim_k, sim_v, hk, hv, 0, w, s)
    assert np.array_equal(bits(c.k), sim_k), f"final K, SWA({w},4)"
    assert np.array_equal(bits(c.v), sim_v), f"final V, SWA({w},4)"
