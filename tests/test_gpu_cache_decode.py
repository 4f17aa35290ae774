"""Cache append (bit-exact) and decode parity against the oracle (GPU)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, bits
from sliding_window_attention_prefill_gb300 import W_INF, Cache, build, decode, device_error, inputs, prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def _host_cache(c: Cache):
    return np.zeros((c.B, c.Hkv, c.cap, c.d), np.uint16), np.zeros((c.B, c.Hkv, c.cap, c.d), np.uint16)


@pytest.mark.parametrize("w,s,d", [(64, 4, 128), (16, 0, 64), (9, 8, 64), (W_INF, 0, 128)])
def test_append_bit_exact(w, s, d):
    """Random schedule of bulk and single appends; the cache bytes equal the
    oracle's host simulation after every call."""
    B, Hkv = 3, 2
    cap = 400 if w == W_INF else w
    c = Cache(B, Hkv, d, w, s, max_len=cap if w == W_INF else None)
    hk, hv = _host_cache(c)
    orc = oracle.get()
    g = inputs.generator(11)
    pos = 0
    for n in [100, 1, 1, 7, 0, 64, 1, 3, 150, 1]:
        if w == W_INF and pos + n > cap:
            break
        kn = inputs.normal_bf16((B, n, Hkv, d), g)
        vn = inputs.normal_bf16((B, n, Hkv, d), g)
        c.append(kn.cuda(), vn.cuda(), pos)
        orc.cache_append(hk, hv, bits(kn), bits(vn), pos, w, s)
        torch.cuda.synchronize()
        assert np.array_equal(bits(c.k), hk), f"K after append n={n} at {pos}"
        assert np.array_equal(bits(c.v), hv), f"V after append n={n} at {pos}"
        pos += n


def test_append_more_positions_than_a_grid_dimension():
    """A bulk append whose surviving positions (every one of them, w = inf)
    outnumber the 65535 limit of a grid's y dimension, into a cache at an
    offset; plus a finite-window cache from a prompt of the same length."""
    B, Hkv, d, n = 2, 1, 64, 70000
    g = inputs.generator(12)
    kn = inputs.normal_bf16((B, n, Hkv, d), g)
    vn = inputs.normal_bf16((B, n, Hkv, d), g)
    orc = oracle.get()
    for w, s, pos0, cap in [(W_INF, 0, 16, n + 32), (512, 4, 0, None)]:
        c = Cache(B, Hkv, d, w, s, max_len=cap)
        hk, hv = _host_cache(c)
        c.append(kn.cuda(), vn.cuda(), pos0)
        orc.cache_append(hk, hv, bits(kn), bits(vn), pos0, w, s)
        torch.cuda.synchronize()
        assert np.array_equal(bits(c.k), hk), f"K, w={w}"
        assert np.array_equal(bits(c.v), hv), f"V, w={w}"


def _decode_case(B, Hq, Hkv, d, w, s, prompt, steps, check, seed=0, max_len=None):
    kp, vp, ks, vs, qs = inputs.decode_stream(B, Hq, Hkv, d, prompt, steps, seed=seed)
    c = Cache(B, Hkv, d, w, s, max_len=max_len)
    c.append(kp.cuda(), vp.cuda(), 0)
    outs = {}
    pos_t = torch.empty(B, dtype=torch.int32, device="cuda")
    for j in range(steps):
        p = prompt + j
        c.append(ks[j].cuda(), vs[j].cuda(), p)
        pos_t.fill_(p)
        o = decode(qs[j].cuda(), c, pos_t)
        if j in check:
            outs[j] = o.cpu()
    torch.cuda.synchronize()
    assert device_error() == 0
    hist_k = torch.cat([kp] + [ks[j] for j in range(steps)], dim=1)
    hist_v = torch.cat([vp] + [vs[j] for j in range(steps)], dim=1)
    hk, hv = bits(hist_k), bits(hist_v)
    orc = oracle.get()
    for j, o in outs.items():
        ref = orc.decode(bits(qs[j]), hk, hv, [prompt + j] * B, w, s)
        assert_close(o, ref, f"decode step {j} SWA({w},{s}) B={B}")


@pytest.mark.parametrize("w", [64, 512])
def test_decode_llama_batch64(w):
    """B=64, Hq=32, Hkv=8, d=128, SWA(w,4): 4096-token prompt, then steps."""
    _decode_case(64, 32, 8, 128, w, 4, 4096, 24, check={0, 1, 11, 23})


@pytest.mark.parametrize("B,Hq,Hkv,d,w,s,prompt", [
    (2, 8, 8, 128, 64, 4, 10),     # G=1, cache still filling
    (3, 8, 4, 128, 33, 1, 200),    # G=2, odd window
    (2, 16, 2, 64, 100, 4, 300),   # G=8 (d=64)
    (2, 16, 2, 128, 96, 4, 150),   # G=8 (d=128)
    (3, 8, 8, 64, 70, 2, 140),     # G=1, d=64, ragged tail chunks
    (1, 4, 1, 64, 5, 4, 40),       # ring of one slot
    (2, 8, 2, 128, 128, 0, 50),    # no sinks, filling
])
def test_decode_shapes(B, Hq, Hkv, d, w, s, prompt):
    _decode_case(B, Hq, Hkv, d, w, s, prompt, 6, check={0, 5}, seed=5)


def test_decode_full_causal_many_splits():
    """w = infinity, B=1, Hq=32, Hkv=8: long history so the split-K merge runs."""
    _decode_case(1, 32, 8, 128, W_INF, 0, 15000, 3, check={0, 2}, seed=7, max_len=20000)


def test_decode_ragged_positions():
    """Per-sequence positions on one SWA(64,4) cache (device pos array)."""
    B, Hq, Hkv, d, w, s = 4, 8, 2, 128, 64, 4
    ends = [0, 3, 63, 500]
    P = max(ends) + 1
    g = inputs.generator(21)
    k = inputs.normal_bf16((B, P, Hkv, d), g)
    v = inputs.normal_bf16((B, P, Hkv, d), g)
    q = inputs.normal_bf16((B, Hq, d), g)
    out = torch.empty(B, Hq, d, dtype=torch.bfloat16)
    orc = oracle.get()
    for b, e in enumerate(ends):
        c = Cache(1, Hkv, d, w, s)
        c.append(k[b:b + 1, :e + 1].contiguous().cuda(), v[b:b + 1, :e + 1].contiguous().cuda(), 0)
        # one cache per sequence here; the batched call below uses a stacked cache
        if b == 0:
            stacked_k = torch.zeros(B, Hkv, w, d, dtype=torch.bfloat16, device="cuda")
            stacked_v = torch.zeros_like(stacked_k)
        stacked_k[b] = c.k[0]
        stacked_v[b] = c.v[0]
    cache = Cache.from_tensors(stacked_k, stacked_v, w, s)
    pos = torch.tensor(ends, dtype=torch.int32, device="cuda")
    o = decode(q.cuda(), cache, pos).cpu()
    for b, e in enumerate(ends):
        ref = orc.decode(bits(q[b:b + 1]), bits(k[b:b + 1]), bits(v[b:b + 1]), [e], w, s)
        assert_close(o[b:b + 1], ref, f"ragged b={b} pos={e}")


def test_decode_matches_prefill_row():
    """Decoding position t from the cache gives prefill's row t (both on the GPU)."""
    B, L, Hq, Hkv, d, w, s = 2, 700, 32, 8, 128, 256, 4
    q, k, v = inputs.prefill_inputs(B, L, Hq, Hkv, d, seed=9)
    o_pre = prefill(q.cuda(), k.cuda(), v.cuda(), w, s).cpu()
    for t in [0, 5, 255, 256, 699]:
        c = Cache(B, Hkv, d, w, s)
        c.append(k[:, :t + 1].contiguous().cuda(), v[:, :t + 1].contiguous().cuda(), 0)
        pos = torch.full((B,), t, dtype=torch.int32, device="cuda")
        o_dec = decode(q[:, t].contiguous().cuda(), c, pos).cpu()
        d_ = (o_dec.float() - o_pre[:, t].float()).abs().max().item()
        assert d_ <= 2e-2, (t, d_)


def test_decode_position_out_of_range_is_reported():
    """pos >= cap on an infinite-window cache: the kernel skips the sequence and
    records SWA_ERR_BOUNDS (-7) instead of reading past the cache."""
    c = Cache(1, 2, 128, W_INF, 0, max_len=64)
    q = torch.zeros(1, 8, 128, dtype=torch.bfloat16, device="cuda")
    pos = torch.tensor([64], dtype=torch.int32, device="cuda")
    decode(q, c, pos)
    assert device_error() == -7
    assert device_error() == 0


@pytest.mark.parametrize("B,Hq,Hkv,d,w,prompt", [(2, 32, 8, 128, 512, 100), (1, 8, 2, 64, 256, 5)])
def test_decode_unfilled_slots_are_masked(B, Hq, Hkv, d, w, prompt):
    """A finite-window cache not yet full: its unfilled slots hold NaN.  The
    decode reads chunks of those slots (a window's splits cover all w slots,
    some of them past the filled ones) and must mask every one of them."""
    s = 4
    g = inputs.generator(31)
    kp = inputs.normal_bf16((B, prompt, Hkv, d), g)
    vp = inputs.normal_bf16((B, prompt, Hkv, d), g)
    q = inputs.normal_bf16((B, Hq, d), g)
    c = Cache(B, Hkv, d, w, s)
    c.k.fill_(float("nan"))
    c.v.fill_(float("nan"))
    c.append(kp.cuda(), vp.cuda(), 0)
    pos = torch.full((B,), prompt - 1, dtype=torch.int32, device="cuda")
    o = decode(q.cuda(), c, pos).cpu()
    assert device_error() == 0
    assert not torch.isnan(o.float()).any()
    ref = oracle.get().decode(bits(q), bits(kp), bits(vp), [prompt - 1] * B, w, s)
    assert_close(o, ref, f"filling SWA({w},4) at {prompt - 1}")


def test_decode_negative_position_finite_window():
    """pos < 0 for one sequence of a finite-window cache: SWA_ERR_BOUNDS is
    recorded, that sequence's output is left alone, the others are exact."""
    B, Hq, Hkv, d, w, s, prompt = 3, 8, 2, 128, 64, 4, 80
    g = inputs.generator(32)
    kp = inputs.normal_bf16((B, prompt, Hkv, d), g)
    vp = inputs.normal_bf16((B, prompt, Hkv, d), g)
    q = inputs.normal_bf16((B, Hq, d), g)
    c = Cache(B, Hkv, d, w, s)
    c.append(kp.cuda(), vp.cuda(), 0)
    pos = torch.tensor([prompt - 1, -1, prompt - 1], dtype=torch.int32, device="cuda")
    out = torch.full((B, Hq, d), 7.0, dtype=torch.bfloat16, device="cuda")
    decode(q.cuda(), c, pos, out=out)
    assert device_error() == -7
    o = out.cpu()
    assert torch.all(o[1] == 7.0)
    ref = oracle.get().decode(bits(q), bits(kp), bits(vp), [prompt - 1] * B, w, s)
    for b in (0, 2):
        assert_close(o[b:b + 1], ref[b:b + 1], f"b={b}")
