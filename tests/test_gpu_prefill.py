"""Prefill parity: the CUDA path against the fp64 oracle (GPU)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, bits
from sliding_window_attention_prefill_gb300 import W_INF, build, inputs, prefill

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def _run(B, L, Hq, Hkv, d, w, s, seed=0, sink_rows=0, lse=True):
    q, k, v = inputs.prefill_inputs(B, L, Hq, Hkv, d, seed=seed, sink_rows=sink_rows)
    o, l = prefill(q.cuda(), k.cuda(), v.cuda(), w, s, return_lse=True)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.get().prefill(bits(q), bits(k), bits(v), w, s)
    assert_close(o, ref_o, f"o {B, L, Hq, Hkv, d, w, s}")
    if lse:
        # l sums the bf16-rounded weights the P*V product uses, each within a
        # relative 2^-9 of its exact value, so ln(l) is within ~2^-9 of the
        # exact log-sum-exp (plus fp32 / ex2.approx error): bound 4e-3.
        assert_close(l, ref_l, f"lse {B, L, Hq, Hkv, d, w, s}", max_abs=4e-3, mean_rel=1e-3)
    return o


def test_tiny_config():
    """SWA(64,4), B=1, L=256, Hq=4, Hkv=1, d=64 -- the small case the oracle runs in full."""
    _run(1, 256, 4, 1, 64, 64, 4)


CASES = [
    # B, L, Hq, Hkv, d, w, s
    (2, 300, 8, 2, 128, 64, 4),      # ragged tail, GQA 4, two sequences
    (1, 200, 2, 2, 64, 96, 0),       # MHA (G=1, 128 positions per tile), no sinks
    (1, 333, 4, 2, 128, W_INF, 0),   # full causal, several key tiles per query tile
    (1, 150, 4, 1, 64, 1000, 4),     # window longer than the prompt = causal
    (1, 100, 16, 2, 64, 40, 4),      # G=8: 16 positions per tile
    (1, 77, 32, 2, 128, 20, 4),      # G=16: 8 positions per tile
    (1, 90, 4, 1, 128, 16, 12),      # 12 sinks (16 sink rows), tiny ring
    (1, 1100, 4, 1, 128, 512, 4),    # long window: 5 key tiles per query tile
    (1, 5, 4, 1, 64, 64, 4),         # every position is a sink position
    (1, 1, 8, 2, 128, 64, 4),        # one token
    (3, 129, 4, 4, 64, 33, 1),       # odd window and one sink
    # Long windows (a unit of G=4 spans w + 35 key columns): 112-column
    # tiles up to 1280 columns at d=128, ending in a 16-column MMA step
    # (w=989) or a 17-column one rounded to 32 (w=990); 256-column tiles
    # beyond, ending in a single column (w=1246) or exactly (w=1501); d=64
    # with 128-column tiles.
    (1, 2600, 8, 2, 128, 989, 4),
    (1, 2600, 8, 2, 128, 990, 4),
    (1, 2600, 8, 2, 128, 1246, 4),
    (1, 2600, 8, 2, 128, 1501, 4),
    (1, 5000, 4, 1, 128, 2048, 4),
    (2, 700, 8, 2, 64, 300, 4),      # d=64 on the two-tile kernel, two sequences
    (1, 900, 4, 4, 64, 300, 4),      # d=64, G=1: 256-column tiles (2 instead of 4 of 128)
    # Large groups over several key tiles (the epilogue warpgroup's row ->
    # position / head mapping): G=16 (8 positions per unit) and G=8 at d=64.
    (1, 600, 32, 2, 128, 300, 4),
    (2, 400, 16, 2, 64, 300, 4),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}L{}Hq{}Hkv{}d{}w{}s{}".format(*c))
def test_shapes(case):
    _run(*case)


def test_llama_shape_sink_heavy_full():
    """SWA(64,4), B=1, L=4096, Hq=32, Hkv=8, d=128, first 4 key rows x8: every output row."""
    _run(1, 4096, 32, 8, 128, 64, 4, sink_rows=4)


@pytest.mark.parametrize("w", [128, 256, 512])
def test_long_prompt_sampled(w):
    """B=2, L=32768, Hq=32, Hkv=8, d=128, SWA(w,4): sampled rows against the oracle."""
    B, L, Hq, Hkv, d, s = 2, 32768, 32, 8, 128, 4
    q, k, v = _long_inputs()
    o = prefill(q.cuda(), k.cuda(), v.cuda(), w, s)
    torch.cuda.synchronize()
    rng = np.random.default_rng(w)
    n = 768
    rows = np.stack([rng.integers(0, B, n), rng.integers(0, L, n), rng.integers(0, Hq, n)], 1)
    edge_t = [0, 1, 3, 4, 5, 31, 32, 33, w - 1, w, w + 1, L - 33, L - 32, L - 1]
    extra = np.array([[b, t, h] for b in range(B) for t in edge_t for h in (0, 3, Hq - 1)])
    rows = np.concatenate([rows, extra]).astype(np.int64)
    ref, _ = oracle.get().prefill_rows(_long_bits["q"], _long_bits["k"], _long_bits["v"], rows, w, s)
    got = o.cpu()[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert_close(got, ref, f"L=32768 SWA({w},4)")


_long = {}
_long_bits = {}


def _long_inputs():
    if not _long:
        q, k, v = inputs.prefill_inputs(2, 32768, 32, 8, 128, seed=0)
        _long.update(q=q, k=k, v=v)
        _long_bits.update(q=bits(q), k=bits(k), v=bits(v))
    return _long["q"], _long["k"], _long["v"]


def test_deterministic_and_empty():
    q, k, v = inputs.prefill_inputs(1, 500, 8, 2, 128, seed=3)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    a = prefill(q, k, v, 128, 4)
    b = prefill(q, k, v, 128, 4)
    assert torch.equal(a, b)
    z = prefill(q[:, :0].contiguous(), k[:, :0].contiguous(), v[:, :0].contiguous(), 64, 4)
    assert z.shape[1] == 0


@pytest.mark.parametrize("case", [(2, 300, 8, 2, 128, 64, 0), (2, 1100, 8, 2, 128, 512, 4),
                                  (2, 300, 8, 2, 64, 64, 4), (1, 700, 4, 1, 128, W_INF, 0)],
                         ids=lambda c: "B{}L{}Hq{}Hkv{}d{}w{}s{}".format(*c))
def test_repeatable(case):
    """Bit-identical outputs and LSE over repeated calls.  The CTAs of a call
    land on different SMs from call to call, so a read of anything a kernel
    did not write itself (stale shared or tensor memory) shows up here even
    when it stays inside the parity tolerance."""
    B, L, Hq, Hkv, d, w, s = case
    q, k, v = inputs.prefill_inputs(B, L, Hq, Hkv, d, seed=3)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o0, l0 = prefill(q, k, v, w, s, return_lse=True)
    for _ in range(7):
        o, l = prefill(q, k, v, w, s, return_lse=True)
        assert torch.equal(o, o0) and torch.equal(l, l0)
