"""Chunked prefill from a cache (GPU) against the fp64 oracle.

A prompt prefilled chunk by chunk with prefill_chunk must give, chunk by
chunk, the rows of the oracle's prefill of the whole prompt (each position's
attended set is the same), and leave the cache the oracle's append
simulation builds from the whole prompt, byte for byte.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, bits
from sliding_window_attention_prefill_gb300 import (W_INF, Cache, build, device_error, inputs,
                                                    prefill_chunk)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


CASES = [
    # B, Hq, Hkv, d, w, s, chunk sizes
    (2, 8, 2, 128, 64, 4, [300, 1, 200, 499]),        # chunks longer and shorter than w, n = 1
    (1, 32, 8, 128, 512, 4, [1024, 1024, 952]),       # the first chunk fills the cache
    (1, 8, 2, 128, 64, 4, [40, 40, 40, 41]),          # starts before w, then wraps
    (2, 4, 4, 64, 16, 12, [7, 30, 5, 100]),           # G = 1, d = 64, 12 sinks of 16
    (1, 16, 2, 64, 96, 0, [128, 128, 77]),            # G = 8, no sinks
    (1, 8, 2, 128, 1400, 4, [900, 700]),              # 256-column key tiles
    (1, 8, 2, 64, W_INF, 0, [128, 300, 272]),         # infinite window, in place
    (2, 32, 8, 128, W_INF, 0, [500, 1, 523]),         # infinite window, d = 128
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "B{}Hq{}Hkv{}d{}w{}s{}n{}".format(
    *c[:6], "-".join(map(str, c[6]))))
def test_chunks_equal_whole_prompt(case):
    B, Hq, Hkv, d, w, s, chunks = case
    L = sum(chunks)
    q, k, v = inputs.prefill_inputs(B, L, Hq, Hkv, d, seed=17)
    ref_o, ref_lse = oracle.get().prefill(bits(q), bits(k), bits(v), w, s)
    cache = Cache(B, Hkv, d, w, s, max_len=(L + 16 if w == W_INF else None))
    pos0 = 0
    for i, n in enumerate(chunks):
        sl = slice(pos0, pos0 + n)
        o, lse = prefill_chunk(q[:, sl].contiguous().cuda(), k[:, sl].contiguous().cuda(),
                               v[:, sl].contiguous().cuda(), cache, pos0, return_lse=True)
        torch.cuda.synchronize()
        assert device_error() == 0
        assert_close(o, ref_o[:, sl], f"chunk {i} at {pos0} (n={n})")
        assert_close(lse, ref_lse[:, :, sl], f"lse of chunk {i}", max_abs=4e-3, mean_rel=1e-3)
        pos0 += n
    hk = np.zeros((B, Hkv, cache.cap, d), np.uint16)
    hv = np.zeros_like(hk)
    oracle.get().cache_append(hk, hv, bits(k), bits(v), 0, w, s)
    ck, cv = bits(cache.k), bits(cache.v)
    if w == W_INF:  # slots past the prompt were never written
        ck, cv, hk, hv = ck[:, :, :L], cv[:, :, :L], hk[:, :, :L], hv[:, :, :L]
    assert np.array_equal(ck, hk), "cache K after the last chunk"
    assert np.array_equal(cv, hv), "cache V after the last chunk"


def test_llama_prompt_in_chunks():
    """SWA(64,4) Llama shape (Hq=32, Hkv=8, d=128), sink-heavy keys, a
    4096-token prompt in 512-token chunks: every output row."""
    B, L, Hq, Hkv, d, w, s, n = 1, 4096, 32, 8, 128, 64, 4, 512
    q, k, v = inputs.prefill_inputs(B, L, Hq, Hkv, d, seed=0, sink_rows=4)
    ref_o, _ = oracle.get().prefill(bits(q), bits(k), bits(v), w, s)
    cache = Cache(B, Hkv, d, w, s)
    outs = []
    for pos0 in range(0, L, n):
        sl = slice(pos0, pos0 + n)
        outs.append(prefill_chunk(q[:, sl].contiguous().cuda(), k[:, sl].contiguous().cuda(),
                                  v[:, sl].contiguous().cuda(), cache, pos0))
    o = torch.cat(outs, dim=1)
    torch.cuda.synchronize()
    assert device_error() == 0
    assert_close(o, ref_o, "4096 tokens in chunks of 512")
