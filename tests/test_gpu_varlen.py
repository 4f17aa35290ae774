"""Variable-length (ragged) prefill on the GPU against the fp64 oracle.

Sequences of different lengths are packed along the first dimension; every
sequence's rows must equal the oracle's prefill of that sequence alone, and
no row of another sequence may be touched.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, bits
from sliding_window_attention_prefill_gb300 import W_INF, build, device_error, inputs, prefill_varlen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()


def _packed(lengths, Hq, Hkv, d, dtype, seed):
    total = int(sum(lengths))
    q, k, v = inputs.prefill_inputs(1, total, Hq, Hkv, d, seed=seed, dtype=dtype)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return q[0], k[0], v[0], cu


def _check(lengths, Hq, Hkv, d, w, s, dtype=torch.bfloat16, seed=0):
    q, k, v, cu = _packed(lengths, Hq, Hkv, d, dtype, seed)
    total = q.shape[0]
    out = torch.full((total, Hq, d), float("nan"), dtype=dtype, device="cuda")
    o, lse = prefill_varlen(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(cu).cuda(), w, s,
                            max_len=max(lengths), out=out, return_lse=True)
    torch.cuda.synchronize()
    assert device_error() == 0
    o, lse = o.cpu(), lse.cpu()
    dt = "f16" if dtype == torch.float16 else "bf16"
    orc = oracle.get()
    for b, n in enumerate(lengths):
        if n == 0:
            continue
        a, e = int(cu[b]), int(cu[b + 1])
        ref_o, ref_l = orc.prefill(bits(q[a:e].unsqueeze(0)), bits(k[a:e].unsqueeze(0)),
                                   bits(v[a:e].unsqueeze(0)), w, s, dtype=dt)
        assert_close(o[a:e].unsqueeze(0), ref_o, f"sequence {b} (n={n})")
        assert_close(lse[:, a:e].unsqueeze(0), ref_l, f"lse of sequence {b}", max_abs=4e-3,
                     mean_rel=1e-3)


CASES = [
    # lengths, Hq, Hkv, d, w, s
    ([1, 31, 32, 33, 100, 300, 0, 513], 32, 8, 128, 64, 4),   # G=4, tails of every kind, empty
    ([5, 128, 129, 400], 4, 4, 64, 96, 0),                     # G=1 (128 positions per tile)
    ([17, 200, 3, 64], 16, 2, 128, W_INF, 0),                  # G=8, full causal
    ([1500, 10, 700], 32, 8, 128, 512, 4),                     # several key tiles per unit
    ([1600, 50], 8, 2, 128, 1400, 4),                          # 256-column key tiles
    ([3, 9, 2], 8, 2, 64, 16, 12),                             # 12 sinks, sequences shorter than s
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "n{}-Hq{}Hkv{}d{}w{}s{}".format(
    "_".join(map(str, c[0][:4])), *c[1:]))
def test_varlen_matches_each_sequence(case):
    lengths, Hq, Hkv, d, w, s = case
    _check(lengths, Hq, Hkv, d, w, s, seed=len(lengths))


def test_varlen_fp16_pages_shape():
    """The pages' attention shape (16 heads of 64, fp16) as a ragged batch."""
    _check([1000, 37, 512, 1], 16, 16, 64, 64, 4, dtype=torch.float16, seed=3)


def test_varlen_random_ragged_batch():
    """Forty sequences with seeded random lengths in [0, 300]."""
    rng = np.random.default_rng(11)
    lengths = [int(x) for x in rng.integers(0, 301, 40)]
    _check(lengths, 32, 8, 128, 128, 4, seed=4)


def test_varlen_invalid_cu_seqlens_computes_nothing():
    """A cu_seqlens that is not a partition of [0, total): SWA_ERR_BOUNDS on
    the device, the output untouched."""
    q, k, v, _ = _packed([64, 64], 8, 2, 128, torch.bfloat16, 5)
    for cu in ([0, 70, 64], [0, 64, 100], [1, 64, 128]):
        out = torch.full((128, 8, 128), 7.0, dtype=torch.bfloat16, device="cuda")
        prefill_varlen(q.cuda(), k.cuda(), v.cuda(), torch.tensor(cu, dtype=torch.int32).cuda(), 64, 4,
                       out=out)
        assert device_error() == -7, cu
        assert torch.all(out == 7.0), cu
