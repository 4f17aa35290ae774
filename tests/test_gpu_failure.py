"""Failure detection without a GPU fault: a bounded wait that runs out.

The library's kernels never wait without a limit: every mbarrier wait gives
up after SWA_WAIT_LIMIT_NS (0.2 s), records SWA_ERR_TIMEOUT in the device
error word, releases what it holds and returns.  swa_selftest_wait_timeout
runs that path on purpose -- a wait on a barrier nothing arrives on, with a
TMEM allocation held -- and the host reads the status.  Afterwards the
context must still compute correctly.
"""
import time

import pytest
import torch

import oracle
from gpu_helpers import assert_close, bits
from sliding_window_attention_prefill_gb300 import build, device_error, inputs, prefill
from sliding_window_attention_prefill_gb300 import swa as binding

pytestmark = pytest.mark.gpu


def test_wait_limit_reports_timeout_and_context_survives():
    build.build()
    assert device_error() == 0
    t0 = time.perf_counter()
    binding.selftest_wait_timeout()
    assert device_error() == -6          # SWA_ERR_TIMEOUT, read once ...
    waited = time.perf_counter() - t0
    assert device_error() == 0           # ... and cleared
    assert 0.15 < waited < 5.0, waited   # the 0.2 s limit, not a hang
    # the context (and TMEM, freed by the timed-out kernel) is still usable
    q, k, v = inputs.prefill_inputs(1, 300, 8, 2, 128, seed=4)
    o = prefill(q.cuda(), k.cuda(), v.cuda(), 64, 4)
    torch.cuda.synchronize()
    assert device_error() == 0
    ref, _ = oracle.get().prefill(bits(q), bits(k), bits(v), 64, 4)
    assert_close(o, ref, "prefill after a timed-out wait")
