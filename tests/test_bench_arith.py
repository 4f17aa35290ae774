"""The algorithmic work figures the bench's roofline divides by (CPU only).

`achieved` in the bench line is bytes (or flops) per launch over the launch
time, so these counts decide the reported fraction of peak.  They are pinned
here to counts taken independently: the attended set A(t) of the oracle's
window test, summed position by position, and the tensor sizes of the
workload.
"""
import pytest

import bench
import oracle


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


@pytest.mark.parametrize("L,w,s", [(1, 64, 4), (10, 4, 2), (37, 8, 4), (64, 64, 4), (65, 64, 4),
                                   (100, 16, 0), (23, -1, 0), (300, 64, 4)])
def test_window_sum_is_the_attended_pairs(orc, L, w, s):
    pairs = sum(len(orc.window(t, w, s)) for t in range(L))
    assert bench.window_sum(L, w) == pairs


def test_flops_count_two_products_per_attended_pair(orc):
    # per (batch, query head, position t, attended key i): q.k and p.v, d
    # multiply-adds each, 2 flops per multiply-add
    B, L, Hq, d, w, s = 2, 50, 3, 16, 12, 4
    pairs = sum(len(orc.window(t, w, s)) for t in range(L))
    assert bench.prefill_flops(B, L, Hq, d, w) == B * Hq * pairs * 2 * (2 * d)


def test_prefill_bytes_read_q_k_v_once_and_write_o():
    B, L, Hq, Hkv, d = 2, 7, 8, 2, 64
    elems = B * L * Hq * d * 2 + B * L * Hkv * d * 2  # q and o; k and v
    assert bench.prefill_bytes(B, L, Hq, Hkv, d) == 2 * elems


def test_decode_bytes():
    # q read and o written; the new k, v read and written to the cache; the
    # K and V rows of the n_valid attended slots read
    B, Hq, Hkv, d, n = 3, 8, 2, 64, 40
    expect = 2 * B * (2 * Hq * d + 4 * Hkv * d + 2 * Hkv * d * n)
    assert bench.decode_bytes(B, Hq, Hkv, d, n) == expect


def test_the_bench_workload_figures():
    """Prefill SWA(64,4), B=1, L=4096, 32 query and 8 key/value heads of 128:
    Q and O of 32 MiB, K and V of 8 MiB; 4.26 GFLOP over the window."""
    W = bench.WORK
    assert bench.prefill_bytes(W["B"], W["L"], W["Hq"], W["Hkv"], W["d"]) == 83886080
    assert bench.window_sum(W["L"], W["w"]) == 64 * 65 // 2 + (4096 - 64) * 64
    assert bench.prefill_flops(W["B"], W["L"], W["Hq"], W["d"], W["w"]) == 4261937152
    assert bench.tokens_per_step(1) == 4097
