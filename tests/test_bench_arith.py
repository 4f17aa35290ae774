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
    """The configurations the line measures, Llama attention shape (32 query
    and 8 key/value heads of 128, bf16).
    Prefill B=2, L=32768: Q and O of 512 MiB, K and V of 128 MiB; 137.2,
    273.8 and 545.5 GFLOP over the windows 128, 256, 512.
    Decode B=64 after a 4096-token prompt: the cache holds w slots, each
    step reads K and V of all of them (128 MiB at w=512) and 2 x 64 x 1024
    tokens are decoded per step.
    The 4096-token SWA(64,4) prompt: Q and O of 32 MiB, K and V of 8 MiB."""
    P, D, S = bench.PREFILL_CFG, bench.DECODE_CFG, bench.SMALL_PREFILL
    assert bench.prefill_bytes(P["B"], P["L"], P["Hq"], P["Hkv"], P["d"]) == 1342177280
    gf = [bench.prefill_flops(P["B"], P["L"], P["Hq"], P["d"], w) / 1e9 for w in P["windows"]]
    assert [round(x, 1) for x in gf] == [137.2, 273.8, 545.5]
    assert bench.window_sum(P["L"], 512) == 512 * 513 // 2 + (32768 - 512) * 512
    assert bench.kv_read_bytes(D["B"], D["Hkv"], D["d"], 512) == 128 << 20
    assert bench.decode_bytes(D["B"], D["Hq"], D["Hkv"], D["d"], 512) == 135790592
    assert bench.decoded_tokens_per_step(1) == 131072 * 16
    assert bench.prefill_bytes(S["B"], S["L"], S["Hq"], S["Hkv"], S["d"]) == 83886080
    assert bench.prefill_flops(S["B"], S["L"], S["Hq"], S["d"], S["w"]) == 4261937152


def test_roofline_entry_picks_the_bound_by_intensity():
    pk = {"hbm_gbs": 6794.5, "bf16_tflops": 1924.1, "source": "measured"}
    P = bench.PREFILL_CFG
    by = bench.prefill_bytes(P["B"], P["L"], P["Hq"], P["Hkv"], P["d"])
    for w, bound in [(128, "hbm"), (256, "hbm"), (512, "tensor")]:
        fl = bench.prefill_flops(P["B"], P["L"], P["Hq"], P["d"], w)
        e = bench.roofline_entry("k", 1.0, fl, by, pk)
        assert e["bound"] == bound
        if bound == "tensor":
            assert abs(e["achieved"] - fl / 1e-3 / 1e12) < 1e-6 * e["achieved"]
        else:
            assert abs(e["achieved"] - by / 1e-3 / 1e9) < 1e-6 * e["achieved"]
        assert abs(e["frac"] - e["achieved"] / e["peak"]) < 1e-12
