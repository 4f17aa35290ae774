"""Checks that pin the oracle to things other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError on
a mismatch.  ``test_oracle.py`` runs them against the oracle as built; the
mutation test runs them against copies of the oracle with a plausible mistake
planted in the C source and expects at least one pin to fail for each.

What pins what:
  * hand-written fixtures of attended sets and cache contents
    (tests/golden/, each line citing the page statement it follows);
  * brute force: dense L x L attention with a boolean mask built by slicing
    "the first s" and "the latest w-s" positions, in numpy;
  * a library routine: torch's scaled_dot_product_attention (fp64, causal),
    which SWA(w,s) must equal when the window covers the whole prefix;
  * fp16 inputs: every one of the 65536 binary16 bit patterns widened by the
    oracle equals numpy's float16 -> float64 conversion, and brute force on
    fp16 inputs (widened by numpy) matches every attention entry point;
  * the hybrid window + linear decode: a numpy restatement of its definition
    with dense masks, the no-eviction case (equal to SWA decode), W = 0 (a
    closed form: every linear weight is the feature count), and the state
    form (S, z) giving the same outputs as the direct sum;
  * closed forms: t = 0 gives v_0; q = 0 gives the plain mean of the attended
    values; two keys in d = 1 give a two-term weighted mean;
  * invariants: equal values give that value; permuting the history inside
    the attended set changes nothing; decoding at position t equals prefill
    row t; decoding over the ring cache equals decoding over the history.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import oracle as oracle_mod
from oracle import W_INF, bits_to_f64

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden")


def _bf16(x: np.ndarray) -> np.ndarray:
    return oracle_mod.bf16_bits(torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16))


def _rand_bits(rng: np.random.Generator, shape) -> np.ndarray:
    return _bf16(rng.standard_normal(shape).astype(np.float32))


def _rand_f16_bits(rng: np.random.Generator, shape) -> np.ndarray:
    """N(0,1) rounded to IEEE binary16 by numpy, as bit patterns."""
    return np.ascontiguousarray(rng.standard_normal(shape).astype(np.float16).view(np.uint16))


def _f16_to_f64(bits: np.ndarray) -> np.ndarray:
    """numpy's own binary16 -> float64 conversion of bit patterns."""
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def _parse_ranges(text: str) -> list[int]:
    out: list[int] = []
    for part in text.split(","):
        lo, hi = part.strip().split("-")
        out.extend(range(int(lo), int(hi) + 1))
    return out


def _read_fixture(name: str):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, ranges, cite = [x.strip() for x in line.split("|")]
            a, b, c = head.split()
            w = W_INF if a == "inf" else int(a)
            rows.append((w, int(b), int(c), _parse_ranges(ranges), cite))
    return rows


def _first_and_latest(t: int, w: int, s: int) -> list[int]:
    """The attended set built by slicing the prefix [0..t]: first s, latest w-s."""
    prefix = list(range(t + 1))
    if w == W_INF:
        return prefix
    first = prefix[:s]
    latest = prefix[-(w - s):] if w - s <= len(prefix) else prefix
    return sorted(set(first) | set(latest))


def _dense_reference(q, k, v, w, s, widen=bits_to_f64):
    """Brute-force masked attention: full score matrix, -inf outside the set."""
    qf, kf, vf = widen(q), widen(k), widen(v)
    B, L, Hq, d = qf.shape
    Hkv = kf.shape[2]
    G = Hq // Hkv
    mask = np.zeros((L, L), dtype=bool)
    for t in range(L):
        mask[t, _first_and_latest(t, w, s)] = True
    o = np.zeros_like(qf)
    for b in range(B):
        for h in range(Hq):
            kk = kf[b, :, h // G, :]
            vv = vf[b, :, h // G, :]
            sc = (qf[b, :, h, :] @ kk.T) / math.sqrt(d)
            sc = np.where(mask, sc, -np.inf)
            sc = sc - sc.max(axis=1, keepdims=True)
            p = np.exp(sc)
            o[b, :, h, :] = (p @ vv) / p.sum(axis=1, keepdims=True)
    return o


def _sdpa_causal(q, k, v):
    """torch scaled_dot_product_attention in fp64 with a causal mask (BSHD in/out)."""
    qf, kf, vf = (torch.from_numpy(bits_to_f64(x)) for x in (q, k, v))
    G = qf.shape[2] // kf.shape[2]
    kf = kf.repeat_interleave(G, dim=2)
    vf = vf.repeat_interleave(G, dim=2)
    out = torch.nn.functional.scaled_dot_product_attention(
        qf.transpose(1, 2), kf.transpose(1, 2), vf.transpose(1, 2), is_causal=True)
    return out.transpose(1, 2).numpy()


# ---------------------------------------------------------------------------
def pin_golden_sets(orc) -> None:
    for w, s, t, expect, cite in _read_fixture("attended_sets.txt"):
        got = orc.window(t, w, s)
        assert got == expect, f"A({t}) for SWA({w},{s}) [{cite}]: {got[:8]}... != {expect[:8]}..."


def pin_window_size(orc) -> None:
    for w, s in [(8, 0), (8, 2), (8, 7), (5, 1), (64, 4)]:
        for t in range(0, 3 * w):
            n = len(orc.window(t, w, s))
            assert n == min(t + 1, w), (w, s, t, n)


def pin_brute_force(orc) -> None:
    rng = np.random.default_rng(1)
    cases = [(2, 37, 4, 2, 8, 8, 2), (1, 29, 2, 2, 16, 5, 0), (1, 40, 4, 1, 8, 12, 4),
             (1, 23, 3, 1, 4, 64, 4), (1, 33, 2, 1, 8, W_INF, 0), (1, 21, 8, 2, 8, 6, 5)]
    for B, L, Hq, Hkv, d, w, s in cases:
        q = _rand_bits(rng, (B, L, Hq, d))
        k = _rand_bits(rng, (B, L, Hkv, d))
        v = _rand_bits(rng, (B, L, Hkv, d))
        o, _ = orc.prefill(q, k, v, w, s, threads=2)
        ref = _dense_reference(q, k, v, w, s)
        err = np.abs(o - ref).max()
        assert err < 1e-12, f"brute force {B, L, Hq, Hkv, d, w, s}: {err}"


def pin_causal_library(orc) -> None:
    rng = np.random.default_rng(2)
    B, L, Hq, Hkv, d = 2, 48, 4, 2, 16
    q = _rand_bits(rng, (B, L, Hq, d))
    k = _rand_bits(rng, (B, L, Hkv, d))
    v = _rand_bits(rng, (B, L, Hkv, d))
    ref = _sdpa_causal(q, k, v)
    for w, s in [(W_INF, 0), (L, 4), (L + 7, 0), (1000, 3)]:
        o, _ = orc.prefill(q, k, v, w, s, threads=2)
        assert np.abs(o - ref).max() < 1e-12, (w, s)
    # rows whose prefix fits the window are plain causal attention
    for w, s in [(16, 4), (9, 0), (12, 11)]:
        o, _ = orc.prefill(q, k, v, w, s, threads=2)
        assert np.abs(o[:, :w] - ref[:, :w]).max() < 1e-12, (w, s)
        assert np.abs(o[:, w:] - ref[:, w:]).max() > 1e-6, (w, s)


def pin_closed_forms(orc) -> None:
    rng = np.random.default_rng(3)
    B, L, Hq, Hkv, d = 1, 30, 4, 2, 8
    q = _rand_bits(rng, (B, L, Hq, d))
    k = _rand_bits(rng, (B, L, Hkv, d))
    v = _rand_bits(rng, (B, L, Hkv, d))
    vf = bits_to_f64(v)
    o, _ = orc.prefill(q, k, v, 6, 2, threads=1)
    for h in range(Hq):                      # t = 0 attends only to itself
        assert np.array_equal(o[0, 0, h], vf[0, 0, h // 2])
    zero = np.zeros_like(q)                  # q = 0: uniform weights over A(t)
    o, _ = orc.prefill(zero, k, v, 6, 2, threads=1)
    for t in range(L):
        idx = _first_and_latest(t, 6, 2)
        for h in range(Hq):
            mean = vf[0, idx, h // 2].mean(axis=0)
            assert np.abs(o[0, t, h] - mean).max() < 1e-12, (t, h)
    # d = 1, two keys: a two-term weighted mean with weights exp(q k_i)
    q1 = _bf16(np.array([0.75], np.float32)).reshape(1, 1, 1, 1).repeat(2, axis=1)
    k1 = _bf16(np.array([1.5, -0.5], np.float32)).reshape(1, 2, 1, 1)
    v1 = _bf16(np.array([2.0, 10.0], np.float32)).reshape(1, 2, 1, 1)
    o, lse = orc.prefill(q1, k1, v1, W_INF, 0, threads=1)
    a, b = 0.75 * 1.5, 0.75 * -0.5
    expect = (math.exp(a) * 2.0 + math.exp(b) * 10.0) / (math.exp(a) + math.exp(b))
    assert abs(o[0, 1, 0, 0] - expect) < 1e-14
    assert abs(lse[0, 0, 1] - math.log(math.exp(a) + math.exp(b))) < 1e-14


def pin_equal_values(orc) -> None:
    rng = np.random.default_rng(4)
    B, L, Hq, Hkv, d = 2, 40, 4, 1, 8
    q = _rand_bits(rng, (B, L, Hq, d))
    k = _rand_bits(rng, (B, L, Hkv, d))
    row = _rand_bits(rng, (B, 1, Hkv, d))
    v = np.ascontiguousarray(np.repeat(row, L, axis=1))
    o, _ = orc.prefill(q, k, v, 10, 3, threads=2)
    vf = bits_to_f64(row)
    for h in range(Hq):
        assert np.abs(o[:, :, h] - vf[:, :, 0]).max() < 1e-13


def pin_decode_history(orc) -> None:
    """Decode at position t equals prefill row t; permutations inside A(t) change nothing."""
    rng = np.random.default_rng(5)
    B, P, Hq, Hkv, d, w, s = 2, 50, 4, 2, 8, 12, 3
    q = _rand_bits(rng, (B, P, Hq, d))
    k = _rand_bits(rng, (B, P, Hkv, d))
    v = _rand_bits(rng, (B, P, Hkv, d))
    o_pre, _ = orc.prefill(q, k, v, w, s, threads=2)
    for t in [0, 2, 11, 12, 30, P - 1]:
        o_dec = orc.decode(np.ascontiguousarray(q[:, t]), k, v, [t] * B, w, s, threads=2)
        assert np.abs(o_dec - o_pre[:, t]).max() < 1e-13, t
    t = P - 1
    idx = _first_and_latest(t, w, s)
    perm = rng.permutation(idx)
    kp, vp = k.copy(), v.copy()
    kp[:, idx] = k[:, perm]
    vp[:, idx] = v[:, perm]
    qt = np.ascontiguousarray(q[:, t])
    a = orc.decode(qt, k, v, [t] * B, w, s, threads=1)
    b = orc.decode(qt, kp, vp, [t] * B, w, s, threads=1)
    assert np.abs(a - b).max() < 1e-12
    # changing a key outside A(t) leaves the result as it is; changing one
    # inside A(t) (the oldest of the latest w-s) does not
    outside = [i for i in range(t + 1) if i not in idx]
    kq = k.copy()
    kq[:, outside[-1]] = k[:, idx[-1]]
    c = orc.decode(qt, kq, v, [t] * B, w, s, threads=1)
    assert np.abs(a - c).max() == 0.0
    kr = k.copy()
    kr[:, idx[s]] = k[:, idx[-1]]
    e = orc.decode(qt, kr, v, [t] * B, w, s, threads=1)
    assert np.abs(a - e).max() > 1e-9


def pin_golden_cache(orc) -> None:
    """Cache contents after a prompt match the hand-written fixtures."""
    for w, s, P, expect, cite in _read_fixture("cache_contents.txt"):
        B, Hkv, d = 1, 1, 2
        ck = np.zeros((B, Hkv, w, d), np.uint16)
        cv = np.zeros((B, Hkv, w, d), np.uint16)
        # payload: the position in the low 15 bits (+1 so that 0 means "empty")
        pay = (np.arange(P, dtype=np.uint16) + 1).reshape(1, P, 1, 1).repeat(d, axis=3)
        orc.cache_append(ck, cv, pay, pay, 0, w, s)
        held = sorted(int(x) - 1 for x in ck[0, 0, :, 0] if x != 0)
        assert held == expect, f"SWA({w},{s}) after {P} [{cite}]: {held[:6]}..."
        assert np.array_equal(ck, cv)


def pin_ring_mapping(orc) -> None:
    """Exhaustive over p < 4w: slots stay in [0, w) and the cache holds A(p)."""
    for w, s in [(8, 0), (8, 3), (9, 4), (64, 4), (5, 4), (16, 1)]:
        cap = w
        ck = np.zeros((1, 1, cap, 1), np.uint16)
        cv = np.zeros((1, 1, cap, 1), np.uint16)
        for p in range(4 * w):
            slot = orc.cache_slot(p, w, s)
            assert 0 <= slot < cap, (w, s, p, slot)
            pay = np.array([[[[p + 1]]]], np.uint16)
            orc.cache_append(ck, cv, pay, pay, p, w, s)
            held = sorted(int(x) - 1 for x in ck[0, 0, :, 0] if x != 0)
            assert held == _first_and_latest(p, w, s), (w, s, p)
        # bulk append of the same stream gives the same bits
        bk = np.zeros_like(ck)
        bv = np.zeros_like(cv)
        pay = (np.arange(4 * w, dtype=np.uint16) + 1).reshape(1, 4 * w, 1, 1)
        orc.cache_append(bk, bv, pay, pay, 0, w, s)
        assert np.array_equal(bk, ck), (w, s)


def pin_decode_cache(orc) -> None:
    """Decode over the ring cache equals decode over the full history."""
    rng = np.random.default_rng(6)
    B, Hq, Hkv, d = 2, 4, 2, 8
    for w, s, P in [(16, 4, 60), (16, 4, 10), (7, 0, 30), (W_INF, 0, 25)]:
        cap = P if w == W_INF else w
        k = _rand_bits(rng, (B, P, Hkv, d))
        v = _rand_bits(rng, (B, P, Hkv, d))
        q = _rand_bits(rng, (B, Hq, d))
        ck = np.zeros((B, Hkv, cap, d), np.uint16)
        cv = np.zeros((B, Hkv, cap, d), np.uint16)
        orc.cache_append(ck, cv, k[:, : P // 2], v[:, : P // 2], 0, w, s)
        for j in range(P // 2, P):
            orc.cache_append(ck, cv, np.ascontiguousarray(k[:, j:j + 1]),
                             np.ascontiguousarray(v[:, j:j + 1]), j, w, s)
        a = orc.decode(q, k, v, [P - 1] * B, w, s, threads=2)
        b = orc.decode_cache(q, ck, cv, [P - 1] * B, w, s, threads=2)
        assert np.abs(a - b).max() < 1e-12, (w, s, P)


def pin_rows_match_full(orc) -> None:
    """The selected-rows entry gives the same rows as the full prefill (so the
    sampled parity checks at full size inherit the full prefill's pins)."""
    rng = np.random.default_rng(7)
    B, L, Hq, Hkv, d, w, s = 2, 45, 8, 2, 16, 10, 3
    q = _rand_bits(rng, (B, L, Hq, d))
    k = _rand_bits(rng, (B, L, Hkv, d))
    v = _rand_bits(rng, (B, L, Hkv, d))
    o, lse = orc.prefill(q, k, v, w, s, threads=2)
    rows = np.array([[b, t, h] for b in range(B) for t in (0, 2, 9, 10, 44) for h in (0, 5, 7)])
    ro, rl = orc.prefill_rows(q, k, v, rows, w, s, threads=2)
    assert np.array_equal(ro, o[rows[:, 0], rows[:, 1], rows[:, 2]])
    assert np.array_equal(rl, lse[rows[:, 0], rows[:, 2], rows[:, 1]])


def pin_f16_every_pattern(orc) -> None:
    """t = 0 attends only to itself, so o = v_0 exactly: with v_0 holding all
    65536 binary16 bit patterns (q = k = 0), the oracle's fp16 widening must
    agree with numpy's for each one (zeros, subnormals, normals, infinities,
    NaN)."""
    v = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).reshape(1, 1, 1, 1 << 16)
    z = np.zeros_like(v)
    o, _ = orc.prefill(z, z, v, W_INF, 0, threads=1, dtype="f16")
    ref = _f16_to_f64(v)
    assert np.array_equal(o, ref, equal_nan=True), "fp16 widening"
    # the same bits read as bf16 give other values: the type argument is used
    o_bf, _ = orc.prefill(z, z, v, W_INF, 0, threads=1)
    assert not np.array_equal(o_bf, ref, equal_nan=True)


def pin_f16_brute_force(orc) -> None:
    """fp16 inputs through prefill, prefill_rows, decode and decode over the
    cache, against dense masked attention on numpy-widened values."""
    rng = np.random.default_rng(8)
    for B, L, Hq, Hkv, d, w, s in [(1, 37, 4, 4, 16, 8, 2), (2, 30, 4, 2, 8, W_INF, 0),
                                   (1, 41, 2, 1, 8, 12, 4)]:
        q = _rand_f16_bits(rng, (B, L, Hq, d))
        k = _rand_f16_bits(rng, (B, L, Hkv, d))
        v = _rand_f16_bits(rng, (B, L, Hkv, d))
        ref = _dense_reference(q, k, v, w, s, widen=_f16_to_f64)
        o, _ = orc.prefill(q, k, v, w, s, threads=2, dtype="f16")
        assert np.abs(o - ref).max() < 1e-12, ("prefill", B, L, w, s)
        rows = np.array([[b, t, h] for b in range(B) for t in (0, 5, L - 1) for h in range(Hq)])
        ro, _ = orc.prefill_rows(q, k, v, rows, w, s, threads=2, dtype="f16")
        assert np.abs(ro - ref[rows[:, 0], rows[:, 1], rows[:, 2]]).max() < 1e-12
        t = L - 1
        qt = np.ascontiguousarray(q[:, t])
        od = orc.decode(qt, k, v, [t] * B, w, s, threads=2, dtype="f16")
        assert np.abs(od - ref[:, t]).max() < 1e-12, ("decode", B, L, w, s)
        cap = L if w == W_INF else w
        ck = np.zeros((B, Hkv, cap, d), np.uint16)
        cv = np.zeros((B, Hkv, cap, d), np.uint16)
        orc.cache_append(ck, cv, k, v, 0, w, s)
        oc = orc.decode_cache(qt, ck, cv, [t] * B, w, s, threads=2, dtype="f16")
        assert np.abs(oc - ref[:, t]).max() < 1e-12, ("decode_cache", B, L, w, s)


def _hedgehog(x, W):
    """phi(x) = (exp(xW), exp(-xW)) for rows x [..., d], W [d, df] (numpy)."""
    f = x @ W
    return np.concatenate([np.exp(f), np.exp(-f)], axis=-1)


def _hybrid_dense(q, k, v, W, pos, w, s):
    """Hybrid decode by dense masks in numpy: softmax weights exp(c q.k) on
    A(t), linear weights phi(q).phi(k) on the earlier positions outside it,
    one normaliser."""
    qf, kf, vf = bits_to_f64(q), bits_to_f64(k), bits_to_f64(v)
    B, Hq, d = qf.shape
    Hkv = kf.shape[2]
    G = Hq // Hkv
    out = np.zeros_like(qf)
    for b in range(B):
        t = pos[b]
        inside = np.zeros(t + 1, bool)
        inside[_first_and_latest(t, w, s)] = True
        for h in range(Hq):
            kk, vv = kf[b, :t + 1, h // G], vf[b, :t + 1, h // G]
            sc = kk @ qf[b, h] / math.sqrt(d)
            m = sc[inside].max()
            wt = np.where(inside, np.exp(sc - m),
                          np.exp(-m) * (_hedgehog(kk, W[h // G]) @ _hedgehog(qf[b, h], W[h // G])))
            out[b, h] = wt @ vv / wt.sum()
    return out


def pin_hybrid_dense(orc) -> None:
    rng = np.random.default_rng(9)
    for B, P, Hq, Hkv, d, df, w, s in [(2, 40, 4, 2, 8, 4, 8, 2), (1, 33, 2, 1, 16, 8, 12, 0),
                                       (1, 25, 4, 4, 8, 2, 6, 5)]:
        q = _rand_bits(rng, (B, Hq, d))
        k = _rand_bits(rng, (B, P, Hkv, d))
        v = _rand_bits(rng, (B, P, Hkv, d))
        W = 0.2 * rng.standard_normal((Hkv, d, df))
        pos = [P - 1 - 3 * b for b in range(B)]
        got = orc.hybrid_decode(q, k, v, W, pos, w, s, threads=2)
        ref = _hybrid_dense(q, k, v, W, pos, w, s)
        assert np.abs(got - ref).max() < 1e-12, (B, P, w, s)


def pin_hybrid_special_cases(orc) -> None:
    rng = np.random.default_rng(10)
    B, P, Hq, Hkv, d, df, w, s = 2, 50, 4, 2, 8, 4, 10, 3
    q = _rand_bits(rng, (B, Hq, d))
    k = _rand_bits(rng, (B, P, Hkv, d))
    v = _rand_bits(rng, (B, P, Hkv, d))
    W = 0.3 * rng.standard_normal((Hkv, d, df))
    # nothing evicted yet (t < w): exactly the SWA decode
    for t in (0, 4, w - 1):
        a = orc.hybrid_decode(q, k, v, W, [t] * B, w, s, threads=1)
        b = orc.decode(q, k, v, [t] * B, w, s, threads=1)
        assert np.abs(a - b).max() < 1e-13, t
    # W = 0: phi = all ones, every linear weight is F = 2 df (closed form)
    t = P - 1
    o = orc.hybrid_decode(q, k, v, np.zeros_like(W), [t] * B, w, s, threads=1)
    qf, kf, vf = bits_to_f64(q), bits_to_f64(k), bits_to_f64(v)
    inside = _first_and_latest(t, w, s)
    outside = [i for i in range(t + 1) if i not in inside]
    for bb in range(B):
        for h in range(Hq):
            sc = kf[bb, inside, h // 2] @ qf[bb, h] / math.sqrt(d)
            e = np.exp(sc)
            num = e @ vf[bb, inside, h // 2] + 2 * df * vf[bb, outside, h // 2].sum(axis=0)
            den = e.sum() + 2 * df * len(outside)
            assert np.abs(o[bb, h] - num / den).max() < 1e-12, (bb, h)


def pin_hybrid_state(orc) -> None:
    """The state (S, z) after a prefix reproduces the decode's linear part:
    (window part + e^-m phi(q) S) / (... + e^-m phi(q).z) equals hybrid_decode."""
    rng = np.random.default_rng(11)
    B, P, Hq, Hkv, d, df, w, s = 2, 45, 4, 2, 8, 4, 9, 2
    q = _rand_bits(rng, (B, Hq, d))
    k = _rand_bits(rng, (B, P, Hkv, d))
    v = _rand_bits(rng, (B, P, Hkv, d))
    W = 0.25 * rng.standard_normal((Hkv, d, df))
    S, z = orc.hybrid_state(k, v, W, w, s, threads=2)
    t = P - 1
    ref = orc.hybrid_decode(q, k, v, W, [t] * B, w, s, threads=2)
    qf, kf, vf = bits_to_f64(q), bits_to_f64(k), bits_to_f64(v)
    inside = _first_and_latest(t, w, s)
    for bb in range(B):
        for h in range(Hq):
            g = h // 2
            sc = kf[bb, inside, g] @ qf[bb, h] / math.sqrt(d)
            m = sc.max()
            e = np.exp(sc - m)
            ph = _hedgehog(qf[bb, h], W[g])
            num = e @ vf[bb, inside, g] + np.exp(-m) * (ph @ S[bb, g])
            den = e.sum() + np.exp(-m) * (ph @ z[bb, g])
            assert np.abs(num / den - ref[bb, h]).max() < 1e-12, (bb, h)
    # infinite window: nothing is ever evicted
    S0, z0 = orc.hybrid_state(k, v, W, W_INF, 0, threads=1)
    assert not S0.any() and not z0.any()


ALL_PINS = [pin_golden_sets, pin_window_size, pin_brute_force, pin_causal_library,
            pin_closed_forms, pin_equal_values, pin_decode_history, pin_golden_cache,
            pin_ring_mapping, pin_decode_cache, pin_rows_match_full, pin_f16_every_pattern,
            pin_f16_brute_force, pin_hybrid_dense, pin_hybrid_special_cases, pin_hybrid_state]
