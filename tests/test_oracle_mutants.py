"""Plant plausible mistakes in a copy of the oracle; the pins must catch each one.

Every mutant is a textual edit of oracle/swa_oracle.c compiled to a temporary
library and checked in a child process (a planted mistake may write past a
buffer; the child keeps that away from the test process).  The real oracle is
never modified.
"""
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

MUTANTS = {
    # off-by-one in the start of the latest w-s tokens
    "window_one_too_wide": ("int64_t lo = t - (w - s) + 1;", "int64_t lo = t - (w - s);"),
    # sinks counted twice when they also fall inside the recent window
    "sink_double_count": ("if (lo < s) lo = s;", ""),
    # the 1/sqrt(d) scale dropped
    "no_scale": ("score[r] = dot * scale;", "score[r] = dot;"),
    # the wrong key/value head for a query head
    "gqa_modulo": ("int64_t kvh = h / G;", "int64_t kvh = h % Hkv;"),
    # keys and values transposed
    "k_v_swapped": ("return attend_list(qrow, kbase, vbase,", "return attend_list(qrow, vbase, kbase,"),
    # ring slot computed from p instead of p - s
    "ring_offset": ("return s + (p - s) % (w - s);", "return s + p % (w - s);"),
    # membership test with a strict bound
    "in_window_strict": ("return i >= t - (w - s) + 1;", "return i > t - (w - s) + 1;"),
    # the sinks dropped from the attended set
    "no_sinks": ("int64_t sink_end = s < t + 1 ? s : t + 1;", "int64_t sink_end = 0;"),
    # the query's own position left out (causal end exclusive)
    "exclusive_end": ("for (int64_t i = lo; i <= t; ++i) idx[n++] = i;",
                      "for (int64_t i = lo; i < t; ++i) idx[n++] = i;"),
    # fp16: exponent bias off by one
    "f16_bias": ("mag = ldexp((double)(1024 + f), e - 25);", "mag = ldexp((double)(1024 + f), e - 24);"),
    # fp16: subnormals read as if they had the implicit leading one
    "f16_subnormal": ("mag = ldexp((double)f, -24);", "mag = ldexp((double)(1024 + f), -24);"),
    # fp16 inputs widened as bf16
    "f16_as_bf16": ("if (dtype == ORACLE_F16) return f16_bits_to_double;",
                    "if (dtype == ORACLE_F16) return bf16_bits_to_double;"),
    # hybrid: the second half of the feature map with the wrong sign
    "phi_sign": ("out[df + j] = exp(-f);", "out[df + j] = exp(f);"),
    # hybrid: the linear part not brought to the softmax part's scale
    "linear_unscaled": ("const double em = exp(-m);", "const double em = 1.0;"),
    # hybrid: the last evicted position left out of the state
    "state_off_by_one": ("for (int64_t i = s; i <= last; ++i) {", "for (int64_t i = s; i < last; ++i) {"),
    # hybrid: W read transposed
    "w_transposed": ("f += widen(x[c]) * W[(int64_t)c * df + j];", "f += widen(x[c]) * W[(int64_t)j * d + c];"),
    # the log-sum-exp without the running max added back
    "lse_without_max": ("return m + log(den);", "return log(den);"),
    # decode over the cache: the newest filled slot left out
    "cache_decode_drops_newest": ("int64_t n = pos[b] + 1 < cap_eff ? pos[b] + 1 : cap_eff;",
                                  "int64_t n = pos[b] < cap_eff ? pos[b] : cap_eff;"),
    # decode over the cache: the wrong key/value head for a query head
    "cache_decode_gqa_modulo": ("kvh = h / G;\n        int64_t n = pos[b] + 1 < cap_eff",
                                "kvh = h % Hkv;\n        int64_t n = pos[b] + 1 < cap_eff"),
    # cache append: positions written last-first, so an earlier position that
    # shares a ring slot with a later one is what remains
    "append_reverse_order": ("for (int64_t j = 0; j < n; ++j) {", "for (int64_t j = n - 1; j >= 0; --j) {"),
}

CHILD = r"""
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, oracle_pins
orc = oracle.Oracle({lib!r})
caught = []
for pin in oracle_pins.ALL_PINS:
    try:
        pin(orc)
    except Exception:
        caught.append(pin.__name__)
print("CAUGHT", ",".join(caught), flush=True)
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path = os.path.join(tmp_path, "mutant.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.compile_source(path, os.path.join(tmp_path, "libmutant.so"))
    code = CHILD.format(root=ROOT, tests=HERE, lib=lib)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    lines = [l for l in r.stdout.splitlines() if l.startswith("CAUGHT")]
    if r.returncode != 0 and not lines:
        return  # the planted mistake crashed the oracle outright: caught
    caught = [c for c in lines[-1][len("CAUGHT"):].strip().split(",") if c]
    assert caught, f"no pin catches the mutant {name}"
