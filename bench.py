#!/usr/bin/env python3
"""Benchmark of the SWA(w,s) hot path on GB300.

The line measures the metric on the configurations it is quoted on
(Llama-3.1-8B attention shape: 32 query heads, 8 key/value heads, d = 128,
bf16, N(0,1) inputs, s = 4 sinks):
  decode  B=64, SWA(w,4) for w in {64, 512}: a cache filled by the bulk
          append of a 4096-token prompt, then 1024 steps that each append one
          token per sequence and decode it (one append_decode call);
  prefill B=2, L=32768, SWA(w,4) for w in {128, 256, 512}.
The decode stream runs through a stack of 16 attention layers, each with a
cache of its own, so that the caches a step reads (268 MB at w = 64, 2.1 GB
at w = 512) exceed the 129 MB L2 and every launch reads its cache from HBM.
One step is one pass over all of it: the three prefills, and for each decode
window the prompt's bulk append into every layer's cache and the 1024 decode
steps through the 16 layers.  Prefill and append launches are timed alone
with CUDA events on their stream, L2 flushed before each (256 MiB written,
then another 256 MiB read); each window's 1024 x 16 decode launches are one
CUDA graph, timed with one event pair around its replay (L2 also flushed
before it).  `value` is decoded tokens/s of one attention layer: the pass's
2 x 64 x 1024 x 16 layer-tokens over the device time of its decode graphs;
`prefill` holds the TFLOP/s, `decode` the KV-read GB/s, `rooflines` every
kernel against the measured peaks, `flatness` the 4-layer decode sweep over
1K..256K positions, `small_prefill` the 4096-token SWA(64,4) prefill.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl swa|reference]
Under torchrun each rank runs its own batch on its own GPU (no data exchange;
weak scaling) and rank 0 prints one JSON line.  `e2e` is the decode stream
through the public API with pinned host buffers, every step's h2d of its
inputs and d2h of its output inside the timed region.  `--impl reference`
times the fp64 CPU oracle on a bounded sample of the same decode workload on
the host cores.
"""
from __future__ import annotations

import argparse
import functools
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "SWA(w,4) decode tok/s + KV-read GB/s vs HBM peak; prefill TFLOP/s vs tensor peak"
# The configurations the metric is quoted on.
PREFILL_CFG = dict(B=2, L=32768, Hq=32, Hkv=8, d=128, s=4, windows=(128, 256, 512))
DECODE_CFG = dict(B=64, Hq=32, Hkv=8, d=128, s=4, windows=(64, 512), prompt=4096, steps=1024,
                  layers=16)
# The 4096-token prompt of one sequence, SWA(64,4), first 4 key rows x8.
SMALL_PREFILL = dict(B=1, L=4096, Hq=32, Hkv=8, d=128, w=64, s=4, sink_rows=4)
WORKLOAD_NAME = ("decode SWA(w,4) w in {64,512}: B=64 Hq=32 Hkv=8 d=128 bf16, cache filled from a "
                 "4096-token N(0,1) prompt, then 1024 steps each appending one N(0,1) token and "
                 "decoding it; prefill SWA(w,4) w in {128,256,512}: B=2 L=32768 Hq=32 Hkv=8 d=128 "
                 "bf16 N(0,1)")
L2_FLUSH_BYTES = 256 << 20
L2_NOTE = {
    "prefill_and_append": (f"flushed before every timed launch: {L2_FLUSH_BYTES >> 20} MiB written, "
                           f"then another {L2_FLUSH_BYTES >> 20} MiB read, so each launch starts on a "
                           f"cold L2 that holds no dirty lines of the flush"),
    "decode": ("inputs larger than L2: each launch reads the cache of one of 16 layers, and the "
               "15 launches since that cache was last read moved 15 other caches (252 MB at "
               "w = 64, 2 GB at w = 512) through the 129 MB L2; L2 also flushed before each "
               "replay of the graph"),
}
# Decode context sweep of the flatness key: 4 attention layers, positions
# 1K .. 256K, every finite window at batch 1 and 256; full causal at batch 1
# for contrast.
FLAT_POSITIONS = [1 << e for e in range(10, 19, 2)]
FLAT_WINDOWS = (64, 128, 256, 512)
FLAT_BATCHES = (1, 256)
FLAT_LAYERS = 4
FLAT_STEPS = 16
L2_BYTES = 129 * 10**6
CPU_DECODE_STEPS = 16
SMALL_SETS = 8   # prompts of the small-prefill graph (8 x 84 MB of inputs)
SMALL_REPS = 4   # passes over them per replay


class L2Flush:
    """Evicts the timed kernels' data from L2 (129 MB on GB300): write one
    buffer larger than L2, then read a second one, which also writes the
    first buffer's dirty lines back before the timed launch starts.  The read
    is a float32 sum, reduced as it is read (an integer sum would first copy
    the buffer to int64, leaving that copy's dirty lines in L2)."""

    def __init__(self, device="cuda"):
        import torch
        self.wbuf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.rbuf = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)

    def __call__(self, i: int = 1) -> None:
        self.wbuf.fill_(i & 0xFF)
        self.rbuf.sum()


# ----------------------------------------------------------------------------- arithmetic
def window_sum(L: int, w: int) -> int:
    """sum over t < L of |A(t)| = min(t+1, w) (w < 0: t+1)."""
    if w < 0 or w >= L:
        return L * (L + 1) // 2
    return w * (w + 1) // 2 + (L - w) * w


def prefill_flops(B, L, Hq, d, w) -> float:
    return 4.0 * d * Hq * B * window_sum(L, w)


def prefill_bytes(B, L, Hq, Hkv, d) -> float:
    return 2.0 * (2 * B * L * Hq * d + 2 * B * L * Hkv * d)


def decode_bytes(B, Hq, Hkv, d, n_valid) -> float:
    return B * (2 * Hq * d * 2 + 4 * Hkv * d * 2 + 2 * Hkv * d * 2 * n_valid)


def kv_read_bytes(B, Hkv, d, n_valid) -> float:
    """K and V bytes of the attended slots that one decode step reads."""
    return 2.0 * B * Hkv * d * 2 * n_valid


def decoded_tokens_per_step(world: int) -> int:
    """Layer-tokens all ranks decode in one step: each decode window's batch,
    every step, in every layer of the stack (one layer's tokens/s is then
    this over the decode time)."""
    C = DECODE_CFG
    return len(C["windows"]) * C["B"] * C["steps"] * C["layers"] * world


def peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return {"hbm_gbs": float(m["hbm_gbs"]), "bf16_tflops": float(m["bf16_tflops"]),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def roofline_entry(kernel: str, ms: float, flops: float, nbytes: float, pk: dict) -> dict:
    """The kernel against its bound: tensor if its intensity reaches the ridge
    of the two measured peaks, else HBM; achieved = algorithmic work per
    launch / the launch's mean CUDA-event time."""
    secs = ms * 1e-3
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    tflops, gbs = flops / secs / 1e12, nbytes / secs / 1e9
    if flops / nbytes >= ridge:
        e = {"bound": "tensor", "achieved": tflops, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
             "frac": tflops / pk["bf16_tflops"],
             "peak_source": pk["source"] + " bf16_tflops (burst: each launch is timed alone)"}
    else:
        e = {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
             "frac": gbs / pk["hbm_gbs"], "peak_source": pk["source"] + " hbm_gbs (copy)"}
    attainable = min(pk["bf16_tflops"], flops / nbytes * pk["hbm_gbs"] / 1e3)
    e.update({"kernel": kernel, "ms": ms, "algorithmic_flops_per_launch": flops,
              "algorithmic_bytes_per_launch": nbytes, "flop_per_byte": flops / nbytes,
              "tflops": tflops, "gbs": gbs, "frac_of_attainable": tflops / attainable,
              "attainable_tflops": attainable})
    return e


def kernel_traffic(source: str, workload: str):
    """DRAM bytes per launch from the committed ncu records (profiles/traffic.json)
    for this workload, if they were taken on the current kernel source (the
    file's sha256); else None."""
    src = os.path.join(ROOT, "sliding_window_attention_prefill_gb300", "csrc", source)
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            recs = json.load(f)["records"]
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()
        for rec in recs:
            if (rec.get("source") == source and rec.get("kernel_sha256") == h
                    and rec.get("workload") == workload):
                return float(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def prefill_workload(w: int) -> str:
    P = PREFILL_CFG
    return f"prefill SWA({w},4) B={P['B']} L={P['L']} Hq={P['Hq']} Hkv={P['Hkv']} d={P['d']} bf16"


def decode_workload(w: int) -> str:
    D = DECODE_CFG
    return (f"append_decode SWA({w},4) B={D['B']} Hq={D['Hq']} Hkv={D['Hkv']} d={D['d']} bf16, "
            f"positions {D['prompt']}..{D['prompt'] + D['steps'] - 1}")


SMALL_WORKLOAD = "prefill SWA(64,4) B=1 L=4096 Hq=32 Hkv=8 d=128 bf16, first 4 key rows x8"


# ----------------------------------------------------------------------------- ranks
def rank_seed(rank: int) -> int:
    """Each rank draws its own batch (weak scaling: independent sequences)."""
    return 1000 * rank


def max_over_ranks(values, device):
    """Element-wise max of per-rank timings (the slowest rank sets the pace)."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


def line_config(world: int) -> dict:
    """The `config` of both arms' lines (identical, so the two compare)."""
    P, D = PREFILL_CFG, DECODE_CFG
    return {"workload": WORKLOAD_NAME, "global_batch": D["B"] * world,
            "decode": {k: (list(v) if isinstance(v, tuple) else v) for k, v in D.items()},
            "prefill": {k: (list(v) if isinstance(v, tuple) else v) for k, v in P.items()},
            "seq_len": P["L"], "sinks": D["s"], "l2": L2_NOTE,
            "parallelism": f"replicas x{world} (independent batches)"}


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 50 ms for the whole run; summaries per named
    window of wall-clock time (start/stop marks)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.marks = {}
        self.rows = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(gpu_index)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.4)

    def start(self, name: str):
        self.marks[name] = [time.time(), None]

    def stop(self, name: str):
        self.marks[name][1] = time.time()

    def _collect(self):
        if self.rows is not None or self.proc is None:
            return
        time.sleep(0.15)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        self.rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                self.rows.append((ts, float(parts[2]), float(parts[3]), float(parts[4]), parts[6:10]))
            except Exception:
                continue

    def result(self, name: str) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self._collect()
        t0, t1 = self.marks[name]
        inside = [r for r in self.rows if t0 - 0.06 <= r[0] <= t1 + 0.06]
        used = inside if inside else self.rows
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in used:
            for n, v in zip(names, r[4]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median([r[1] for r in used]) if used else None,
                "sm_max_mhz": max(r[2] for r in used) if used else None,
                "power_w_max": max(r[3] for r in used) if used else None,
                "reasons": sorted(reasons), "samples": len(used), "seconds": t1 - t0,
                "window": "timed region" if inside else "around the timed region"}


# ----------------------------------------------------------------------------- oracle legs
def oracle_decode_state(kp, vp, w: int):
    """The oracle's cache after the prompt's bulk append (host bit patterns)."""
    import numpy as np

    import oracle
    D = DECODE_CFG
    orc = oracle.get()
    ck = np.zeros((D["B"], D["Hkv"], w, D["d"]), np.uint16)
    cv = np.zeros_like(ck)
    orc.cache_append(ck, cv, kp, vp, 0, w, D["s"])
    return ck, cv


def oracle_decode_steps(state, ks, vs, qs, w: int, n: int, threads=None) -> float:
    """Seconds the oracle takes for decode steps 0..n-1 of the stream (each:
    append the step's token, decode its query over the cache), on a copy of
    the post-prompt cache state."""
    import oracle
    D = DECODE_CFG
    orc = oracle.get()
    ck, cv = state[0].copy(), state[1].copy()
    t0 = time.perf_counter()
    for i in range(n):
        p = D["prompt"] + i
        orc.cache_append(ck, cv, ks[i], vs[i], p, w, D["s"])
        orc.decode_cache(qs[i], ck, cv, [p] * D["B"], w, D["s"], threads=threads)
    return time.perf_counter() - t0


def host_prompt(seed: int):
    """The decode workload's prompt as host bit patterns: k, v [B, 4096, Hkv, d]
    (CPU generator)."""
    import oracle
    from sliding_window_attention_prefill_gb300 import inputs
    D = DECODE_CFG
    g = inputs.generator(seed)
    kp = inputs.normal_bf16((D["B"], D["prompt"], D["Hkv"], D["d"]), g)
    vp = inputs.normal_bf16((D["B"], D["prompt"], D["Hkv"], D["d"]), g)
    return oracle.bits16(kp), oracle.bits16(vp)


def host_steps(n_steps: int, seed: int):
    """n_steps decode steps as host bit patterns: k, v [B, 1, Hkv, d] and
    q [B, Hq, d] per step (CPU generator)."""
    import oracle
    from sliding_window_attention_prefill_gb300 import inputs
    D = DECODE_CFG
    g = inputs.generator(seed)
    ks = inputs.normal_bf16((n_steps, D["B"], 1, D["Hkv"], D["d"]), g)
    vs = inputs.normal_bf16((n_steps, D["B"], 1, D["Hkv"], D["d"]), g)
    qs = inputs.normal_bf16((n_steps, D["B"], D["Hq"], D["d"]), g)
    b = oracle.bits16
    return [b(ks[i]) for i in range(n_steps)], [b(vs[i]) for i in range(n_steps)], \
        [b(qs[i]) for i in range(n_steps)]


def run_reference(args, rank: int):
    if rank != 0:
        return
    import oracle
    oracle.build()
    orc = oracle.get()
    cores = orc.threads(None)
    D = DECODE_CFG
    # size the sample (decode steps per window per bench step) to --ref-seconds
    calib = 2
    kp, vp = host_prompt(rank_seed(0))
    states = {w: oracle_decode_state(kp, vp, w) for w in D["windows"]}
    ks, vs, qs = host_steps(calib, rank_seed(0) + 1)
    t_step = sum(oracle_decode_steps(states[w], ks, vs, qs, w, calib) for w in D["windows"]) / calib
    budget = args.ref_seconds / max(1, args.steps + args.warmup)
    n = int(max(1, min(D["steps"], budget / max(t_step, 1e-9))))
    if n > calib:
        ks, vs, qs = host_steps(n, rank_seed(0) + 1)
    for _ in range(args.warmup):
        for w in D["windows"]:
            oracle_decode_steps(states[w], ks, vs, qs, w, n)
    times = []
    for _ in range(args.steps):
        times.append(sum(oracle_decode_steps(states[w], ks, vs, qs, w, n) for w in D["windows"]))
    mean = sum(times) / len(times)
    tokens = len(D["windows"]) * D["B"] * n
    value = tokens / mean
    sample = (f"decode steps 0..{n - 1} of the {D['steps']}-step stream in each window "
              f"(B={D['B']}, each step: the token's cache append + the decode of its query), "
              f"after the prompt's bulk append (untimed); no prefill")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": mean * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": line_config(1),
            "oracle": "fp64 C (gcc -O2, OpenMP over output rows)",
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline(kp, vp, ks, vs, qs, pre3) -> dict:
    """The oracle on bounded samples of the workload, all cores and one
    thread: the decode stream's first 16 steps per window (the headline
    unit), the 4096-token SWA(64,4) prompt in full, and 4096 sampled output
    rows (b, t, h) of the B=2 L=32768 prefill per window."""
    import numpy as np

    import oracle
    from sliding_window_attention_prefill_gb300 import inputs
    oracle.build()
    orc = oracle.get()
    D, P, S = DECODE_CFG, PREFILL_CFG, SMALL_PREFILL
    cores = orc.threads(None)
    n = CPU_DECODE_STEPS
    out = {"kind": "oracle", "unit": "tok/s", "cores": cores, "nproc": os.cpu_count()}
    dec = {}
    for th, key, nn in ((None, "all_cores", n), (1, "one_thread", max(1, n // 4))):
        secs = 0.0
        for w in D["windows"]:
            st = oracle_decode_state(kp, vp, w)
            t = oracle_decode_steps(st, ks, vs, qs, w, nn, threads=th)
            dec[f"w{w}_{key}_ms_per_step"] = t / nn * 1e3
            secs += t
        dec[key] = len(D["windows"]) * D["B"] * nn / secs
        dec[f"{key}_steps_per_window"] = nn
    out["value"] = dec["all_cores"]
    out["one_thread"] = dec["one_thread"]
    out["decode"] = dec
    out["sample"] = (f"decode: steps 0..{n - 1} of the 1024-step stream in each window "
                     f"(B={D['B']}; append + decode per step), value over all {cores} threads; "
                     f"one thread over steps 0..{max(1, n // 4) - 1}")
    # the 4096-token prompt, in full
    q, k, v = inputs.prefill_inputs(S["B"], S["L"], S["Hq"], S["Hkv"], S["d"], seed=0,
                                    sink_rows=S["sink_rows"])
    small = {}
    for th, key in ((None, "all_cores"), (1, "one_thread")):
        t0 = time.perf_counter()
        orc.prefill(q, k, v, S["w"], S["s"], threads=th)
        small[f"{key}_s"] = time.perf_counter() - t0
        small[f"{key}_tok_s"] = S["B"] * S["L"] / small[f"{key}_s"]
    out["small_prefill_full"] = small
    # the L=32768 prefill: 4096 sampled rows per window
    q3, k3, v3 = pre3
    rows_total = P["B"] * P["L"] * P["Hq"]
    nr = 4096
    idx = np.linspace(0, rows_total - 1, nr).astype(np.int64)
    rows = np.stack([idx // (P["L"] * P["Hq"]), (idx // P["Hq"]) % P["L"], idx % P["Hq"]], 1)
    big = {"rows_sampled": nr, "row": "one (b, t, h) output row of d values"}
    for w in P["windows"]:
        for th, key in ((None, "all_cores"), (1, "one_thread")):
            t0 = time.perf_counter()
            orc.prefill_rows(q3, k3, v3, rows, w, P["s"], threads=th)
            dt = time.perf_counter() - t0
            big[f"w{w}_{key}_rows_s"] = nr / dt
            big[f"w{w}_{key}_full_s_extrapolated"] = rows_total / (nr / dt)
    out["prefill_L32768_sample"] = big
    return out


# ----------------------------------------------------------------------------- GPU arm
def run_swa(args, rank: int, world: int, local_rank: int):
    import torch

    import sliding_window_attention_prefill_gb300 as swa
    from sliding_window_attention_prefill_gb300 import build, inputs
    build.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    P, D, S = PREFILL_CFG, DECODE_CFG, SMALL_PREFILL
    pk = peaks()
    gen = inputs.device_generator(rank_seed(rank) + 7, dev)
    # prefill inputs (B=2, L=32768)
    q3 = inputs.normal16_on((P["B"], P["L"], P["Hq"], P["d"]), gen)
    k3 = inputs.normal16_on((P["B"], P["L"], P["Hkv"], P["d"]), gen)
    v3 = inputs.normal16_on((P["B"], P["L"], P["Hkv"], P["d"]), gen)
    o3 = torch.empty_like(q3)
    # decode inputs: the prompt and the 1024 steps
    B, Hq, Hkv, d, s = D["B"], D["Hq"], D["Hkv"], D["d"], D["s"]
    prompt, nsteps = D["prompt"], D["steps"]
    kp = inputs.normal16_on((B, prompt, Hkv, d), gen)
    vp = inputs.normal16_on((B, prompt, Hkv, d), gen)
    ks = inputs.normal16_on((nsteps, B, 1, Hkv, d), gen)
    vs = inputs.normal16_on((nsteps, B, 1, Hkv, d), gen)
    qs = inputs.normal16_on((nsteps, B, Hq, d), gen)
    pos = (prompt + torch.arange(nsteps, dtype=torch.int32, device=dev))[:, None]
    pos = pos.expand(nsteps, B).contiguous()
    nlay = D["layers"]
    caches = {w: [swa.Cache(B, Hkv, d, w, s, device=dev) for _ in range(nlay)] for w in D["windows"]}
    wsp = {w: swa.workspace_for(caches[w][0], Hq) for w in D["windows"]}
    od = {w: torch.empty(B, Hq, d, dtype=torch.bfloat16, device=dev) for w in D["windows"]}
    flush = L2Flush(dev)
    # Layer l of step i takes the inputs drawn for step (i + l * stride) mod
    # 1024: different in every layer of a step.
    stride = nsteps // nlay

    def layer_inputs(i, l):
        j = (i + l * stride) % nsteps
        return qs[j], ks[j], vs[j]

    def reset_caches(w):
        for c in caches[w]:
            c.append(kp, vp, 0)

    def decode_stream(w):
        for i in range(nsteps):
            for l in range(nlay):
                q_, k_, v_ = layer_inputs(i, l)
                swa.append_decode(q_, k_, v_, caches[w][l], pos[i], out=od[w], workspace=wsp[w])

    # Each window's 1024 x 16 decode launches as one CUDA graph (one call
    # warmed up outside the capture; the step's appends reset the caches).
    cap = torch.cuda.Stream(dev)
    dgraphs = {}
    for w in D["windows"]:
        reset_caches(w)
        q_, k_, v_ = layer_inputs(0, 0)
        swa.append_decode(q_, k_, v_, caches[w][0], pos[0], out=od[w], workspace=wsp[w])
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        cap.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                decode_stream(w)
        torch.cuda.current_stream(dev).wait_stream(cap)
        torch.cuda.synchronize()
        dgraphs[w] = g

    # the timed units of one step, in order: (kind, window, call, kernels it launches)
    units = []
    for w in P["windows"]:
        units.append(("prefill", w, functools.partial(swa.prefill, q3, k3, v3, w, P["s"], out=o3), 1))
    for w in D["windows"]:
        for c in caches[w]:
            units.append(("append", w, functools.partial(c.append, kp, vp, 0), 1))
        nl = 1 + (1 if wsp[w] is not None else 0)
        units.append(("decode", w, dgraphs[w].replay, nsteps * nlay * nl))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in units]

    def run_step():
        # The GPU idles while the host reads the previous step's events; the
        # first launch after that idle ran up to 30 % slower, so the step's
        # first unit runs once untimed before the timed pass.
        flush(len(units))
        units[0][2]()
        for j, u in enumerate(units):
            flush(j)
            ev[j][0].record()
            u[2]()
            ev[j][1].record()

    for _ in range(args.warmup):
        run_step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.start("step")
    per_step = []  # [step][unit] ms
    for _ in range(args.steps):  # the timed steps (an NVTX range each, for a profiler's filter)
        rid = torch.cuda.nvtx.range_start("bench timed step")
        run_step()
        torch.cuda.nvtx.range_end(rid)
        torch.cuda.synchronize()
        per_step.append([a.elapsed_time(b) for a, b in ev])
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    if sampler:
        sampler.stop("step")

    def mean_of(kind, w):
        js = [j for j, u in enumerate(units) if u[0] == kind and u[1] == w]
        return sum(t[j] for t in per_step for j in js) / (len(per_step) * len(js))

    # The cost of the measurement itself: an event pair with nothing between
    # it, after a flush, timed the same way (reported beside the results;
    # every launch timed alone still includes it, a decode graph once).
    eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(200)]
    for i, (a, b_) in enumerate(eev):
        flush(i)
        a.record()
        b_.record()
    torch.cuda.synchronize()
    event_pair_ms = sum(a.elapsed_time(b_) for a, b_ in eev) / len(eev)

    step_ms = sum(sum(t) for t in per_step) / len(per_step)
    dec_ms = sum(sum(t[j] for j, u in enumerate(units) if u[0] == "decode")
                 for t in per_step) / len(per_step)
    pre_ms = {w: mean_of("prefill", w) for w in P["windows"]}
    app_ms = {w: mean_of("append", w) for w in D["windows"]}  # one layer's prompt append
    graph_ms = {w: mean_of("decode", w) for w in D["windows"]}  # the window's decode graph
    tok_ms = {w: graph_ms[w] / (nsteps * nlay) for w in D["windows"]}  # per launch

    # ---- the 4096-token SWA(64,4) prefill (one sequence).  A launch of
    # about 20 µs is too short for the GPU's event timer (2.048 µs steps,
    # about 5 µs around an isolated launch), so the prompts of SMALL_SETS
    # sequences (84 MB of Q, K and V each, 8 x that together: more than four
    # times L2) are prefilled one after another in one CUDA graph, each
    # launch reading its own cold inputs; events around each replay, L2
    # flushed before it.  The launch timed alone is reported beside it.
    small_sets = []
    for j in range(SMALL_SETS):
        sq, sk, sv = inputs.prefill_inputs(S["B"], S["L"], S["Hq"], S["Hkv"], S["d"],
                                           seed=rank_seed(rank) + j, sink_rows=S["sink_rows"])
        sq, sk, sv = sq.to(dev), sk.to(dev), sv.to(dev)
        small_sets.append((sq, sk, sv, torch.empty_like(sq)))

    def small_pass():
        for _ in range(SMALL_REPS):
            for sq, sk, sv, so in small_sets:
                swa.prefill(sq, sk, sv, S["w"], S["s"], out=so)

    n_small = max(20, args.steps)
    if sampler:
        sampler.start("small")
    small_ms = _time_graph(small_pass, n_small, flush, stat="trimmed") / (SMALL_SETS * SMALL_REPS)
    if sampler:
        sampler.stop("small")
    sq, sk, sv, so = small_sets[0]
    sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n_small)]
    for i in range(n_small):
        flush(i)
        sev[i][0].record()
        swa.prefill(sq, sk, sv, S["w"], S["s"], out=so)
        sev[i][1].record()
    torch.cuda.synchronize()
    small_alone_ms = sum(a.elapsed_time(b) for a, b in sev) / n_small

    # ---- end to end: the decode stream through the public API with host
    # buffers.  Each step's inputs (q, k, v packed in one pinned host row)
    # go up, append_decode runs in each of the 16 layers (every layer takes
    # the step's q, k, v), the last layer's output comes back; consecutive steps
    # overlap (step i+1's copy up while step i computes and step i-1's output
    # comes down: double-buffered device buffers).  Every copy is inside the
    # timed region.
    nq, nkv = B * Hq * d, B * Hkv * d
    host_in = torch.empty(nsteps, nq + 2 * nkv, dtype=torch.bfloat16, pin_memory=True)
    host_in[:, :nq] = qs.reshape(nsteps, nq).cpu()
    host_in[:, nq:nq + nkv] = ks.reshape(nsteps, nkv).cpu()
    host_in[:, nq + nkv:] = vs.reshape(nsteps, nkv).cpu()
    host_out = torch.empty(nsteps, B, Hq, d, dtype=torch.bfloat16, pin_memory=True)
    dev_in = [torch.empty(nq + 2 * nkv, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    views = [(b[:nq].view(B, Hq, d), b[nq:nq + nkv].view(B, 1, Hkv, d), b[nq + nkv:].view(B, 1, Hkv, d))
             for b in dev_in]
    dev_out = [torch.empty(B, Hq, d, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    up, down, comp = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.current_stream(dev)

    def enqueue_stream(w, comp):
        """Enqueue the window's 1024 steps (copy up, append_decode in every
        layer, copy down) on comp and the two copy streams, forked from and
        joined back to comp."""
        up.wait_stream(comp)
        down.wait_stream(comp)
        done = []
        for i in range(nsteps):
            j = i & 1
            if i >= 2:  # dev_in[j] was read by step i-2's kernel
                up.wait_event(done[i - 2][0])
            with torch.cuda.stream(up):
                dev_in[j].copy_(host_in[i], non_blocking=True)
            e_up = torch.cuda.Event()
            e_up.record(up)
            comp.wait_event(e_up)
            if i >= 2:  # dev_out[j] was read back by step i-2's copy
                comp.wait_event(done[i - 2][1])
            qv, kv, vv = views[j]
            for c in caches[w]:
                swa.append_decode(qv, kv, vv, c, pos[i], out=dev_out[j], workspace=wsp[w])
            e_comp = torch.cuda.Event()
            e_comp.record(comp)
            down.wait_event(e_comp)
            with torch.cuda.stream(down):
                host_out[i].copy_(dev_out[j], non_blocking=True)
            e_down = torch.cuda.Event()
            e_down.record(down)
            done.append((e_comp, e_down))
        comp.wait_stream(up)
        comp.wait_stream(down)

    def e2e_eager(w):
        reset_caches(w)  # back to the post-prompt state (device inputs; untimed)
        torch.cuda.synchronize()
        comp = torch.cuda.current_stream(dev)
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(comp)
        enqueue_stream(w, comp)
        b_.record(comp)
        b_.synchronize()
        return a.elapsed_time(b_)

    # The same stream captured once as a CUDA graph per window (the calls are
    # graph-replayable: positions and buffers live on the device) and
    # replayed: the host's per-call overhead leaves the loop, every step's
    # copies stay in it.
    cap = torch.cuda.Stream(dev)
    graphs = {}
    for w in D["windows"]:
        enqueue_stream(w, torch.cuda.current_stream(dev))  # warm-up outside capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        cap.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap):
                enqueue_stream(w, cap)
        torch.cuda.current_stream(dev).wait_stream(cap)
        torch.cuda.synchronize()
        graphs[w] = g

    def e2e_graph(w):
        reset_caches(w)  # back to the post-prompt state (device inputs; untimed)
        torch.cuda.synchronize()
        comp = torch.cuda.current_stream(dev)
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(comp)
        graphs[w].replay()
        b_.record(comp)
        b_.synchronize()
        return a.elapsed_time(b_)

    for w in D["windows"]:  # warm-up
        e2e_graph(w)
    if sampler:
        sampler.start("e2e")
    # each window's stream replayed three times; the median replay counts
    # (one replay is a single sample of the host link's state)
    e2e_ms = sum(sorted(e2e_graph(w) for _ in range(3))[1] for w in D["windows"])
    if sampler:
        sampler.stop("e2e")
    e2e_eager_ms = sum(e2e_eager(w) for w in D["windows"])
    del graphs
    h2d = len(D["windows"]) * nsteps * (nq + 2 * nkv) * 2
    d2h = len(D["windows"]) * nsteps * nq * 2

    # ---- flatness: the decode context sweep
    flat = flatness_sweep(dev, flush, sampler)

    vals = [step_ms, dec_ms, small_ms, e2e_ms, event_pair_ms, e2e_eager_ms, small_alone_ms] + \
        [pre_ms[w] for w in P["windows"]] + \
        [app_ms[w] for w in D["windows"]] + [tok_ms[w] for w in D["windows"]]
    if world > 1:
        vals = max_over_ranks(vals, dev)
    step_ms, dec_ms, small_ms, e2e_ms, event_pair_ms, e2e_eager_ms, small_alone_ms = vals[:7]
    rest = vals[7:]
    pre_ms = dict(zip(P["windows"], rest[:len(P["windows"])]))
    rest = rest[len(P["windows"]):]
    app_ms = dict(zip(D["windows"], rest[:len(D["windows"])]))
    tok_ms = dict(zip(D["windows"], rest[len(D["windows"]):]))
    if rank != 0:
        return

    tokens = decoded_tokens_per_step(world)
    value = tokens / (dec_ms * 1e-3)
    rl, shares = {}, {}
    prefill_key = {}
    for w in P["windows"]:
        fl = prefill_flops(P["B"], P["L"], P["Hq"], P["d"], w)
        by = prefill_bytes(P["B"], P["L"], P["Hq"], P["Hkv"], P["d"])
        e = roofline_entry("swa_prefill_kernel", pre_ms[w], fl, by, pk)
        e["traffic"] = kernel_traffic("swa_prefill.cu", prefill_workload(w))
        e["workload"] = prefill_workload(w)
        rl[f"prefill_w{w}"] = e
        shares[f"prefill_w{w}"] = pre_ms[w] / step_ms
        prefill_key[f"w{w}"] = {"ms": pre_ms[w], "tflops": e["tflops"],
                                "frac_tensor_peak": e["tflops"] / pk["bf16_tflops"],
                                "frac_attainable": e["frac_of_attainable"],
                                "attainable_tflops": e["attainable_tflops"], "gbs": e["gbs"],
                                "algorithmic_gflop": fl / 1e9}
    decode_key = {}
    for w in D["windows"]:
        nv = min(prompt + 1, w)
        by = decode_bytes(B, Hq, Hkv, d, nv)
        kv = kv_read_bytes(B, Hkv, d, nv)
        e = roofline_entry("swa_decode_kernel (append_decode)", tok_ms[w], 4.0 * d * Hq * B * nv, by, pk)
        e["traffic"] = kernel_traffic("swa_decode.cu", decode_workload(w))
        e["workload"] = decode_workload(w)
        rl[f"decode_w{w}"] = e
        shares[f"decode_w{w}"] = tok_ms[w] * nsteps * nlay / step_ms
        shares[f"append_w{w}"] = app_ms[w] * nlay / step_ms
        decode_key[f"w{w}"] = {"ms_step": tok_ms[w], "tok_s": B * world / (tok_ms[w] * 1e-3),
                               "kv_read_gbs": kv / (tok_ms[w] * 1e-3) / 1e9,
                               "frac_hbm": e["frac"], "bytes_per_step": by,
                               "kv_bytes_per_step": kv, "cache_bytes": 2 * B * Hkv * w * d * 2,
                               "prompt_append_ms": app_ms[w], "layers": nlay,
                               "graph_ms": tok_ms[w] * nsteps * nlay}
    dom = max((k for k in rl), key=lambda k: shares[k])
    roof = {k: rl[dom][k] for k in ("bound", "achieved", "peak", "unit", "frac")}
    roof.update({"traffic": rl[dom]["traffic"], "kernel": rl[dom]["kernel"], "which": dom,
                 "workload": rl[dom]["workload"],
                 "share_of_step": shares[dom],
                 "algorithmic_bytes_per_launch": rl[dom]["algorithmic_bytes_per_launch"],
                 "peak_source": rl[dom]["peak_source"]})
    sb = prefill_bytes(S["B"], S["L"], S["Hq"], S["Hkv"], S["d"])
    sf = prefill_flops(S["B"], S["L"], S["Hq"], S["d"], S["w"])
    small_rl = roofline_entry("swa_prefill_kernel", small_ms, sf, sb, pk)
    small_rl["traffic"] = kernel_traffic("swa_prefill.cu", SMALL_WORKLOAD)
    launches = (sum(u[3] for u in units) + units[0][3]) * args.steps  # with the untimed first unit
    line = {
        "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": line_config(world),
        "timing": ("prefill and append launches timed alone: CUDA events on their stream "
                   "around each, L2 flushed before it; each decode window's 1024 steps x 16 "
                   "layers as one CUDA graph, events around its replay (L2 flushed before "
                   "it); ms_per_step = the sum of those times; value = decoded_tokens_per_step "
                   "(layer-tokens) / ms_decode_per_step"),
        "decoded_tokens_per_step": tokens, "ms_decode_per_step": dec_ms,
        "event_pair_us": event_pair_ms * 1e3,
        "gpu_launches": launches,
        "roofline": roof,
        "decode": decode_key,
        "prefill": prefill_key,
        "rooflines": rl,
        "time_shares": shares,
        "small_prefill": {"workload": SMALL_WORKLOAD, "ms": small_ms, "roofline": small_rl,
                          "timing": (f"{SMALL_SETS} prompts prefilled one after another, {SMALL_REPS} "
                                     "times, in one CUDA graph (each launch on its own cold inputs); "
                                     "events around each replay, L2 flushed before it; ms per launch"),
                          "ms_launch_alone": small_alone_ms,
                          "tok_s": S["B"] * S["L"] / (small_ms * 1e-3),
                          "clocks": sampler.result("small") if sampler else None},
        "flatness": flat,
        "e2e": {"value": tokens / (e2e_ms * 1e-3), "unit": "tok/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "timing": "the 1024-step decode stream of each window through the Python API "
                          "(append_decode in each of the 16 layers), captured once as a CUDA "
                          "graph and replayed: every step's q, k, v copied up from pinned host "
                          "memory once (all layers take them) and the last layer's output "
                          "copied back, steps overlapped (double-buffered device buffers, "
                          "copies on two streams of their own), events around the replay; "
                          "the median of three replays per window",
                "eager": {"value": tokens / (e2e_eager_ms * 1e-3), "ms_per_step": e2e_eager_ms,
                          "timing": "the same stream issued call by call from Python"},
                "clocks": sampler.result("e2e") if sampler else None},
        "clocks": sampler.result("step") if sampler else None,
    }
    if world == 1:
        from oracle import bits16
        line["cpu_baseline"] = cpu_baseline(
            bits16(kp), bits16(vp), [bits16(ks[i]) for i in range(CPU_DECODE_STEPS)],
            [bits16(vs[i]) for i in range(CPU_DECODE_STEPS)],
            [bits16(qs[i]) for i in range(CPU_DECODE_STEPS)], (bits16(q3), bits16(k3), bits16(v3)))
    print(json.dumps(line), flush=True)


def flatness_sweep(dev, flush, sampler) -> dict:
    """Decode tok/s of a 4-layer attention-only stack at positions 1K .. 256K
    (every layer's cache in the state a prompt of that length leaves, N(0,1)
    values; one step appends the token and decodes it in each layer).  Each
    point is one CUDA graph of FLAT_STEPS steps, L2 flushed before each
    replay: a single step is too short for the GPU's event timer, which moves
    in 2.048 µs steps.  Every step of a replay reads caches that are cold in
    L2: when a stack's caches are smaller than four times L2, the steps go
    through FLAT_STEPS copies of the stack, one each; larger stacks do not
    fit in L2 from one step to the next.  The trimmed mean of the replays, per step.
    Reports tok/s per point and max/min over the positions for each finite
    window at batch 1 and 256; full causal at batch 1 for contrast."""
    import torch

    import sliding_window_attention_prefill_gb300 as swa
    D = DECODE_CFG
    Hq, Hkv, d, s = D["Hq"], D["Hkv"], D["d"], D["s"]
    gen = torch.Generator(device=dev)
    reps = 12
    out = {"positions": FLAT_POSITIONS, "layers": FLAT_LAYERS, "steps_per_replay": FLAT_STEPS,
           "replays_per_point": reps,
           "statistic": "mean of the replays without the fastest and slowest, per step"}
    if sampler:
        sampler.start("flatness")
    pts = [(B, w) for B in FLAT_BATCHES for w in FLAT_WINDOWS] + [(1, -1)]
    for B, w in pts:
        toks, copies = [], []
        for P in FLAT_POSITIONS:
            gen.manual_seed(B * 1000003 + P * 7 + (w + 1))
            cap = P + 1 if w < 0 else w
            stack_bytes = FLAT_LAYERS * 2 * B * Hkv * cap * d * 2
            n_copies = FLAT_STEPS if stack_bytes < 4 * L2_BYTES else 1
            stacks = []
            for _ in range(n_copies):
                layers = []
                for _ in range(FLAT_LAYERS):
                    c = swa.Cache(B, Hkv, d, w, s if w > 0 else 0, max_len=(P + 1 if w < 0 else None),
                                  device=dev)
                    c.k.normal_(generator=gen)
                    c.v.normal_(generator=gen)
                    kn = torch.randn(B, 1, Hkv, d, generator=gen, device=dev).to(torch.bfloat16)
                    vn = torch.randn(B, 1, Hkv, d, generator=gen, device=dev).to(torch.bfloat16)
                    q = torch.randn(B, Hq, d, generator=gen, device=dev).to(torch.bfloat16)
                    layers.append((c, kn, vn, q, torch.empty_like(q), swa.workspace_for(c, Hq)))
                stacks.append(layers)
            pos = torch.full((B,), P, dtype=torch.int32, device=dev)

            def steps():
                for i in range(FLAT_STEPS):
                    for c, kn, vn, q, o, ws in stacks[i % n_copies]:
                        swa.append_decode(q, kn, vn, c, pos, out=o, workspace=ws)

            ms = _time_graph(steps, reps, flush, stat="trimmed") / FLAT_STEPS
            toks.append(B / (ms * 1e-3))
            copies.append(n_copies)
            del stacks, steps
            torch.cuda.empty_cache()
        key = f"B{B}_w{w}" if w > 0 else f"B{B}_full_causal"
        out[key] = {"tok_s": toks, "max_over_min": max(toks) / min(toks), "stack_copies": copies}
    finite = [out[f"B{B}_w{w}"]["max_over_min"] for B in FLAT_BATCHES for w in FLAT_WINDOWS]
    out["worst_max_over_min_finite_w"] = max(finite)
    if sampler:
        sampler.stop("flatness")
        out["clocks"] = sampler.result("flatness")
    return out


def _time_graph(fn, steps: int, flush, warm: int = 3, stat: str = "mean") -> float:
    """Mean (or median, or trimmed mean) ms of `fn` replayed as a CUDA graph,
    L2 flushed before each replay."""
    import torch
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(warm):
        flush(1)
        g.replay()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for i in range(steps):
        flush(i)
        evs[i][0].record()
        g.replay()
        evs[i][1].record()
    torch.cuda.synchronize()
    t = [a.elapsed_time(b) for a, b in evs]
    if stat == "median":
        return sorted(t)[len(t) // 2]
    if stat == "trimmed" and steps > 2:  # without the fastest and the slowest replay
        return sum(sorted(t)[1:-1]) / (steps - 2)
    return sum(t) / steps


def suite_prefill(steps: int, only_w=None, B_=None, L_=None):
    """Prefill kernel alone on the prefill configs: B=1 L=4096 SWA(64,4) and
    B=2 L=32768 SWA(w,4) for w in {128, 256, 512} (Hq=32, Hkv=8, d=128, bf16).
    Also full causal attention (w = infinity) at B=1, L=16384; SWA(512,4) in
    fp16; and the pages' system-test attention shape (16 heads of 64, fp16,
    batch 1) at L=32768 for SWA(64,4), SWA(512,4) and full causal.
    only_w / B_ / L_ restrict or resize the list (smaller cases for ncu)."""
    import torch

    import sliding_window_attention_prefill_gb300 as swa
    from sliding_window_attention_prefill_gb300 import build, inputs
    build.build()
    pk = peaks()
    flush = L2Flush()
    llama, paper = (32, 8, 128), (16, 16, 64)
    cases = [(1, 4096, 64, 4, llama, "bf16"), (2, 32768, 128, 0, llama, "bf16"),
             (2, 32768, 256, 0, llama, "bf16"), (2, 32768, 512, 0, llama, "bf16"),
             (1, 16384, -1, 0, llama, "bf16"), (2, 32768, 512, 0, llama, "f16"),
             (1, 32768, 64, 4, paper, "f16"), (1, 32768, 512, 0, paper, "f16"),
             (1, 32768, -1, 0, paper, "f16")]
    if only_w is not None:
        cases = [c for c in cases if c[2] == only_w]
    cases = [(B_ or c[0], L_ or c[1]) + c[2:] for c in cases]
    for B, L, w, sink_rows, (Hq, Hkv, d), dts in cases:
        s = 4
        dt = torch.float16 if dts == "f16" else torch.bfloat16
        q, k, v = inputs.prefill_inputs(B, L, Hq, Hkv, d, seed=0, sink_rows=sink_rows, dtype=dt)
        q, k, v = q.cuda(), k.cuda(), v.cuda()
        o = torch.empty_like(q)
        ms = _time_graph(lambda: swa.prefill(q, k, v, w, s, out=o), steps, flush)
        fl, by = prefill_flops(B, L, Hq, d, w), prefill_bytes(B, L, Hq, Hkv, d)
        tf = fl / (ms * 1e-3) / 1e12
        attainable = min(pk["bf16_tflops"], fl / by * pk["hbm_gbs"] / 1e3)
        print(json.dumps({"suite": "prefill", "dtype": dts, "Hq": Hq, "Hkv": Hkv, "d": d,
                          "B": B, "L": L, "w": w if w > 0 else "inf",
                          "s": s if w > 0 else 0, "ms": ms,
                          "tflops": tf, "frac_tensor_peak": tf / pk["bf16_tflops"],
                          "frac_attainable": tf / attainable, "attainable_tflops": attainable,
                          "gbs": by / (ms * 1e-3) / 1e9, "flop_per_byte": fl / by}), flush=True)
        del q, k, v, o
        torch.cuda.empty_cache()


def suite_decode(steps: int, only_w=None, n_steps: int = 1024, B_=None):
    """Decode configuration: B=64 (or B_), Hq=32, Hkv=8, d=128, SWA(w,4) for w
    in {64, 512}; the cache is filled from a 4096-token N(0,1) prompt, then
    `n_steps` decode steps each append one N(0,1) token and decode it (one
    append_decode call).  Every step is its own captured CUDA graph; L2 is
    flushed before each step.  Also times the decode kernel alone."""
    import torch

    import sliding_window_attention_prefill_gb300 as swa
    from sliding_window_attention_prefill_gb300 import build, inputs
    build.build()
    pk = peaks()
    flush = L2Flush()
    B, Hq, Hkv, d, s, prompt = B_ or 64, 32, 8, 128, 4, 4096
    for w in [x for x in (64, 512) if only_w is None or x == only_w]:
        gen = inputs.device_generator(0)
        kp = inputs.normal16_on((B, prompt, Hkv, d), gen)
        vp = inputs.normal16_on((B, prompt, Hkv, d), gen)
        ks = inputs.normal16_on((n_steps, B, 1, Hkv, d), gen)
        vs = inputs.normal16_on((n_steps, B, 1, Hkv, d), gen)
        qs = inputs.normal16_on((n_steps, B, Hq, d), gen)
        c = swa.Cache(B, Hkv, d, w, s)
        c.append(kp, vp, 0)
        del kp, vp
        pos = (prompt + torch.arange(n_steps, dtype=torch.int32, device="cuda"))[:, None]
        pos = pos.expand(n_steps, B).contiguous()
        od = torch.empty_like(qs[0])
        ws = swa.workspace_for(c, Hq)

        def step(i):
            swa.append_decode(qs[i], ks[i], vs[i], c, pos[i], out=od, workspace=ws)

        step(0)  # kernel attributes are set outside capture
        torch.cuda.synchronize()
        cs = torch.cuda.Stream()
        cs.wait_stream(torch.cuda.current_stream())
        graphs = []
        with torch.cuda.stream(cs):
            for i in range(n_steps):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=cs):
                    step(i)
                graphs.append(g)
        torch.cuda.current_stream().wait_stream(cs)
        torch.cuda.synchronize()
        # step 0 ran once above; its graph re-appends the same token (idempotent)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(n_steps)]
        for i, g in enumerate(graphs):
            flush(i)
            evs[i][0].record()
            g.replay()
            evs[i][1].record()
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in evs) / n_steps
        last = n_steps - 1
        ms_dec = _time_graph(lambda: swa.decode(qs[last], c, pos[last], out=od, workspace=ws),
                             steps, flush)
        n_valid = min(prompt + n_steps, w)
        by = decode_bytes(B, Hq, Hkv, d, n_valid)
        kv = 2 * B * Hkv * d * 2 * n_valid
        print(json.dumps({"suite": "decode", "B": B, "w": w, "s": s, "prompt": prompt,
                          "decode_steps": n_steps, "ms_step": ms, "tok_s": B / (ms * 1e-3),
                          "ms_decode": ms_dec, "kv_read_gbs": kv / (ms_dec * 1e-3) / 1e9,
                          "frac_hbm": by / (ms_dec * 1e-3) / 1e9 / pk["hbm_gbs"],
                          "bytes_decode": by, "l2": L2_NOTE}), flush=True)
        del graphs, c, ks, vs, qs
        torch.cuda.empty_cache()


def suite_chunk(steps: int):
    """Chunked prefill from a cache (prefill_chunk) against one prefill of the
    whole prompt, Llama attention shape (Hq=32, Hkv=8, d=128): SWA(64,4)
    B=1 L=4096 in chunks of 512, SWA(512,4) B=2 L=32768 in chunks of 4096,
    and full causal B=1 L=16384 in chunks of 4096.  A step is the whole
    prompt (all chunks, each gathering, attending and appending); L2 is
    flushed before each step."""
    import torch

    import sliding_window_attention_prefill_gb300 as swa
    from sliding_window_attention_prefill_gb300 import build, inputs
    build.build()
    pk = peaks()
    flush = L2Flush()
    Hq, Hkv, d = 32, 8, 128
    for B, L, w, s, n in [(1, 4096, 64, 4, 512), (2, 32768, 512, 4, 4096), (1, 16384, -1, 0, 4096)]:
        q, k, v = inputs.prefill_inputs(B, L, Hq, Hkv, d, seed=0)
        q, k, v = q.cuda(), k.cuda(), v.cuda()
        qc = [q[:, i:i + n].contiguous() for i in range(0, L, n)]
        kc = [k[:, i:i + n].contiguous() for i in range(0, L, n)]
        vc = [v[:, i:i + n].contiguous() for i in range(0, L, n)]
        oc = [torch.empty_like(x) for x in qc]
        cache = swa.Cache(B, Hkv, d, w, s, max_len=(L if w < 0 else None))
        o = torch.empty_like(q)

        def chunked():
            for j in range(len(qc)):
                swa.prefill_chunk(qc[j], kc[j], vc[j], cache, j * n, out=oc[j])

        ms_chunk = _time_graph(chunked, steps, flush)
        ms_full = _time_graph(lambda: swa.prefill(q, k, v, w, s, out=o), steps, flush)
        fl = prefill_flops(B, L, Hq, d, w)
        print(json.dumps({"suite": "chunk", "B": B, "L": L, "w": w if w > 0 else "inf", "s": s,
                          "chunk": n, "ms_chunked": ms_chunk, "ms_whole": ms_full,
                          "tflops_chunked": fl / (ms_chunk * 1e-3) / 1e12,
                          "tok_s_chunked": B * L / (ms_chunk * 1e-3),
                          "overhead": ms_chunk / ms_full - 1.0,
                          "frac_tensor_peak_chunked": fl / (ms_chunk * 1e-3) / 1e12 / pk["bf16_tflops"],
                          "l2": L2_NOTE}), flush=True)
        del q, k, v, qc, kc, vc, oc, cache, o
        torch.cuda.empty_cache()


def suite_varlen(steps: int):
    """Ragged-batch prefill (prefill_varlen) against a padded batch and
    against one prefill per sequence, Llama attention shape (Hq=32, Hkv=8,
    d=128): 64 sequences with seeded lengths uniform in [256, 8192]
    (about 270K tokens), SWA(64,4) and SWA(512,4).  TFLOP/s count only the
    attended pairs of the real tokens; L2 is flushed before each step."""
    import numpy as np
    import torch

    import sliding_window_attention_prefill_gb300 as swa
    from sliding_window_attention_prefill_gb300 import build, inputs
    build.build()
    pk = peaks()
    flush = L2Flush()
    Hq, Hkv, d = 32, 8, 128
    rng = np.random.default_rng(0)
    lengths = [int(x) for x in rng.integers(256, 8193, 64)]
    total, max_len = sum(lengths), max(lengths)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device="cuda")
    q, k, v = inputs.prefill_inputs(1, total, Hq, Hkv, d, seed=0)
    q, k, v = q[0].cuda(), k[0].cuda(), v[0].cuda()
    o = torch.empty_like(q)
    seqs = []
    for b, n in enumerate(lengths):
        a = int(cu[b])
        seqs.append((q[a:a + n].unsqueeze(0), k[a:a + n].unsqueeze(0), v[a:a + n].unsqueeze(0),
                     o[a:a + n].unsqueeze(0)))
    qp = torch.zeros(len(lengths), max_len, Hq, d, dtype=q.dtype, device="cuda")
    kp = torch.zeros(len(lengths), max_len, Hkv, d, dtype=q.dtype, device="cuda")
    vp = torch.zeros_like(kp)
    op = torch.empty_like(qp)
    for w, s in [(64, 4), (512, 4)]:
        fl = sum(prefill_flops(1, n, Hq, d, w) for n in lengths)
        ms_var = _time_graph(lambda: swa.prefill_varlen(q, k, v, cu, w, s, max_len=max_len, out=o),
                             steps, flush)
        ms_pad = _time_graph(lambda: swa.prefill(qp, kp, vp, w, s, out=op), steps, flush)

        def per_seq():
            for qs, ks, vs, os_ in seqs:
                swa.prefill(qs, ks, vs, w, s, out=os_)

        ms_seq = _time_graph(per_seq, steps, flush)
        tf = fl / (ms_var * 1e-3) / 1e12
        print(json.dumps({"suite": "varlen", "sequences": len(lengths), "tokens": total,
                          "max_len": max_len, "w": w, "s": s, "ms_varlen": ms_var,
                          "ms_padded_batch": ms_pad, "ms_per_sequence_calls": ms_seq,
                          "tflops_varlen": tf, "tok_s_varlen": total / (ms_var * 1e-3),
                          "frac_tensor_peak": tf / pk["bf16_tflops"], "l2": L2_NOTE}), flush=True)
    del q, k, v, o, qp, kp, vp, op, seqs
    torch.cuda.empty_cache()


CONTEXT_POSITIONS = [1 << e for e in range(7, 19)]  # 128 .. 262144
CONTEXT_WINDOWS = [64, 128, 256, 512, -1]
CONTEXT_LAYERS = 4
CONTEXT_MAX_CACHE_BYTES = 160 << 30  # all layers' caches of one point


def context_cache_bytes(B, Hkv, d, cap, layers=CONTEXT_LAYERS) -> int:
    """Bytes of K and V cache of `layers` layers with `cap` slots each."""
    return layers * 2 * B * Hkv * cap * d * 2


# Attention shapes of the context sweep: the Llama-3.1-8B layer (bf16), and
# the pages' own system-test model (paper summary page, section "Method
# steps", step five: D = 1024, 16 heads of 64, batch 1, fp16).
CONTEXT_SHAPES = {
    "llama": {"Hq": 32, "Hkv": 8, "d": 128, "dtype": "bf16"},
    "paper": {"Hq": 16, "Hkv": 16, "d": 64, "dtype": "f16"},
}


def context_points(batches=(1, 256), Hkv: int = 8, d: int = 128):
    """(B, w, pos) of the context sweep whose caches fit the memory budget;
    an infinite window needs pos+1 slots, a finite one w."""
    pts, skipped = [], []
    for B in batches:
        for w in CONTEXT_WINDOWS:
            for P in CONTEXT_POSITIONS:
                cap = P + 1 if w < 0 else w
                if context_cache_bytes(B, Hkv, d, cap) > CONTEXT_MAX_CACHE_BYTES:
                    skipped.append((B, w, P))
                else:
                    pts.append((B, w, P))
    return pts, skipped


def suite_context(steps: int, batches=(1, 256), shape: str = "llama", hybrid: bool = False):
    """Decode context sweep through a stack of 4 attention layers: the Llama
    shape (Hq=32, Hkv=8, d=128, bf16) or the pages' system-test shape
    (Hq=Hkv=16, d=64, fp16), N(0,1) values.  For each window w in
    {64,128,256,512} with s=4, and w = infinity (full causal), each batch
    size, and position P from 128 to 262144: every layer holds a cache in the
    state reached after P tokens (every slot a decode at P reads holds an
    N(0,1) value), and one step appends token P and decodes it in each of the
    4 layers.  Prints tok/s, the decode kernel's KV read rate and the cache
    bytes held.  Points whose caches exceed 160 GiB are skipped (an infinite
    window at batch 256 beyond 32768 positions) and listed.  With ``hybrid``
    the layers are instead the LoLCATs-style mixture the pages compare
    against: a 256-token window without sinks plus a linear-attention state
    of the evicted tokens (df = d/2 Hedgehog features per half), each step
    a hybrid append and a hybrid decode."""
    import torch

    import sliding_window_attention_prefill_gb300 as swa
    from sliding_window_attention_prefill_gb300 import build
    build.build()
    pk = peaks()
    flush = L2Flush()
    sh = CONTEXT_SHAPES[shape]
    Hq, Hkv, d, s = sh["Hq"], sh["Hkv"], sh["d"], 4
    dt = torch.float16 if sh["dtype"] == "f16" else torch.bfloat16
    gen = torch.Generator(device="cuda")
    pts, skipped = context_points(batches, Hkv, d)
    if hybrid:
        pts = [(B, 256, P) for B in batches for P in CONTEXT_POSITIONS]
        skipped = []
    df = d // 2
    for B, w, P in pts:
        gen.manual_seed(B * 1000003 + P * 7 + (w + 1))
        layers = []
        for _ in range(CONTEXT_LAYERS):
            c = swa.Cache(B, Hkv, d, w, (s if w > 0 else 0) if not hybrid else 0,
                          max_len=(P + 1 if w < 0 else None), dtype=dt)
            c.k.normal_(generator=gen)
            c.v.normal_(generator=gen)
            kn = torch.randn(B, 1, Hkv, d, generator=gen, device="cuda").to(dt)
            vn = torch.randn(B, 1, Hkv, d, generator=gen, device="cuda").to(dt)
            q = torch.randn(B, Hq, d, generator=gen, device="cuda").to(dt)
            st = None
            if hybrid:
                Wf = torch.randn(Hkv, d, df, generator=gen, device="cuda") * (0.3 / d ** 0.5)
                st = swa.LinearState(c, Wf)
            layers.append((c, kn, vn, q, torch.empty_like(q), swa.workspace_for(c, Hq), st))
        pos = torch.full((B,), P, dtype=torch.int32, device="cuda")

        def step():
            for c, kn, vn, q, o, ws, st in layers:
                if hybrid:
                    swa.hybrid_append(c, st, kn, vn, P)
                    swa.hybrid_decode(q, c, st, pos, out=o)
                else:
                    swa.append_decode(q, kn, vn, c, pos, out=o, workspace=ws)

        def decode_only():
            for c, kn, vn, q, o, ws, st in layers:
                if hybrid:
                    swa.hybrid_decode(q, c, st, pos, out=o)
                else:
                    swa.decode(q, c, pos, out=o, workspace=ws)

        ms = _time_graph(step, steps, flush)
        ms_dec = _time_graph(decode_only, steps, flush)
        n_valid = P + 1 if w < 0 else min(P + 1, w)
        kv = CONTEXT_LAYERS * 2 * B * Hkv * d * 2 * n_valid
        by = CONTEXT_LAYERS * decode_bytes(B, Hq, Hkv, d, n_valid)
        if hybrid:  # the state S, z of every (sequence, kv head) is read too
            by += CONTEXT_LAYERS * B * Hkv * (2 * df) * (d + 1) * 4
        cap = layers[0][0].cap
        state_bytes = CONTEXT_LAYERS * B * Hkv * (2 * df) * (d + 1) * 4 if hybrid else 0
        print(json.dumps({"suite": "context", "mode": "hybrid" if hybrid else "swa",
                          "shape": shape, "dtype": sh["dtype"], "Hq": Hq,
                          "Hkv": Hkv, "d": d, "B": B, "w": w if w > 0 else "inf",
                          "s": s if w > 0 else 0, "pos": P, "layers": CONTEXT_LAYERS,
                          "ms_step": ms, "tok_s": B / (ms * 1e-3), "ms_decode": ms_dec,
                          "kv_read_gbs": kv / (ms_dec * 1e-3) / 1e9,
                          "frac_hbm": by / (ms_dec * 1e-3) / 1e9 / pk["hbm_gbs"],
                          "cache_bytes_held": context_cache_bytes(B, Hkv, d, cap) + state_bytes,
                          "cache_bytes_read": kv}), flush=True)
        del layers, step, decode_only
        torch.cuda.empty_cache()
    if skipped:
        print(json.dumps({"suite": "context", "shape": shape, "skipped": [
            {"B": B, "w": "inf" if w < 0 else w, "pos": P} for B, w, P in skipped],
            "reason": "caches above 160 GiB"}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["swa", "reference"], default="swa")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="reference arm: oracle time for the whole run (sizes its sample)")
    ap.add_argument("--suite", choices=["prefill", "decode", "context", "chunk", "varlen"], default=None,
                    help="auxiliary per-config lines instead of the headline step")
    ap.add_argument("--reps", type=int, default=40, help="suites: timed replays per case")
    ap.add_argument("--w", type=int, default=None, help="prefill suite: only this window")
    ap.add_argument("--B", type=int, default=None, help="prefill and decode suites: batch override")
    ap.add_argument("--L", type=int, default=None, help="prefill suite: length override")
    ap.add_argument("--decode-steps", type=int, default=1024, help="decode suite: steps")
    ap.add_argument("--batches", type=str, default="1,256", help="context suite: batch sizes")
    ap.add_argument("--hybrid", action="store_true",
                    help="context suite: the window + linear mixture instead of SWA(w,4)")
    ap.add_argument("--shape", choices=sorted(CONTEXT_SHAPES), default="llama",
                    help="context suite: attention shape (llama: 32/8 heads of 128, bf16; "
                         "paper: 16 heads of 64, fp16)")
    args = ap.parse_args()
    if args.suite == "prefill":
        suite_prefill(args.reps, args.w, args.B, args.L)
        return
    if args.suite == "decode":
        suite_decode(args.reps, args.w, args.decode_steps, args.B)
        return
    if args.suite == "chunk":
        suite_chunk(max(args.reps // 2, 10))
        return
    if args.suite == "varlen":
        suite_varlen(max(args.reps // 2, 10))
        return
    if args.suite == "context":
        suite_context(max(min(args.reps // 2, 20), 5),
                      tuple(int(b) for b in args.batches.split(",")), args.shape, args.hybrid)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    run_swa(args, rank, world, local_rank)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
