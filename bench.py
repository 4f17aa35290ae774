#!/usr/bin/env python3
"""Benchmark of the SWA(w,s) hot path on GB300.

One step = the whole path over one batch of synthetic input:
  prefill of a 4096-token prompt (sliding-window attention with sinks, SWA(64,4),
  Llama-3.1-8B attention shape: 32 query heads, 8 key/value heads, d = 128,
  first 4 key rows x8), bulk append of the prompt's keys/values into a fixed
  SWA(64,4) cache, then one decode token (append + decode).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl swa|reference]
Under torchrun each rank runs its own batch on its own GPU (no data exchange;
weak scaling) and rank 0 prints one JSON line.

`value` is tokens/s of the whole step (prompt tokens + decoded tokens), device
time from CUDA events on the launching stream, inputs resident in HBM, L2
flushed (256 MiB written, another 256 MiB read) before every timed step.  `e2e` is the same metric
through the C ABI with pinned host buffers, copies inside the timed region.
`--impl reference` times the fp64 CPU oracle on a bounded sample of the same
workload on the host cores.
"""
from __future__ import annotations

import argparse
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

WORK = dict(B=1, L=4096, Hq=32, Hkv=8, d=128, w=64, s=4, sink_rows=4)
METRIC = "SWA(w,4) decode tok/s + KV-read GB/s vs HBM peak; prefill TFLOP/s vs tensor peak"
WORKLOAD_NAME = ("prefill SWA(64,4) B=1 L=4096 Hq=32 Hkv=8 d=128 (first 4 key rows x8) "
                 "+ bulk cache append + 1 decode token")
L2_FLUSH_BYTES = 256 << 20
L2_NOTE = (f"flushed before each step: {L2_FLUSH_BYTES >> 20} MiB written, then another "
           f"{L2_FLUSH_BYTES >> 20} MiB read, so the timed kernels start on a cold L2 that holds "
           f"no dirty lines of the flush")


class L2Flush:
    """Evicts the timed kernels' data from L2 (129 MB on GB300): write one
    buffer larger than L2, then read a second one, which also writes the
    first buffer's dirty lines back before the timed region starts."""

    def __init__(self, device="cuda"):
        import torch
        self.wbuf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.rbuf = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=device)

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


def peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return {"hbm_gbs": float(m["hbm_gbs"]), "bf16_tflops": float(m["bf16_tflops"]),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def prefill_traffic():
    """dram bytes per prefill launch from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "prefill_traffic.json")
    src = os.path.join(ROOT, "sliding_window_attention_prefill_gb300", "csrc", "swa_prefill.cu")
    try:
        with open(path) as f:
            rec = json.load(f)
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()
        if rec.get("kernel_sha256") == h and rec.get("workload") == WORKLOAD_NAME:
            return float(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# ----------------------------------------------------------------------------- ranks
def rank_seed(rank: int) -> int:
    """Each rank draws its own batch (weak scaling: independent sequences)."""
    return 1000 * rank


def tokens_per_step(world: int) -> int:
    """Tokens all ranks process in one step: every rank's prompt + decoded token."""
    return WORK["B"] * (WORK["L"] + 1) * world


def max_over_ranks(values, device):
    """Element-wise max of per-rank timings (the slowest rank sets the pace)."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return t.tolist()


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.t0 = self.t1 = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(gpu_index)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.4)

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def result(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except Exception:
                continue
        inside = [r for r in rows if self.t0 - 0.06 <= r[0] <= self.t1 + 0.06]
        used = inside if inside else rows
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in used:
            for n, v in zip(names, r[3]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median([r[1] for r in used]) if used else None,
                "sm_max_mhz": max(r[2] for r in used) if used else None,
                "reasons": sorted(reasons), "samples": len(used),
                "window": "timed region" if inside else "around the timed region"}


# ----------------------------------------------------------------------------- oracle arm
def oracle_step_rate(sample_positions: int, seed: int = 0):
    """The oracle's step restricted to `sample_positions` prompt positions (all
    heads) + the decode token.  Returns (run, tokens, oracle, k history,
    v history): run() performs one such step, `tokens` is what it counts."""
    import numpy as np

    import oracle
    from sliding_window_attention_prefill_gb300 import inputs
    W = WORK
    q, k, v = inputs.prefill_inputs(W["B"], W["L"], W["Hq"], W["Hkv"], W["d"], seed=seed,
                                    sink_rows=W["sink_rows"])
    orc = oracle.get()
    qb, kb, vb = oracle.bf16_bits(q), oracle.bf16_bits(k), oracle.bf16_bits(v)
    L = W["L"]
    ts = np.linspace(0, L - 1, sample_positions).astype(np.int64)
    rows = np.array([[b, t, h] for b in range(W["B"]) for t in ts for h in range(W["Hq"])], np.int64)
    g = inputs.generator(seed + 1)
    k1 = oracle.bf16_bits(inputs.normal_bf16((W["B"], 1, W["Hkv"], W["d"]), g))
    v1 = oracle.bf16_bits(inputs.normal_bf16((W["B"], 1, W["Hkv"], W["d"]), g))
    q1 = oracle.bf16_bits(inputs.normal_bf16((W["B"], W["Hq"], W["d"]), g))
    hist_k = np.concatenate([kb, k1], axis=1)
    hist_v = np.concatenate([vb, v1], axis=1)
    ck = np.zeros((W["B"], W["Hkv"], W["w"], W["d"]), np.uint16)
    cv = np.zeros_like(ck)

    def run():
        orc.prefill_rows(qb, kb, vb, rows, W["w"], W["s"])
        orc.cache_append(ck, cv, kb, vb, 0, W["w"], W["s"])
        orc.cache_append(ck, cv, k1, v1, L, W["w"], W["s"])
        orc.decode_cache(q1, ck, cv, [L] * W["B"], W["w"], W["s"])

    return run, W["B"] * (sample_positions + 1), orc, hist_k, hist_v


def run_reference(args, rank: int):
    if rank != 0:
        return
    import oracle
    oracle.build()
    orc = oracle.get()
    cores = orc.threads(None)
    # size the sample so the whole run stays within about --ref-seconds
    calib_run, calib_tok, *_ = oracle_step_rate(64)
    t = time.perf_counter()
    calib_run()
    per_pos = (time.perf_counter() - t) / 64
    budget = args.ref_seconds / max(1, args.steps + args.warmup)
    S = int(max(16, min(WORK["L"], budget / max(per_pos, 1e-9))))
    run, tokens, *_ = oracle_step_rate(S)
    for _ in range(args.warmup):
        run()
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        run()
        times.append(time.perf_counter() - t)
    mean = sum(times) / len(times)
    value = tokens / mean
    sample = (f"{S} of {WORK['L']} prompt positions (all {WORK['Hq']} heads, evenly spaced) + "
              f"the cache append + 1 decode token per step")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": mean * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_NAME, "oracle": "fp64 C, OpenMP over rows"},
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- GPU arm
def run_swa(args, rank: int, world: int, local_rank: int):
    import torch

    import sliding_window_attention_prefill_gb300 as swa
    from sliding_window_attention_prefill_gb300 import build, inputs

    build.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    W = WORK
    B, L, Hq, Hkv, d, w, s = W["B"], W["L"], W["Hq"], W["Hkv"], W["d"], W["w"], W["s"]
    seed = rank_seed(rank)
    q_h, k_h, v_h = inputs.prefill_inputs(B, L, Hq, Hkv, d, seed=seed, sink_rows=W["sink_rows"])
    g = inputs.generator(seed + 1)
    k1_h = inputs.normal_bf16((B, 1, Hkv, d), g)
    v1_h = inputs.normal_bf16((B, 1, Hkv, d), g)
    q1_h = inputs.normal_bf16((B, Hq, d), g)
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    k1, v1, q1 = k1_h.to(dev), v1_h.to(dev), q1_h.to(dev)
    o = torch.empty_like(q)
    od = torch.empty_like(q1)
    cache = swa.Cache(B, Hkv, d, w, s, device=dev)
    pos = torch.full((B,), L, dtype=torch.int32, device=dev)
    flush = L2Flush(dev)

    side = torch.cuda.Stream(dev)  # the prompt's cache append, beside the prefill

    def prefill_part():
        # The prefill and the prompt's cache append read the same k, v and
        # nothing of each other: the append runs on a second stream beside
        # the prefill (joined before the decode token, which needs it).
        cur = torch.cuda.current_stream(dev)
        fork = torch.cuda.Event()
        fork.record(cur)
        side.wait_event(fork)
        swa.prefill(q, k, v, w, s, out=o)
        with torch.cuda.stream(side):
            cache.append(k, v, 0)
        join = torch.cuda.Event()
        join.record(side)
        cur.wait_event(join)

    def cache_decode_part():
        swa.append_decode(q1, k1, v1, cache, pos, out=od)  # the token's append + its decode

    def step_part():
        prefill_part()
        cache_decode_part()

    launches_per_step = 1 + 1 + 1 + (1 if swa.decode_workspace_bytes(B, Hq, Hkv, d, cache.cap, w) else 0)
    stream = torch.cuda.current_stream(dev)
    # Warm up once outside capture (sets kernel attributes), then capture the
    # whole step as one CUDA graph (the timed step), and its two halves as
    # graphs of their own (the kernel timings: events between graphs; timing
    # events recorded inside a graph add nodes that slow it down).
    step_part()
    torch.cuda.synchronize()
    graph, g1, g2 = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream(dev)
    cs.wait_stream(stream)
    with torch.cuda.stream(cs):
        with torch.cuda.graph(graph, stream=cs):
            step_part()
        with torch.cuda.graph(g1, stream=cs, pool=graph.pool()):
            prefill_part()
        with torch.cuda.graph(g2, stream=cs, pool=graph.pool()):
            cache_decode_part()
    stream.wait_stream(cs)
    torch.cuda.synchronize()

    # flush time, to stretch the timed region so clock samples land in it
    ev_a, ev_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev_a.record()
    for _ in range(5):
        flush(1)
    ev_b.record()
    torch.cuda.synchronize()
    t_flush = ev_a.elapsed_time(ev_b) / 5e3
    flush_reps = max(1, math.ceil((0.6 / max(args.steps, 1)) / max(t_flush, 1e-6)))
    flush_reps = min(flush_reps, 64)

    for _ in range(args.warmup):
        flush(1)
        graph.replay()
        flush(1)
        g1.replay()
        g2.replay()
    torch.cuda.synchronize()

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    evk = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(local_rank) if rank == 0 else None
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark_start()
    for i in range(args.steps):  # the timed steps
        for _ in range(flush_reps):
            flush(i)
        ev[i][0].record()
        graph.replay()
        ev[i][1].record()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    for i in range(args.steps):  # the same steps in two halves: kernel times
        for _ in range(flush_reps):
            flush(i)
        evk[i][0].record()
        g1.replay()
        evk[i][1].record()
        g2.replay()
        evk[i][2].record()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark_end()
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    pre_ms = [e[0].elapsed_time(e[1]) for e in evk]
    dec_ms = [e[1].elapsed_time(e[2]) for e in evk]
    mean_step = sum(step_ms) / len(step_ms)
    mean_pre = sum(pre_ms) / len(pre_ms)
    mean_dec = sum(dec_ms) / len(dec_ms)

    # ---- end to end: pinned host buffers, copies inside the timed region.
    # Each step copies its inputs up (q, k, v of the prompt, the decode
    # token's k, v, q), runs the library calls and copies both outputs back.
    # Host <-> device copies run at about 200 GB/s per direction here, so
    # they dominate; as a serving loop with double-buffered I/O does, the
    # steps overlap: step i+1's inputs go up on one stream while step i
    # computes and its outputs come back on another (two sets of device and
    # host buffers).  value = steps / total time; every step's copies are in
    # the timed region.  The serial figure (one step at a time, synchronised
    # after each) is reported beside it.
    names = ("q", "k", "v", "k1", "v1", "q1")
    src = dict(q=q_h, k=k_h, v=v_h, k1=k1_h, v1=v1_h, q1=q1_h)
    host = [{n: src[n].pin_memory() for n in names} for _ in range(2)]
    devb = [dict(q=q, k=k, v=v, k1=k1, v1=v1, q1=q1, o=o, od=od),
            {**{n: torch.empty_like(src[n], device=dev) for n in names},
             "o": torch.empty_like(o), "od": torch.empty_like(od)}]
    o_host = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for _ in range(2)]
    od_host = [torch.empty(od.shape, dtype=od.dtype, pin_memory=True) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host[0].values())
    d2h = o_host[0].numel() * 2 + od_host[0].numel() * 2
    up, down, comp = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.current_stream(dev)

    def e2e_step(i, done):
        # done[j] = (inputs consumed, outputs read back) events of step j
        b, hb = devb[i & 1], host[i & 1]
        if i >= 2:  # this buffer set was step i-2's
            up.wait_event(done[i - 2][0])
        with torch.cuda.stream(up):
            for n in names:
                b[n].copy_(hb[n], non_blocking=True)
        e_up = torch.cuda.Event()
        e_up.record(up)
        comp.wait_event(e_up)
        if i >= 2:
            comp.wait_event(done[i - 2][1])
        fork = torch.cuda.Event()
        fork.record(comp)
        side.wait_event(fork)
        swa.prefill(b["q"], b["k"], b["v"], w, s, out=b["o"])
        with torch.cuda.stream(side):
            cache.append(b["k"], b["v"], 0)
        join = torch.cuda.Event()
        join.record(side)
        comp.wait_event(join)
        swa.append_decode(b["q1"], b["k1"], b["v1"], cache, pos, out=b["od"])
        e_comp = torch.cuda.Event()
        e_comp.record(comp)
        down.wait_event(e_comp)
        with torch.cuda.stream(down):
            o_host[i & 1].copy_(b["o"], non_blocking=True)
            od_host[i & 1].copy_(b["od"], non_blocking=True)
        e_down = torch.cuda.Event()
        e_down.record(down)
        done.append((e_comp, e_down))

    for _ in range(max(3, min(args.warmup, 10))):
        e2e_step(0, [])
        torch.cuda.synchronize()
    n_e2e = max(4, min(args.steps, 200))
    # serial: one step at a time
    serial_ms = []
    for i in range(min(n_e2e, 20)):
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(up)
        e2e_step(0, [])
        down.wait_stream(comp)
        b_.record(down)
        b_.synchronize()
        serial_ms.append(a.elapsed_time(b_))
    mean_e2e_serial = sum(serial_ms) / len(serial_ms)
    # overlapped: n_e2e steps back to back
    torch.cuda.synchronize()
    a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(up)
    done = []
    for i in range(n_e2e):
        e2e_step(i, done)
    up.wait_stream(down)
    up.wait_stream(comp)
    b_.record(up)
    b_.synchronize()
    mean_e2e = a.elapsed_time(b_) / n_e2e

    # ---- max over ranks
    if world > 1:
        mean_step, mean_pre, mean_dec, mean_e2e, mean_e2e_serial = max_over_ranks(
            [mean_step, mean_pre, mean_dec, mean_e2e, mean_e2e_serial], dev)

    if rank != 0:
        return
    tokens = tokens_per_step(world)
    value = tokens / (mean_step * 1e-3)
    pk = peaks()
    pbytes = prefill_bytes(B, L, Hq, Hkv, d)
    pflops = prefill_flops(B, L, Hq, d, w)
    n_valid = min(L + 1, w)
    dbytes = decode_bytes(B, Hq, Hkv, d, n_valid)
    achieved_gbs = pbytes / (mean_pre * 1e-3) / 1e9
    tflops = pflops / (mean_pre * 1e-3) / 1e12
    clocks = sampler.result() if sampler else None
    cpu = None
    if world == 1:
        cpu = cpu_baseline()
    line = {
        "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": mean_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME, "global_batch": B * world, "seq_len": L,
                   "window": w, "sinks": s, "l2": L2_NOTE,
                   "timing": "CUDA events around the replay of the step, captured as one CUDA graph; the prefill and decode times from the same steps replayed as two graphs, events between them"},
        "gpu_launches": launches_per_step * args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved_gbs / pk["hbm_gbs"],
                     "traffic": prefill_traffic(), "kernel": "swa_prefill_kernel",
                     "algorithmic_bytes_per_launch": pbytes,
                     "peak_source": pk["source"] + " (MEASURED_PEAKS.json hbm_gbs, burst copy)"},
        "prefill": {"ms": mean_pre, "tflops": tflops, "frac_tensor_peak": tflops / pk["bf16_tflops"],
                    "gbs": achieved_gbs, "algorithmic_gflop": pflops / 1e9},
        "decode": {"ms_append_and_decode": mean_dec, "tok_s": B * world / (mean_dec * 1e-3),
                   "kv_bytes": dbytes,
                   "note": "one token after the prompt (one append_decode; the prompt's cache "
                           "append runs beside the prefill); B=1 is latency-bound"},
        "e2e": {"value": tokens / (mean_e2e * 1e-3), "unit": "tok/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": mean_e2e,
                "timing": f"{n_e2e} steps back to back, the copies of consecutive steps "
                          "overlapping (double-buffered host and device buffers)",
                "serial": {"value": tokens / (mean_e2e_serial * 1e-3), "ms_per_step": mean_e2e_serial,
                           "timing": "one step at a time, synchronised after each"}},
        "clocks": clocks,
    }
    if cpu:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


def cpu_baseline() -> dict:
    """The oracle on a bounded sample of the same step (about 10-20 s of CPU work)."""
    import oracle
    oracle.build()
    S = 512
    run, tokens, orc, *_ = oracle_step_rate(S)
    t0 = time.perf_counter()
    n = 0
    while True:
        run()
        n += 1
        if time.perf_counter() - t0 > 10.0 or n >= 50:
            break
    dt = (time.perf_counter() - t0) / n
    return {"value": tokens / dt, "unit": "tok/s", "cores": orc.threads(None), "kind": "oracle",
            "sample": f"{S} of {WORK['L']} prompt positions (all heads) + cache append + 1 decode "
                      f"token per step, {n} steps"}


# ----------------------------------------------------------------------------- suites
def _time_graph(fn, steps: int, flush, warm: int = 3) -> float:
    """Mean ms of `fn` replayed as a CUDA graph, L2 flushed before each replay."""
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
    return sum(a.elapsed_time(b) for a, b in evs) / steps


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


def suite_decode(steps: int, only_w=None, n_steps: int = 1024):
    """Decode configuration: B=64, Hq=32, Hkv=8, d=128, SWA(w,4) for w in
    {64, 512}; the cache is filled from a 4096-token N(0,1) prompt, then
    `n_steps` decode steps each append one N(0,1) token and decode it (one
    append_decode call).  Every step is its own captured CUDA graph; L2 is
    flushed before each step.  Also times the decode kernel alone."""
    import torch

    import sliding_window_attention_prefill_gb300 as swa
    from sliding_window_attention_prefill_gb300 import build, inputs
    build.build()
    pk = peaks()
    flush = L2Flush()
    B, Hq, Hkv, d, s, prompt = 64, 32, 8, 128, 4, 4096
    for w in [x for x in (64, 512) if only_w is None or x == only_w]:
        kp, vp, ks, vs, qs = inputs.decode_stream(B, Hq, Hkv, d, prompt, n_steps, seed=0)
        c = swa.Cache(B, Hkv, d, w, s)
        c.append(kp.cuda(), vp.cuda(), 0)
        del kp, vp
        ks, vs, qs = ks.cuda(), vs.cuda(), qs.cuda()
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
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["swa", "reference"], default="swa")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="reference arm: oracle time for the whole run (sizes its sample)")
    ap.add_argument("--suite", choices=["prefill", "decode", "context", "chunk", "varlen"], default=None,
                    help="auxiliary per-config lines instead of the headline step")
    ap.add_argument("--w", type=int, default=None, help="prefill suite: only this window")
    ap.add_argument("--B", type=int, default=None, help="prefill suite: batch override")
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
        suite_prefill(max(args.steps // 10, 10), args.w, args.B, args.L)
        return
    if args.suite == "decode":
        suite_decode(max(args.steps // 4, 20), args.w, args.decode_steps)
        return
    if args.suite == "chunk":
        suite_chunk(max(args.steps // 20, 10))
        return
    if args.suite == "varlen":
        suite_varlen(max(args.steps // 20, 10))
        return
    if args.suite == "context":
        suite_context(max(min(args.steps // 40, 20), 5),
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
