"""Seeded synthetic inputs, shared by the tests, the benchmark and the oracle checks.

This module only draws random numbers; it holds none of the attention
arithmetic.  Recipe: a torch CPU generator seeded with ``seed``; each tensor is
drawn as float32 N(0, 1) in a fixed order and rounded to bf16
(round-to-nearest-even).  The bf16 tensors are what both the CUDA path and the
oracle read.

The shapes follow the attention of a Llama-3.1-8B-style layer (32 query heads,
8 key/value heads, head size 128), the model family the paper's long-context
study uses ("Sliding-window beats linear attention", summary page, section
"Method steps", step four); the sink-heavy variant scales the first key rows
by 8 (exact in bf16) so that the first tokens draw a large share of the
attention, the behaviour the pages describe for attention sinks (same page,
"Prerequisites / Attention sinks").
"""
from __future__ import annotations

import torch


def generator(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, gen: torch.Generator) -> torch.Tensor:
    """float32 N(0,1) drawn from ``gen``, rounded to bf16 (CPU tensor)."""
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


def prefill_inputs(B: int, L: int, Hq: int, Hkv: int, d: int, seed: int = 0,
                   sink_rows: int = 0, sink_scale: float = 8.0):
    """q [B,L,Hq,d], k [B,L,Hkv,d], v [B,L,Hkv,d] bf16 on the CPU.

    With ``sink_rows > 0`` the key rows of the first ``sink_rows`` positions are
    multiplied by ``sink_scale`` (a power of two keeps them exact in bf16).
    """
    g = generator(seed)
    q = normal_bf16((B, L, Hq, d), g)
    k = normal_bf16((B, L, Hkv, d), g)
    v = normal_bf16((B, L, Hkv, d), g)
    if sink_rows > 0:
        k[:, :sink_rows] = (k[:, :sink_rows].float() * sink_scale).to(torch.bfloat16)
    return q, k, v


def decode_stream(B: int, Hq: int, Hkv: int, d: int, prompt: int, steps: int, seed: int = 0):
    """A prompt of ``prompt`` tokens followed by ``steps`` decode steps.

    Returns (k_prompt [B,prompt,Hkv,d], v_prompt, k_steps [steps,B,1,Hkv,d],
    v_steps, q_steps [steps,B,Hq,d]), all bf16 on the CPU.
    """
    g = generator(seed)
    k_prompt = normal_bf16((B, prompt, Hkv, d), g)
    v_prompt = normal_bf16((B, prompt, Hkv, d), g)
    k_steps = normal_bf16((steps, B, 1, Hkv, d), g)
    v_steps = normal_bf16((steps, B, 1, Hkv, d), g)
    q_steps = normal_bf16((steps, B, Hq, d), g)
    return k_prompt, v_prompt, k_steps, v_steps, q_steps
