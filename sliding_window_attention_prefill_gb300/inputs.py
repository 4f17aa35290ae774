"""Seeded synthetic inputs, shared by the tests, the benchmark and the oracle checks.

This module only draws random numbers; it holds none of the attention
arithmetic.  Recipe: a torch CPU generator seeded with ``seed``; each tensor is
drawn as float32 N(0, 1) in a fixed order and rounded to bf16, or to fp16
where a ``dtype`` says so (round-to-nearest-even).  The 16-bit tensors are
what both the CUDA path and the oracle read.

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


def normal16(shape, gen: torch.Generator, dtype=torch.bfloat16) -> torch.Tensor:
    """float32 N(0,1) drawn from ``gen``, rounded to ``dtype`` (bf16 or fp16; CPU tensor)."""
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(dtype)


def device_generator(seed: int, device="cuda") -> torch.Generator:
    """A torch generator on ``device``, for inputs too large to draw on the CPU
    in a test's time (multi-GB caches); the draws differ from the CPU
    generator's, so a test that uses it copies what it checks to the host."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal16_on(shape, gen: torch.Generator, dtype=torch.bfloat16) -> torch.Tensor:
    """float32 N(0,1) drawn from ``gen`` on the generator's device, rounded to
    ``dtype`` (bf16 or fp16)."""
    return torch.randn(*shape, generator=gen, device=gen.device, dtype=torch.float32).to(dtype)


def normal_bf16(shape, gen: torch.Generator) -> torch.Tensor:
    """float32 N(0,1) drawn from ``gen``, rounded to bf16 (CPU tensor)."""
    return normal16(shape, gen, torch.bfloat16)


def prefill_inputs(B: int, L: int, Hq: int, Hkv: int, d: int, seed: int = 0,
                   sink_rows: int = 0, sink_scale: float = 8.0, dtype=torch.bfloat16):
    """q [B,L,Hq,d], k [B,L,Hkv,d], v [B,L,Hkv,d] of ``dtype`` on the CPU.

    With ``sink_rows > 0`` the key rows of the first ``sink_rows`` positions are
    multiplied by ``sink_scale`` (a power of two keeps them exact in bf16 and
    fp16).
    """
    g = generator(seed)
    q = normal16((B, L, Hq, d), g, dtype)
    k = normal16((B, L, Hkv, d), g, dtype)
    v = normal16((B, L, Hkv, d), g, dtype)
    if sink_rows > 0:
        k[:, :sink_rows] = (k[:, :sink_rows].float() * sink_scale).to(dtype)
    return q, k, v


def decode_stream(B: int, Hq: int, Hkv: int, d: int, prompt: int, steps: int, seed: int = 0,
                  dtype=torch.bfloat16):
    """A prompt of ``prompt`` tokens followed by ``steps`` decode steps.

    Returns (k_prompt [B,prompt,Hkv,d], v_prompt, k_steps [steps,B,1,Hkv,d],
    v_steps, q_steps [steps,B,Hq,d]), all of ``dtype`` on the CPU.
    """
    g = generator(seed)
    k_prompt = normal16((B, prompt, Hkv, d), g, dtype)
    v_prompt = normal16((B, prompt, Hkv, d), g, dtype)
    k_steps = normal16((steps, B, 1, Hkv, d), g, dtype)
    v_steps = normal16((steps, B, 1, Hkv, d), g, dtype)
    q_steps = normal16((steps, B, Hq, d), g, dtype)
    return k_prompt, v_prompt, k_steps, v_steps, q_steps
