"""Shared helpers for the GPU parity tests."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# Tolerance for bf16 inputs with fp32 accumulation against the fp64 oracle:
# max |gpu - oracle| <= 2e-2 and sum |gpu - oracle| / sum |oracle| <= 1e-2.
MAX_ABS = 2e-2
MEAN_REL = 1e-2


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(got, ref: np.ndarray, what: str = "", max_abs: float = MAX_ABS,
                 mean_rel: float = MEAN_REL) -> tuple[float, float]:
    g = to_f64(got) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    d = np.abs(g - ref)
    mx = float(d.max()) if d.size else 0.0
    mr = float(d.sum() / max(np.abs(ref).sum(), 1e-30)) if d.size else 0.0
    assert mx <= max_abs and mr <= mean_rel, f"{what}: max|d|={mx:.3e} mean-rel={mr:.3e}"
    return mx, mr


def bits(t: torch.Tensor) -> np.ndarray:
    """Bit patterns of a bf16 or fp16 tensor (pass dtype="f16" to the oracle
    for fp16)."""
    return oracle.bits16(t.cpu())
