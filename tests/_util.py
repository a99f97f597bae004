"""Helpers shared by the tests: tolerances, device copies, error norms."""
from __future__ import annotations

import numpy as np
import torch

# Tolerances: normwise max error ‖out − ref‖∞ / ‖ref‖∞, separately for y and the
# final state.  fp32 io: 1e-4; bf16 io with fp32 accumulation and state: 2e-2.
TOL = {"f32": 1e-4, "bf16": 2e-2}


def normwise_err(out, ref) -> float:
    out = out.detach().double().cpu().numpy() if isinstance(out, torch.Tensor) else np.asarray(out, np.float64)
    ref = ref.detach().double().cpu().numpy() if isinstance(ref, torch.Tensor) else np.asarray(ref, np.float64)
    assert out.shape == ref.shape, (out.shape, ref.shape)
    if not np.all(np.isfinite(out)):
        return float("inf")
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    diff = float(np.max(np.abs(out - ref))) if ref.size else 0.0
    return diff / scale if scale > 0 else diff


def to_device(inp: dict, device="cuda") -> dict:
    return {k: (None if v is None else v.to(device)) for k, v in inp.items()}


def poison_like(t: torch.Tensor) -> torch.Tensor:
    """Output buffer pre-filled with NaN so that any element a kernel leaves
    unwritten fails the comparison."""
    return torch.full_like(t, float("nan"))
