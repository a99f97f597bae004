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


def rowwise_normwise_err(out_y, out_f, ref_rows, batch: int):
    """Normwise errors (‖out − ref‖∞ / ‖ref‖∞ over the WHOLE tensors) of y and
    final_state, with the reference produced one batch row at a time so that
    full-size problems fit in host memory: ``ref_rows(b)`` returns the fp64
    (y [L,H,P], final [H,P,N]) of row b.  Every element is compared."""
    dy = sy = df = sf = 0.0
    for b in range(batch):
        ry, rf = ref_rows(b)
        oy = out_y[b].detach().double().cpu().numpy()
        if not np.all(np.isfinite(oy)):
            return float("inf"), float("inf")
        dy = max(dy, float(np.max(np.abs(oy - ry))))
        sy = max(sy, float(np.max(np.abs(ry))))
        del oy
        if out_f is not None:
            of = out_f[b].detach().double().cpu().numpy()
            if not np.all(np.isfinite(of)):
                return float("inf"), float("inf")
            df = max(df, float(np.max(np.abs(of - rf))))
            sf = max(sf, float(np.max(np.abs(rf))))
    ey = dy / sy if sy > 0 else dy
    ef = (df / sf if sf > 0 else df) if out_f is not None else 0.0
    return ey, ef
