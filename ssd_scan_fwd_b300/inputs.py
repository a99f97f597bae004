"""Seeded synthetic inputs for the SSD forward pass.

This module holds no arithmetic of the scan itself: it only draws random
tensors with the distributions of the Mamba-2-shaped workloads and rounds the
io tensors to their storage dtype.  Both the CUDA path (tests, benchmark) and
the oracle receive exactly these tensors (the oracle upcasts them to fp64).

Distributions (per workload):
  x ~ N(0, 1);  dt = softplus(z - 1), z ~ N(0, 1)  (Δ arrives already positive);
  A_h = -exp(u), u ~ U(0, ln 16);  Bm, Cm ~ N(0, 1) / sqrt(N);  D ~ N(0, 1);
  init_state ~ N(0, 0.1²) where the workload has one, else none (zeros).
x, Bm, Cm are drawn in fp32 and rounded to the io dtype; dt, A, D and the
state stay fp32.  Draw order is fixed: x, z, u, Bm, Cm, D, init_state.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seqlen: int
    nheads: int
    headdim: int
    dstate: int
    ngroups: int
    io_dtype: str  # "f32" or "bf16"
    has_init: bool
    seed: int

    @property
    def tokens(self) -> int:
        return self.batch * self.seqlen

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_fp32", 1, 256, 2, 16, 16, 1, "f32", False, 1000),
        Workload("mamba2_130m", 2, 2048, 24, 64, 128, 1, "bf16", False, 1001),
        Workload("mamba2_2p7b", 4, 8192, 80, 64, 128, 1, "bf16", False, 1002),
        Workload("long_grouped", 1, 65536, 32, 64, 128, 8, "bf16", True, 1003),
        Workload("nsweep_16", 8, 4096, 32, 64, 16, 1, "bf16", False, 1040),
        Workload("nsweep_64", 8, 4096, 32, 64, 64, 1, "bf16", False, 1041),
        Workload("nsweep_128", 8, 4096, 32, 64, 128, 1, "bf16", False, 1042),
        Workload("nsweep_256", 8, 4096, 32, 64, 256, 1, "bf16", False, 1043),
    ]
}


def torch_dtype(io_dtype: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[io_dtype]


def generate(w: Workload, seed: int | None = None) -> dict:
    """Draw one problem on the CPU.  Returns a dict of torch CPU tensors:
    x, dt, A, Bm, Cm, D, init_state (None when the workload has none)."""
    g = torch.Generator().manual_seed(w.seed if seed is None else seed)
    B, L, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    io = torch_dtype(w.io_dtype)
    x = torch.randn(B, L, H, P, generator=g)
    z = torch.randn(B, L, H, generator=g)
    dt = torch.nn.functional.softplus(z - 1.0)
    u = torch.rand(H, generator=g) * math.log(16.0)
    A = -torch.exp(u)
    Bm = torch.randn(B, L, G, N, generator=g) / math.sqrt(N)
    Cm = torch.randn(B, L, G, N, generator=g) / math.sqrt(N)
    D = torch.randn(H, generator=g)
    init = torch.randn(B, H, P, N, generator=g) * 0.1 if w.has_init else None
    return {
        "x": x.to(io).contiguous(),
        "dt": dt.contiguous(),
        "A": A.contiguous(),
        "Bm": Bm.to(io).contiguous(),
        "Cm": Cm.to(io).contiguous(),
        "D": D.contiguous(),
        "init_state": None if init is None else init.contiguous(),
    }


def algorithmic_bytes(w: Workload) -> int:
    """Bytes the forward pass must move at minimum: x in, y out, dt in,
    Bm and Cm in, final_state out, init_state in (when present).  A and D are
    negligible and not counted."""
    s = 2 if w.io_dtype == "bf16" else 4
    B, L, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    b = B * L * H * (2 * P * s + 4) + B * L * G * 2 * N * s + B * H * P * N * 4
    if w.has_init:
        b += B * H * P * N * 4
    return b


def algorithmic_flops(w: Workload, chunk: int = 128) -> int:
    """Useful multiply-add work of the chunked forward pass (2 flops per
    multiply-add), counting only what the method needs: per (token, head) the
    causal intra-chunk product (chunk + 1)·P on average, the chunk-state
    contraction 2·N·P and the read-out of the entering state 2·N·P; per
    (token, group) the C·Bᵀ product 2·chunk·N."""
    B, L, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    return B * L * (H * ((chunk + 1) * P + 4 * N * P) + G * 2 * chunk * N)


def generate_mimo(w: Workload, rank: int, seed: int | None = None) -> dict:
    """One problem with retrieval rank ``rank``: per token R value channels
    with their own x, Bm and Cm (same distributions as ``generate``), one Δ
    per token and head.  Shapes: x [B,L,R,H,P], dt [B,L,H], Bm/Cm [B,L,R,G,N].
    Draw order: x, z, u, Bm, Cm, D, init_state."""
    g = torch.Generator().manual_seed(w.seed if seed is None else seed)
    B, L, H, P, N, G, R = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups, rank
    io = torch_dtype(w.io_dtype)
    x = torch.randn(B, L, R, H, P, generator=g)
    z = torch.randn(B, L, H, generator=g)
    dt = torch.nn.functional.softplus(z - 1.0)
    u = torch.rand(H, generator=g) * math.log(16.0)
    A = -torch.exp(u)
    Bm = torch.randn(B, L, R, G, N, generator=g) / math.sqrt(N)
    Cm = torch.randn(B, L, R, G, N, generator=g) / math.sqrt(N)
    D = torch.randn(H, generator=g)
    init = torch.randn(B, H, P, N, generator=g) * 0.1 if w.has_init else None
    return {
        "x": x.to(io).contiguous(),
        "dt": dt.contiguous(),
        "A": A.contiguous(),
        "Bm": Bm.to(io).contiguous(),
        "Cm": Cm.to(io).contiguous(),
        "D": D.contiguous(),
        "init_state": None if init is None else init.contiguous(),
    }
