"""The seeded input recipe (CPU): shapes, dtypes, reproducibility, the stated
distributions, and the algorithmic-byte count the benchmark divides by.

The workloads are the tiny fp32 case, the 130M- and 2.7B-shaped layers, the
long grouped sequence and the state-size sweep; these checks pin the recipe
so that a change to a distribution or a draw order shows up here rather than
as a silent shift of every parity case."""
import math

import pytest
import torch

from ssd_scan_fwd_b300.inputs import WORKLOADS, algorithmic_bytes, generate, torch_dtype


def _small(name):
    w = WORKLOADS[name]
    return w.with_(batch=min(w.batch, 2), seqlen=min(w.seqlen, 512))


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_shapes_dtypes_and_reproducibility(name):
    w = _small(name)
    a, b = generate(w), generate(w)
    B, L, H, P, N, G = w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups
    io = torch_dtype(w.io_dtype)
    shapes = {"x": (B, L, H, P), "dt": (B, L, H), "A": (H,), "Bm": (B, L, G, N), "Cm": (B, L, G, N), "D": (H,)}
    for k, shp in shapes.items():
        assert tuple(a[k].shape) == shp, k
        assert a[k].is_contiguous(), k
        assert torch.equal(a[k], b[k]), k  # same seed, same draw
    for k in ("x", "Bm", "Cm"):
        assert a[k].dtype == io, k
    for k in ("dt", "A", "D"):
        assert a[k].dtype == torch.float32, k
    if w.has_init:
        assert tuple(a["init_state"].shape) == (B, H, P, N) and a["init_state"].dtype == torch.float32
        assert torch.equal(a["init_state"], b["init_state"])
    else:
        assert a["init_state"] is None
    # another seed draws other values
    c = generate(w, seed=w.seed + 1)
    assert not torch.equal(a["x"], c["x"])


def test_distributions_follow_the_recipe():
    w = WORKLOADS["mamba2_130m"].with_(batch=2, seqlen=2048)
    d = generate(w)
    x = d["x"].float()
    assert abs(x.mean().item()) < 0.01 and abs(x.std().item() - 1.0) < 0.01
    # dt = softplus(z - 1), z ~ N(0, 1): positive, with the mean of that law
    dt = d["dt"]
    assert (dt > 0).all()
    zs = torch.randn(2_000_000, generator=torch.Generator().manual_seed(5))
    assert abs(dt.mean().item() - torch.nn.functional.softplus(zs - 1.0).mean().item()) < 0.01
    # A_h = -exp(u), u ~ U(0, ln 16): in [-16, -1]
    A = d["A"]
    assert (A <= -1.0).all() and (A >= -16.0).all()
    # B, C ~ N(0, 1) / sqrt(N)
    for k in ("Bm", "Cm"):
        v = d[k].float()
        assert abs(v.std().item() * math.sqrt(w.dstate) - 1.0) < 0.02, k
    # long grouped: init_state ~ N(0, 0.1^2)
    lg = WORKLOADS["long_grouped"].with_(seqlen=64)
    init = generate(lg)["init_state"]
    assert abs(init.std().item() - 0.1) < 0.005


def test_bf16_rounding_is_the_only_change_of_io_tensors():
    """x, Bm, Cm are drawn in fp32 and rounded once: the bf16 workload's
    values are the fp32 draw of the same seed rounded to bf16."""
    w = WORKLOADS["mamba2_130m"].with_(batch=1, seqlen=128)
    d16 = generate(w)
    d32 = generate(w.with_(io_dtype="f32"))
    for k in ("x", "Bm", "Cm"):
        assert torch.equal(d16[k], d32[k].to(torch.bfloat16)), k
    for k in ("dt", "A", "D"):
        assert torch.equal(d16[k], d32[k]), k


def test_algorithmic_bytes_of_the_headline_layer():
    """x in + y out (bf16), dt in (fp32), Bm and Cm in (bf16), final_state
    out (fp32): 708.8 MB for B=4, L=8192, H=80, P=64, N=128, G=1."""
    w = WORKLOADS["mamba2_2p7b"]
    B, L, H, P, N, G = 4, 8192, 80, 64, 128, 1
    assert (w.batch, w.seqlen, w.nheads, w.headdim, w.dstate, w.ngroups) == (B, L, H, P, N, G)
    expect = B * L * H * P * 2 * 2 + B * L * H * 4 + B * L * G * N * 2 * 2 + B * H * P * N * 4
    assert algorithmic_bytes(w) == expect == 708_837_376
    # with an initial state its read is counted too
    lg = WORKLOADS["long_grouped"]
    assert algorithmic_bytes(lg) - algorithmic_bytes(lg.with_(has_init=False)) == lg.batch * lg.nheads * 64 * 128 * 4
