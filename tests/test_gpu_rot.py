"""GPU parity of the complex-decay forward pass (ssd_fwd_rot) against the
fp64 oracle (oracle.ssd_recurrent_rot, pinned in test_oracle_rot_pins.py).

Bar (normwise, separately for y and both parts of the final state): fp32 io
1e-4, bf16 io 2e-2.
"""
import numpy as np
import pytest
import torch

import oracle
import ssd_scan_fwd_b300 as ssd
from ssd_scan_fwd_b300.inputs import WORKLOADS, generate
from tests._util import TOL, normwise_err

pytestmark = pytest.mark.gpu


def _theta(w, seed, scale=np.pi):
    g = torch.Generator().manual_seed(seed)
    return ((torch.rand(w.batch, w.seqlen, w.nheads, generator=g) * 2 - 1) * scale).contiguous()


def _init_im(w, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(w.batch, w.nheads, w.headdim, w.dstate, generator=g) * 0.1).contiguous()


def _gpu(inp, theta, init_im=None, chunk=0, algo="auto"):
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    init = None
    if d["init_state"] is not None or init_im is not None:
        init = (d["init_state"], None if init_im is None else init_im.cuda())
    y, (fr, fi) = ssd.ssd_fwd_rot(d["x"], d["dt"], theta.cuda(), d["A"], d["Bm"], d["Cm"], d["D"], init,
                                  chunk_size=chunk, algo=algo)
    torch.cuda.synchronize()
    return y, fr, fi


def _ref(inp, theta, init_im=None):
    h0 = None
    if inp["init_state"] is not None or init_im is not None:
        re = inp["init_state"] if inp["init_state"] is not None else torch.zeros_like(init_im)
        im = init_im if init_im is not None else torch.zeros_like(re)
        h0 = (re, im)
    return oracle.ssd_recurrent_rot(inp["x"], inp["dt"], theta, inp["A"], inp["Bm"], inp["Cm"], inp["D"], h0)


CASES = [
    ("tiny_fp32", dict(batch=2, seqlen=150, nheads=4, ngroups=2, has_init=True), 32),
    ("tiny_fp32", dict(batch=1, seqlen=257, nheads=3), 64),
    ("tiny_fp32", dict(batch=2, seqlen=300, nheads=2, headdim=32, dstate=48, has_init=True), 128),
    ("mamba2_130m", dict(batch=2, seqlen=200, nheads=4, ngroups=2, has_init=True), 0),
    ("mamba2_130m", dict(batch=1, seqlen=129, nheads=6), 0),
    # bf16 (64, 128): chunk 128 (tensor-core chunk outputs) and 64 (CUDA cores), ragged and exact tails
    ("mamba2_130m", dict(batch=2, seqlen=300, nheads=4, ngroups=2, has_init=True), 128),
    ("mamba2_130m", dict(batch=1, seqlen=256, nheads=3, has_init=True), 128),
    ("mamba2_130m", dict(batch=1, seqlen=385, nheads=3), 64),
    # dstate 64 and 256: tensor-core chunk states and outputs at the default chunk (128)
    ("nsweep_64", dict(batch=2, seqlen=300, nheads=4, ngroups=2, has_init=True), 0),
    ("nsweep_256", dict(batch=1, seqlen=200, nheads=3, has_init=True), 0),
    ("nsweep_16", dict(batch=2, seqlen=260, nheads=4, ngroups=2, has_init=True), 0),
]


@pytest.mark.parametrize("algo", ["auto", "chunked"])
@pytest.mark.parametrize("name,over,chunk", CASES, ids=[f"{n}-{o}-Q{q}" for n, o, q in CASES])
def test_rot_matches_oracle(name, over, chunk, algo):
    """auto: the fused kernel for the bf16 dstate-128 cases at chunk 0 / 128,
    the chunked path for the rest; chunked: the chunked path for all."""
    w = WORKLOADS[name].with_(**over)
    i = CASES.index((name, over, chunk))
    inp = generate(w, seed=8000 + i)
    theta = _theta(w, 8100 + i)
    init_im = _init_im(w, 8200 + i) if w.has_init else None
    y, fr, fi = _gpu(inp, theta, init_im, chunk, algo)
    ry, (rr, ri) = _ref(inp, theta, init_im)
    tol = TOL[w.io_dtype]
    assert normwise_err(y, ry) <= tol
    assert normwise_err(fr, rr) <= tol
    assert normwise_err(fi, ri) <= tol


def test_rot_zero_angle_matches_ssd_fwd():
    w = WORKLOADS["tiny_fp32"].with_(batch=2, seqlen=200, nheads=4, has_init=True)
    inp = generate(w, seed=8300)
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    y0, f0 = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], d["init_state"], algo="chunked")
    y1, fr, fi = _gpu(inp, torch.zeros(w.batch, w.seqlen, w.nheads))
    assert normwise_err(y1, y0.double().cpu().numpy()) <= 1e-6
    assert normwise_err(fr, f0.double().cpu().numpy()) <= 1e-6
    assert torch.count_nonzero(fi) == 0


def test_rot_parity_task():
    """The parity example of the Foundations page: B = 0, A = 0, h0 = 1,
    θ_t = π·bit_t, C = 1, D = 0 gives y_t = (−1)^(bits so far)."""
    L = 300
    bits = torch.randint(0, 2, (L,), generator=torch.Generator().manual_seed(8400)).float()
    x = torch.zeros(1, L, 1, 1, device="cuda")
    dt = torch.ones(1, L, 1, device="cuda")
    A = torch.zeros(1, device="cuda")
    Bm = torch.zeros(1, L, 1, 1, device="cuda")
    Cm = torch.ones(1, L, 1, 1, device="cuda")
    h0 = torch.ones(1, 1, 1, 1, device="cuda")
    y, _ = ssd.ssd_fwd_rot(x, dt, (np.pi * bits).view(1, L, 1).cuda(), A, Bm, Cm, None, (h0, None))
    torch.cuda.synchronize()
    expect = (-1.0) ** torch.cumsum(bits, 0)
    assert torch.allclose(y.view(-1).cpu(), expect, atol=1e-4)


def test_rot_empty_sequence():
    w = WORKLOADS["tiny_fp32"].with_(seqlen=0, has_init=True)
    inp = generate(w)
    init_im = _init_im(w, 8500)
    y, fr, fi = _gpu(inp, torch.zeros(w.batch, 0, w.nheads), init_im)
    assert torch.equal(fr.cpu(), inp["init_state"]) and torch.equal(fi.cpu(), init_im)


def test_rot_full_130m_sampled():
    """The 130M-shaped layer (B=2, L=2048, H=24, bf16) with random angles,
    sampled heads against the oracle run on those heads alone."""
    w = WORKLOADS["mamba2_130m"]
    inp = generate(w)
    theta = _theta(w, 8600, scale=0.5)
    y, fr, fi = _gpu(inp, theta)
    for b, h in [(0, 0), (1, 13), (1, 23)]:
        sub = dict(x=inp["x"][b:b + 1, :, h:h + 1], dt=inp["dt"][b:b + 1, :, h:h + 1], A=inp["A"][h:h + 1],
                   Bm=inp["Bm"][b:b + 1], Cm=inp["Cm"][b:b + 1], D=inp["D"][h:h + 1], init_state=None)
        ry, (rr, ri) = _ref(sub, theta[b:b + 1, :, h:h + 1])
        assert normwise_err(y[b:b + 1, :, h:h + 1], ry) <= TOL["bf16"], (b, h)
        assert normwise_err(fr[b:b + 1, h:h + 1], rr) <= TOL["bf16"], (b, h)
        assert normwise_err(fi[b:b + 1, h:h + 1], ri) <= TOL["bf16"], (b, h)


# --------------------------------------------------------------------------
# The fused kernel with the complex decay (one head per CTA, Re / Im of the
# state in the places of the two heads): several chunks and a ragged tail,
# grouped heads, with and without init; hand-offs of the complex state
# between CTAs (contiguous ranges) and between segments.
# --------------------------------------------------------------------------
FUSED = [
    dict(batch=2, seqlen=5 * 128 + 37, nheads=4, ngroups=2, has_init=True),
    dict(batch=1, seqlen=300, nheads=3),
    dict(batch=1, seqlen=128, nheads=2, has_init=True),
]


@pytest.mark.parametrize("scale", [0.5, np.pi])
@pytest.mark.parametrize("over", FUSED, ids=[str(f) for f in FUSED])
def test_rot_fused_vs_oracle(over, scale):
    w = WORKLOADS["mamba2_2p7b"].with_(**over)
    seed = 8700 + FUSED.index(over)
    inp = generate(w, seed=seed)
    theta = _theta(w, seed + 50, scale)
    init_im = _init_im(w, seed + 60) if w.has_init else None
    y, fr, fi = _gpu(inp, theta, init_im, algo="fused")
    ry, (rr, ri) = _ref(inp, theta, init_im)
    assert normwise_err(y, ry) <= TOL["bf16"]
    assert normwise_err(fr, rr) <= TOL["bf16"]
    assert normwise_err(fi, ri) <= TOL["bf16"]


@pytest.mark.parametrize("knob,value", [("SSD_FUSED_GRID", "1"), ("SSD_FUSED_GRID", "3"), ("SSD_FUSED_GRID", "5"),
                                        ("SSD_FUSED_NSEG", "3")])
def test_rot_fused_handoffs(knob, value, monkeypatch):
    """Contiguous ranges (complex states handed between CTAs) and forced
    segments (published through the workspace)."""
    monkeypatch.setenv(knob, value)
    w = WORKLOADS["mamba2_2p7b"].with_(batch=2, seqlen=5 * 128 + 37, nheads=6, ngroups=2, has_init=True)
    inp = generate(w, seed=8800)
    theta = _theta(w, 8801, 0.5)
    init_im = _init_im(w, 8802)
    y, fr, fi = _gpu(inp, theta, init_im, algo="fused")
    ry, (rr, ri) = _ref(inp, theta, init_im)
    assert normwise_err(y, ry) <= TOL["bf16"]
    assert normwise_err(fr, rr) <= TOL["bf16"]
    assert normwise_err(fi, ri) <= TOL["bf16"]


def test_rot_fused_matches_chunked_and_real():
    """The fused and the chunked complex-decay paths agree; at θ = 0 the fused
    complex-decay kernel gives the real forward pass and a zero Im part."""
    w = WORKLOADS["mamba2_2p7b"].with_(batch=2, seqlen=640, nheads=4, has_init=True)
    inp = generate(w, seed=8900)
    theta = _theta(w, 8901, 0.5)
    init_im = _init_im(w, 8902)
    y1, r1, i1 = _gpu(inp, theta, init_im, algo="fused")
    y2, r2, i2 = _gpu(inp, theta, init_im, algo="chunked")
    assert normwise_err(y1, y2) < 1e-2 and normwise_err(r1, r2) < 1e-2 and normwise_err(i1, i2) < 1e-2
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    y0, f0 = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], d["init_state"], algo="fused")
    yz, rz, iz = _gpu(inp, torch.zeros(w.batch, w.seqlen, w.nheads), None, algo="fused")
    assert normwise_err(yz, y0) < 1e-2 and normwise_err(rz, f0) < 1e-2
    assert torch.count_nonzero(iz) == 0


def test_rot_fused_full_2p7b():
    """The 2.7B-shaped layer on the fused kernel, every element of y and of
    both parts of the final state against the oracle, one batch row at a time."""
    w = WORKLOADS["mamba2_2p7b"]
    inp = generate(w)
    theta = _theta(w, 9000, 0.5)
    y, fr, fi = _gpu(inp, theta, algo="fused")
    ey = er = ei = 0.0
    sy = sr = si = 0.0
    for b in range(w.batch):
        sub = {k: (None if v is None else (v[b:b + 1] if v.dim() > 1 else v)) for k, v in inp.items()}
        ry, (rr, ri) = _ref(sub, theta[b:b + 1])
        yb = y[b:b + 1].double().cpu().numpy()
        ey = max(ey, float(np.max(np.abs(yb - ry))))
        sy = max(sy, float(np.max(np.abs(ry))))
        er = max(er, float(np.max(np.abs(fr[b:b + 1].double().cpu().numpy() - rr))))
        sr = max(sr, float(np.max(np.abs(rr))))
        ei = max(ei, float(np.max(np.abs(fi[b:b + 1].double().cpu().numpy() - ri))))
        si = max(si, float(np.max(np.abs(ri))))
    assert ey / sy <= TOL["bf16"] and er / sr <= TOL["bf16"] and ei / si <= TOL["bf16"]
