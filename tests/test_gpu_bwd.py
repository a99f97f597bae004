"""GPU parity of the backward pass (ssd_bwd) against the fp64 backward oracle
(oracle.ssd_recurrent_bwd, itself pinned by finite differences and autograd
in tests/test_oracle_bwd_pins.py).

Bar, normwise per gradient (‖got − ref‖∞ / ‖ref‖∞): fp32 io 1e-4, bf16 io
2e-2 -- the forward pass's bars.  Both sides see the same rounded inputs
(x, Bm, Cm and the cotangent dy in the io dtype).
"""
import pytest
import torch

import oracle
import ssd_scan_fwd_b300 as ssd
from ssd_scan_fwd_b300.inputs import WORKLOADS, Workload, generate, torch_dtype
from tests._util import TOL, normwise_err

pytestmark = pytest.mark.gpu

GRADS = ["dx", "ddt", "dA", "dBm", "dCm", "dD", "dinit"]


def _cotangents(w, seed, with_dfinal=True):
    g = torch.Generator().manual_seed(seed)
    dy = torch.randn(w.batch, w.seqlen, w.nheads, w.headdim, generator=g).to(torch_dtype(w.io_dtype))
    dfinal = torch.randn(w.batch, w.nheads, w.headdim, w.dstate, generator=g) if with_dfinal else None
    return dy.contiguous(), dfinal


def _gpu(inp, dy, dfinal, chunk_size=0):
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    out = ssd.ssd_bwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], d["init_state"],
                      dy=dy.cuda(), dfinal=None if dfinal is None else dfinal.cuda(), chunk_size=chunk_size)
    torch.cuda.synchronize()
    return out


def _ref(inp, dy, dfinal):
    return oracle.ssd_recurrent_bwd(inp["x"], inp["dt"], inp["A"], inp["Bm"], inp["Cm"], inp["D"],
                                    inp["init_state"], dy=dy, dfinal=dfinal)


def _compare(w, inp, got, ref, tol=None):
    tol = TOL[w.io_dtype] if tol is None else tol
    for k in GRADS:
        if got[k] is None:
            assert inp["D"] is None and k == "dD"
            continue
        err = normwise_err(got[k], ref[k])
        assert err <= tol, f"{k}: normwise error {err:.3e} > {tol}"


SMALL = [
    # name, overrides
    ("tiny_fp32", dict(batch=2, seqlen=150, nheads=4, ngroups=2, has_init=True)),
    ("tiny_fp32", dict(batch=1, seqlen=1, nheads=2)),
    ("tiny_fp32", dict(batch=1, seqlen=64, nheads=2, headdim=128, dstate=30)),
    ("tiny_fp32", dict(batch=1, seqlen=70, nheads=3, ngroups=3, headdim=8, dstate=256, has_init=True)),
    ("mamba2_130m", dict(batch=2, seqlen=200, nheads=4, ngroups=2, has_init=True)),
    ("mamba2_130m", dict(batch=1, seqlen=129, nheads=6)),
]


@pytest.mark.parametrize("name,over", SMALL, ids=[f"{n}-{o}" for n, o in SMALL])
def test_bwd_matches_oracle(name, over):
    w = WORKLOADS[name].with_(**over)
    i = SMALL.index((name, over))
    inp = generate(w, seed=7000 + i)
    dy, dfinal = _cotangents(w, 7100 + i)
    _compare(w, inp, _gpu(inp, dy, dfinal), _ref(inp, dy, dfinal))


@pytest.mark.parametrize("chunk", [64, 128])
@pytest.mark.parametrize("seqlen", [1, 127, 128, 300, 513])
def test_bwd_chunk_lengths(chunk, seqlen):
    """bf16, headdim 64, dstate 128: the CUDA-core gradient kernel (chunk 64)
    and the tensor-core one (chunk 128) on ragged and exact chunk tails, with
    groups, an initial state and every optional term."""
    w = WORKLOADS["mamba2_130m"].with_(batch=2, seqlen=seqlen, nheads=6, ngroups=2, has_init=True)
    inp = generate(w, seed=7600 + seqlen)
    dy, dfinal = _cotangents(w, 7700 + seqlen)
    _compare(w, inp, _gpu(inp, dy, dfinal, chunk_size=chunk), _ref(inp, dy, dfinal))


@pytest.mark.parametrize("name", ["nsweep_16", "nsweep_64", "nsweep_256"])
def test_bwd_state_sizes(name):
    """bf16 with dstate 16, 64 and 256: CUDA-core gradient kernel (chunk 64) with
    the tensor-core forward and adjoint chunk states."""
    w = WORKLOADS[name].with_(batch=2, seqlen=200, nheads=4, ngroups=2, has_init=True)
    inp = generate(w, seed=7900)
    dy, dfinal = _cotangents(w, 7901)
    _compare(w, inp, _gpu(inp, dy, dfinal), _ref(inp, dy, dfinal))


def test_bwd_tensor_core_strong_decay():
    """Fast decay (large Δ·|A|): e^{cs_s − cs_j} spans many orders inside a
    128-token chunk; the masks are formed from differences of the running sum,
    never from e^{cs} and e^{−cs} separately."""
    w = WORKLOADS["mamba2_130m"].with_(batch=1, seqlen=384, nheads=4, ngroups=1, has_init=True)
    inp = generate(w, seed=7800)
    inp["A"] = inp["A"] * 8.0
    dy, dfinal = _cotangents(w, 7801)
    _compare(w, inp, _gpu(inp, dy, dfinal, chunk_size=128), _ref(inp, dy, dfinal))


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_bwd_without_optional_terms(io):
    """No D, no initial state, no dfinal: dD is not written, dinit still is."""
    w = Workload(name="opt", batch=2, seqlen=97, nheads=4, headdim=16, dstate=32, ngroups=1, io_dtype=io,
                 has_init=False, seed=7200)
    inp = generate(w)
    inp["D"] = None
    dy, _ = _cotangents(w, 7201, with_dfinal=False)
    _compare(w, inp, _gpu(inp, dy, None), _ref(inp, dy, None))


def test_bwd_empty_sequence():
    """L = 0: final_state = init_state, so dinit = dfinal and dA = dD = 0."""
    w = WORKLOADS["tiny_fp32"].with_(seqlen=0, has_init=True)
    inp = generate(w)
    dy, dfinal = _cotangents(w, 7300)
    got = _gpu(inp, dy, dfinal)
    assert torch.equal(got["dinit"].cpu(), dfinal)
    assert torch.count_nonzero(got["dA"]) == 0 and torch.count_nonzero(got["dD"]) == 0


def test_bwd_full_130m():
    """The Mamba-2 130M-shaped layer (B=2, L=2048, H=24, P=64, N=128), every gradient."""
    w = WORKLOADS["mamba2_130m"]
    inp = generate(w)
    dy, dfinal = _cotangents(w, 7400)
    _compare(w, inp, _gpu(inp, dy, dfinal), _ref(inp, dy, dfinal))


def test_bwd_full_2p7b_sampled_heads():
    """The 2.7B-shaped layer: the per-head gradients (dx, ddt, dinit) and the
    per-head sums dA, dD of sampled heads against the oracle run on those
    heads alone (dBm/dCm are sums over all 80 heads; they are checked in full
    on the 130M shape)."""
    w = WORKLOADS["mamba2_2p7b"]
    inp = generate(w)
    dy, dfinal = _cotangents(w, 7500)
    got = _gpu(inp, dy, dfinal)
    for h in (0, 41, 79):
        sub = dict(inp, x=inp["x"][:, :, h:h + 1], dt=inp["dt"][:, :, h:h + 1], A=inp["A"][h:h + 1],
                   D=inp["D"][h:h + 1], init_state=None)
        ref = _ref(sub, dy[:, :, h:h + 1], dfinal[:, h:h + 1])
        for k, sl in (("dx", (slice(None), slice(None), slice(h, h + 1))),
                      ("ddt", (slice(None), slice(None), slice(h, h + 1))),
                      ("dinit", (slice(None), slice(h, h + 1)))):
            err = normwise_err(got[k][sl], ref[k])
            assert err <= TOL["bf16"], (h, k, err)
        for k in ("dA", "dD"):
            err = normwise_err(got[k][h:h + 1], ref[k])
            assert err <= TOL["bf16"], (h, k, err)
    for k in GRADS:
        assert torch.isfinite(got[k].float()).all(), k


def test_bwd_tensor_core_no_dfinal_no_init():
    """Tensor-core path (bf16, P=64, N=128, chunk 128) without init_state and
    dfinal: both state walks start from zero (dinit is still written); three
    heads per group (the last head pair has one head) and a ragged tail."""
    w = WORKLOADS["mamba2_130m"].with_(batch=2, seqlen=3 * 128 + 5, nheads=6, ngroups=2, has_init=False)
    inp = generate(w, seed=7600)
    dy, _ = _cotangents(w, 7601, with_dfinal=False)
    _compare(w, inp, _gpu(inp, dy, None, chunk_size=128), _ref(inp, dy, None))


def test_bwd_tensor_core_many_walks():
    """More head-pair sequences than SMs (2 · 4 · 40 = 320 state walks on at
    most 148 CTAs, some taking three), every gradient against the oracle."""
    w = WORKLOADS["mamba2_2p7b"].with_(batch=4, seqlen=2 * 128 + 33, nheads=80, ngroups=1, has_init=True)
    inp = generate(w, seed=7700)
    dy, dfinal = _cotangents(w, 7701)
    _compare(w, inp, _gpu(inp, dy, dfinal), _ref(inp, dy, dfinal))
