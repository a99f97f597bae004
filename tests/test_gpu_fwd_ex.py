"""GPU parity of ssd_fwd_ex (Δ = softplus(dt + dt_bias), gate y · silu(z))
against the fp64 oracle, on both paths.

Bar (normwise, separately for y and final_state): fp32 io 1e-4, bf16 io 2e-2.
"""
import pytest
import torch

import oracle
import ssd_scan_fwd_b300 as ssd
from ssd_scan_fwd_b300.inputs import WORKLOADS, generate, torch_dtype
from tests._util import TOL, normwise_err, poison_like, rowwise_normwise_err, to_device

pytestmark = pytest.mark.gpu


def _extras(w, seed, softplus=True):
    """Raw dt (so that softplus(dt + bias) has the workload's Δ distribution),
    a per-head bias and the gate input z, all seeded."""
    g = torch.Generator().manual_seed(seed)
    B, L, H, P = w.batch, w.seqlen, w.nheads, w.headdim
    bias = torch.rand(H, generator=g) * 0.5
    if softplus:
        raw = torch.randn(B, L, H, generator=g) - 1.0 - bias[None, None, :]
    else:
        raw = torch.nn.functional.softplus(torch.randn(B, L, H, generator=g) - 1.0)
    z = torch.randn(B, L, H, P, generator=g).to(torch_dtype(w.io_dtype))
    return raw.contiguous(), bias.contiguous(), z.contiguous()


def _compare(w, inp, raw, bias, z, softplus, algo, with_bias=True, with_z=True, chunk=0):
    d = to_device(inp)
    y = poison_like(d["x"])
    fs = torch.full((w.batch, w.nheads, w.headdim, w.dstate), float("nan"), device="cuda")
    ssd.ssd_fwd_ex(d["x"], raw.cuda(), d["A"], d["Bm"], d["Cm"], d["D"], d["init_state"],
                   dt_bias=bias.cuda() if with_bias else None, dt_softplus=softplus,
                   z=z.cuda() if with_z else None, algo=algo, y=y, final_state=fs, chunk_size=chunk)
    torch.cuda.synchronize()
    y_ref, h_ref = oracle.ssd_fwd_ex(inp["x"], raw, inp["A"], inp["Bm"], inp["Cm"], inp["D"], inp["init_state"],
                                     dt_bias=bias if with_bias else None, dt_softplus=softplus,
                                     z=z if with_z else None)
    tol = TOL[w.io_dtype]
    assert normwise_err(y, y_ref) <= tol
    assert normwise_err(fs, h_ref) <= tol


@pytest.mark.parametrize("algo", ["chunked", "fused"])
@pytest.mark.parametrize("softplus", [True, False])
def test_fwd_ex_bf16(algo, softplus):
    w = WORKLOADS["mamba2_2p7b"].with_(batch=2, seqlen=700, nheads=6, ngroups=2, has_init=True)
    inp = generate(w, seed=31)
    raw, bias, z = _extras(w, 6100, softplus)
    _compare(w, inp, raw, bias, z, softplus, algo)


@pytest.mark.parametrize("with_z", [True, False])
def test_fwd_ex_chunked_tensor_core_scan(with_z):
    """Chunk 128 on the bf16 (64, 128) shape: the chunk outputs come from the
    tensor-core kernel, with and without the gate."""
    w = WORKLOADS["mamba2_2p7b"].with_(batch=2, seqlen=333, nheads=4, ngroups=2, has_init=True)
    inp = generate(w, seed=33)
    raw, bias, z = _extras(w, 6102, True)
    _compare(w, inp, raw, bias, z, True, "chunked", with_z=with_z, chunk=128)


def test_fwd_ex_fp32_chunked():
    w = WORKLOADS["tiny_fp32"].with_(seqlen=300, nheads=3, has_init=True)
    inp = generate(w, seed=32)
    raw, bias, z = _extras(w, 6101, True)
    _compare(w, inp, raw, bias, z, True, "chunked")


@pytest.mark.parametrize("algo", ["chunked", "fused"])
def test_fwd_ex_gate_only_and_bias_only(algo):
    w = WORKLOADS["mamba2_130m"].with_(batch=1, seqlen=513, nheads=4)
    inp = generate(w, seed=33)
    raw, bias, z = _extras(w, 6102, False)
    _compare(w, inp, raw, bias, z, False, algo, with_bias=False, with_z=True)
    _compare(w, inp, raw, bias, z, False, algo, with_bias=True, with_z=False)


def test_fwd_ex_without_options_equals_fwd():
    w = WORKLOADS["mamba2_130m"].with_(batch=1, seqlen=300, nheads=4)
    d = to_device(generate(w, seed=34))
    y0, f0 = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"])
    y1, f1 = ssd.ssd_fwd_ex(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"])
    torch.cuda.synchronize()
    assert torch.equal(y0, y1) and torch.equal(f0, f1)


def test_fwd_ex_full_size_whole():
    """The 2.7B-shaped layer through the fused path with both options (Δ =
    softplus(dt + dt_bias), gate silu(z)): every element of y and final_state
    against the oracle, run one batch row at a time."""
    w = WORKLOADS["mamba2_2p7b"]
    inp = generate(w, seed=35)
    raw, bias, z = _extras(w, 6103, True)
    d = to_device(inp)
    y, fs = ssd.ssd_fwd_ex(d["x"], raw.cuda(), d["A"], d["Bm"], d["Cm"], d["D"], dt_bias=bias.cuda(),
                           dt_softplus=True, z=z.cuda(), algo="fused")
    torch.cuda.synchronize()
    del d

    def ref_row(b):
        r = slice(b, b + 1)
        yr, fr = oracle.ssd_fwd_ex(inp["x"][r], raw[r], inp["A"], inp["Bm"][r], inp["Cm"][r], inp["D"], None,
                                   dt_bias=bias, dt_softplus=True, z=z[r])
        return yr[0], fr[0]

    ey, ef = rowwise_normwise_err(y, fs, ref_row, w.batch)
    assert ey <= TOL["bf16"], ey
    assert ef <= TOL["bf16"], ef


@pytest.mark.parametrize("dstate", [16, 64, 256])
def test_fwd_ex_fused_small_states(dstate):
    w = WORKLOADS["mamba2_2p7b"].with_(batch=2, seqlen=700, nheads=6, ngroups=2, has_init=True, dstate=dstate)
    inp = generate(w, seed=31 + dstate)
    raw, bias, z = _extras(w, 6200 + dstate, True)
    _compare(w, inp, raw, bias, z, True, "fused")


def test_fwd_ex_gate_wide_z_elementwise():
    """The gate's arithmetic alone, element by element, over z ∈ [−24, 24]
    (both signs far into the tails): the gated output of the fused kernel
    against its own ungated output times silu(z) in fp64.  The two runs share
    the pre-gate y; what differs is silu and one more bf16 rounding.  Bound:
    two bf16 roundings of the product plus the silu approximation's absolute
    error |z| 2^-12 times |y|."""
    w = WORKLOADS["mamba2_2p7b"].with_(batch=1, seqlen=3 * 128 + 17, nheads=4, ngroups=1, has_init=True)
    d = to_device(generate(w, seed=35))
    g = torch.Generator().manual_seed(6103)
    z = ((torch.rand(w.batch, w.seqlen, w.nheads, w.headdim, generator=g) * 2 - 1) * 24).to(torch.bfloat16)
    y0, _ = ssd.ssd_fwd_ex(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], d["init_state"], algo="fused")
    y1, _ = ssd.ssd_fwd_ex(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], d["init_state"], z=z.cuda(),
                           algo="fused")
    torch.cuda.synchronize()
    zz = z.double()
    ref = y0.cpu().double() * zz * torch.sigmoid(zz)
    err = (y1.cpu().double() - ref).abs()
    bound = 2.0 ** -7 * ref.abs() + 2.0 ** -12 * zz.abs() * y0.cpu().double().abs() * 1.01 + 1e-30
    assert bool((err <= bound).all()), f"worst excess {(err - bound).max().item():.3e}"


def test_fwd_ex_softplus_wide_dt():
    """Δ pre-processing over raw dt + dt_bias spread across [−30, 30]: Δ from
    about 1e-13 (e^v for very negative v, where log1p carries the relative
    accuracy) to 30 (softplus(v) = v), with a ragged tail, on the fused path."""
    w = WORKLOADS["mamba2_2p7b"].with_(batch=2, seqlen=2 * 128 + 45, nheads=4, ngroups=2, has_init=True)
    inp = generate(w, seed=36)
    g = torch.Generator().manual_seed(6104)
    raw = ((torch.rand(w.batch, w.seqlen, w.nheads, generator=g) * 2 - 1) * 30).contiguous()
    bias = (torch.rand(w.nheads, generator=g) * 0.5).contiguous()
    z = torch.randn(w.batch, w.seqlen, w.nheads, w.headdim, generator=g).to(torch.bfloat16).contiguous()
    _compare(w, inp, raw, bias, z, True, "fused")
