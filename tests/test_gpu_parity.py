"""GPU parity: the CUDA library against the fp64 oracle on seeded inputs.

Bar (normwise ‖out − ref‖∞ / ‖ref‖∞, for y and final_state separately):
fp32 io 1e-4, bf16 io 2e-2.  Outputs are pre-filled with NaN so that any
element a kernel leaves unwritten fails.
"""
import pytest
import torch

import oracle
import ssd_scan_fwd_b300 as ssd
from ssd_scan_fwd_b300.inputs import WORKLOADS, generate
from tests._util import TOL, normwise_err, poison_like, rowwise_normwise_err, to_device

pytestmark = pytest.mark.gpu


def _run(inp_dev, algo="auto", chunk=0, with_final=True):
    x = inp_dev["x"]
    B, L, H, P = x.shape
    N = inp_dev["Bm"].shape[3]
    y = poison_like(x)
    fs = torch.full((B, H, P, N), float("nan"), device=x.device) if with_final else None
    y, fs = ssd.ssd_fwd(inp_dev["x"], inp_dev["dt"], inp_dev["A"], inp_dev["Bm"], inp_dev["Cm"],
                        inp_dev["D"], inp_dev["init_state"], return_final_state=with_final,
                        algo=algo, chunk_size=chunk, y=y, final_state=fs)
    torch.cuda.synchronize()
    return y, fs


def _oracle(inp):
    return oracle.ssd_recurrent(inp["x"], inp["dt"], inp["A"], inp["Bm"], inp["Cm"], inp["D"],
                                inp["init_state"])


def _check(inp, y, fs, io):
    ry, rf = _oracle(inp)
    ey, ef = normwise_err(y, ry), normwise_err(fs, rf)
    assert ey <= TOL[io], f"y normwise error {ey:.3e} > {TOL[io]}"
    assert ef <= TOL[io], f"final_state normwise error {ef:.3e} > {TOL[io]}"
    return ey, ef


# --------------------------------------------------------------------------
# Whole forward pass, small sizes the oracle finishes in seconds, spanning
# several chunks and a ragged tail.
# --------------------------------------------------------------------------
SMALL = [
    # name, overrides
    ("tiny_fp32", {}),
    ("mamba2_130m", dict(batch=1, seqlen=333)),
    ("mamba2_2p7b", dict(batch=1, seqlen=300, nheads=8)),
    ("long_grouped", dict(seqlen=517, nheads=16)),
    ("nsweep_16", dict(batch=2, seqlen=260, nheads=4)),
    ("nsweep_64", dict(batch=2, seqlen=260, nheads=4)),
    ("nsweep_128", dict(batch=2, seqlen=260, nheads=4)),
    ("nsweep_256", dict(batch=2, seqlen=260, nheads=4)),
]


@pytest.mark.parametrize("algo", ["chunked", "auto"])
@pytest.mark.parametrize("name,over", SMALL, ids=[s[0] for s in SMALL])
def test_forward_small(name, over, algo):
    w = WORKLOADS[name].with_(**over)
    inp = generate(w)
    y, fs = _run(to_device(inp), algo=algo)
    _check(inp, y, fs, w.io_dtype)


@pytest.mark.parametrize("chunk", [32, 64, 128])
def test_forward_chunk_sizes(chunk):
    w = WORKLOADS["mamba2_130m"].with_(batch=2, seqlen=300, nheads=4)
    inp = generate(w)
    y, fs = _run(to_device(inp), algo="chunked", chunk=chunk)
    _check(inp, y, fs, "bf16")


@pytest.mark.parametrize("chunk", [0, 64, 128])
@pytest.mark.parametrize("name", ["nsweep_16", "nsweep_64", "nsweep_256"])
def test_forward_state_sizes_chunked(name, chunk):
    """dstate 16, 64 and 256 (bf16, headdim 64): tensor-core chunk states at
    chunk 64 and 128, tensor-core chunk outputs at 128 (also the default, 0),
    with groups, an initial state and a ragged last chunk."""
    w = WORKLOADS[name].with_(batch=2, seqlen=333, nheads=4, ngroups=2, has_init=True)
    inp = generate(w, seed=91)
    y, fs = _run(to_device(inp), algo="chunked", chunk=chunk)
    _check(inp, y, fs, "bf16")


@pytest.mark.parametrize("chunk", [32, 64, 128])
def test_forward_fp32_tight(chunk):
    w = WORKLOADS["tiny_fp32"].with_(seqlen=250, nheads=3, has_init=True)
    inp = generate(w, seed=77)
    y, fs = _run(to_device(inp), algo="chunked", chunk=chunk)
    _check(inp, y, fs, "f32")


# --------------------------------------------------------------------------
# Each step of the chunked path against the oracle's chunked intermediates.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("chunk", [32, 64, 128])
@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_steps_vs_oracle_chunked(chunk, io):
    w = WORKLOADS["tiny_fp32"].with_(batch=2, seqlen=3 * chunk + 5, nheads=4, ngroups=2,
                                     headdim=24, dstate=40, io_dtype=io, has_init=True)
    inp = generate(w, seed=5)
    d = to_device(inp)
    ref = oracle.ssd_chunked(inp["x"], inp["dt"], inp["A"], inp["Bm"], inp["Cm"], inp["D"],
                             inp["init_state"], chunk=chunk)
    args = (d["x"], d["dt"], d["A"], d["Bm"], d["Cm"])
    dA, dtc = ssd.chunk_cumsum(*args, chunk)
    st = ssd.chunk_state(*args, dA, dtc, chunk)
    torch.cuda.synchronize()
    tol = TOL[io]
    assert normwise_err(dA, ref["dA_cs"]) < 1e-6
    assert normwise_err(st, ref["chunk_states"]) < tol
    final = torch.full_like(d["init_state"], float("nan"))
    ssd.state_passing(*args, dA, st, chunk, init_state=d["init_state"], final_state=final)
    torch.cuda.synchronize()
    assert normwise_err(st, ref["states_in"]) < tol
    assert normwise_err(final, ref["final_state"]) < tol
    y = ssd.chunk_scan(*args, d["D"], dA, dtc, st, chunk, y=poison_like(d["x"]))
    torch.cuda.synchronize()
    assert normwise_err(y, ref["y"]) < tol


# --------------------------------------------------------------------------
# Edge shapes: ragged tails, single token, B=1, H=G, odd sizes.
# --------------------------------------------------------------------------
EDGE = [
    dict(seqlen=1),
    dict(seqlen=63),
    dict(seqlen=65),
    dict(seqlen=3 * 64 + 5),
    dict(seqlen=129, nheads=3, ngroups=3),
    dict(seqlen=100, nheads=24, ngroups=1),
    dict(seqlen=100, nheads=80, ngroups=1, headdim=8, dstate=8),
    dict(seqlen=77, headdim=17, dstate=24),
    dict(seqlen=77, headdim=130, dstate=200),
]


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("over", EDGE, ids=[str(e) for e in EDGE])
def test_edge_shapes(over, io):
    w = WORKLOADS["tiny_fp32"].with_(io_dtype=io, has_init=True, **over)
    inp = generate(w, seed=11)
    y, fs = _run(to_device(inp))
    _check(inp, y, fs, io)


def test_no_skip_no_init_no_final():
    w = WORKLOADS["mamba2_130m"].with_(batch=1, seqlen=200, nheads=4)
    inp = generate(w)
    inp["D"] = None
    d = to_device(inp)
    y, fs = _run(d, with_final=False)
    assert fs is None
    ry, _ = _oracle(inp)
    assert normwise_err(y, ry) <= TOL["bf16"]


def test_empty_sequence_returns_initial_state():
    w = WORKLOADS["tiny_fp32"].with_(seqlen=0, has_init=True)
    inp = generate(w)
    d = to_device(inp)
    y, fs = _run(d)
    assert y.numel() == 0
    assert torch.equal(fs, d["init_state"])
    d["init_state"] = None
    _, fs = _run(d)
    assert torch.count_nonzero(fs) == 0


def test_in_place_state_update():
    w = WORKLOADS["tiny_fp32"].with_(seqlen=150, has_init=True)
    inp = generate(w, seed=3)
    d = to_device(inp)
    st = d["init_state"].clone()
    y = poison_like(d["x"])
    ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], st, y=y, final_state=st)
    torch.cuda.synchronize()
    _check(inp, y, st, "f32")


# --------------------------------------------------------------------------
# Split / resume through the state, and group expansion.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("algo", ["chunked", "auto"])
def test_split_resume(algo):
    w = WORKLOADS["mamba2_2p7b"].with_(batch=2, seqlen=700, nheads=4, has_init=True)
    d = to_device(generate(w, seed=21))
    y_full, f_full = _run(d, algo=algo)
    cut = 300
    a = {k: (v[:, :cut].contiguous() if k in ("x", "dt", "Bm", "Cm") else v) for k, v in d.items()}
    b = {k: (v[:, cut:].contiguous() if k in ("x", "dt", "Bm", "Cm") else v) for k, v in d.items()}
    ya, fa = _run(a, algo=algo)
    b["init_state"] = fa
    yb, fb = _run(b, algo=algo)
    assert normwise_err(torch.cat([ya, yb], 1), y_full) < 1e-2
    assert normwise_err(fb, f_full) < 1e-3


def test_group_expansion_gpu():
    w = WORKLOADS["long_grouped"].with_(seqlen=300, nheads=8, ngroups=4)
    d = to_device(generate(w, seed=9))
    y1, f1 = _run(d)
    e = dict(d)
    e["Bm"] = d["Bm"].repeat_interleave(2, dim=2).contiguous()
    e["Cm"] = d["Cm"].repeat_interleave(2, dim=2).contiguous()
    y2, f2 = _run(e)
    assert normwise_err(y1, y2) < 1e-6 and normwise_err(f1, f2) < 1e-6


def test_bad_call_raises_without_launch():
    w = WORKLOADS["mamba2_130m"].with_(batch=1, seqlen=64, nheads=4)
    d = to_device(generate(w))
    with pytest.raises(ssd.SsdError):
        ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], chunk_size=48)
    # the context is still usable afterwards
    y, _ = _run(d)
    assert torch.isfinite(y.float()).all()


# --------------------------------------------------------------------------
# Full-size workloads in the benchmark's launch configuration: every element
# of y and final_state against the oracle's recurrence (run one batch row at
# a time to bound host memory), so every head, every chunk and every place
# where the schedule hands a sequence from one CTA to the next is checked.
# --------------------------------------------------------------------------
FULL = ["mamba2_130m", "mamba2_2p7b", "long_grouped", "nsweep_16", "nsweep_64", "nsweep_128",
        "nsweep_256"]


def _oracle_row(inp, b):
    r = slice(b, b + 1)
    y, f = oracle.ssd_recurrent(inp["x"][r], inp["dt"][r], inp["A"], inp["Bm"][r], inp["Cm"][r], inp["D"],
                                None if inp["init_state"] is None else inp["init_state"][r])
    return y[0], f[0]


@pytest.mark.parametrize("name", FULL)
def test_full_size_whole(name):
    w = WORKLOADS[name]
    inp = generate(w)
    y, fs = _run(to_device(inp))
    ey, ef = rowwise_normwise_err(y, fs, lambda b: _oracle_row(inp, b), w.batch)
    assert ey <= TOL[w.io_dtype], (name, "y", ey)
    assert ef <= TOL[w.io_dtype], (name, "final_state", ef)


# --------------------------------------------------------------------------
# The fused tensor-core kernel (bf16, P = 64, N = 128): ragged lengths,
# batch/head counts, groups, optional D / init / final state.
# --------------------------------------------------------------------------
FUSED = [
    dict(batch=1, seqlen=1, nheads=1),
    dict(batch=1, seqlen=128, nheads=2),
    dict(batch=1, seqlen=127, nheads=2),
    dict(batch=2, seqlen=129, nheads=3),
    dict(batch=3, seqlen=3 * 128 + 5, nheads=4, ngroups=2),
    dict(batch=1, seqlen=517, nheads=8, ngroups=8),
    dict(batch=2, seqlen=1000, nheads=160, ngroups=1),
]


@pytest.mark.parametrize("init", [False, True])
@pytest.mark.parametrize("over", FUSED, ids=[str(f) for f in FUSED])
def test_fused_vs_oracle(over, init):
    w = WORKLOADS["mamba2_2p7b"].with_(has_init=init, **over)
    inp = generate(w, seed=31)
    y, fs = _run(to_device(inp), algo="fused")
    _check(inp, y, fs, "bf16")


def test_fused_matches_chunked_closely():
    w = WORKLOADS["mamba2_2p7b"].with_(batch=2, seqlen=640, nheads=6, has_init=True)
    d = to_device(generate(w, seed=41))
    y1, f1 = _run(d, algo="fused")
    y2, f2 = _run(d, algo="chunked")
    assert normwise_err(y1, y2) < 1e-2 and normwise_err(f1, f2) < 1e-2


def test_fused_no_d_no_final():
    w = WORKLOADS["mamba2_2p7b"].with_(batch=1, seqlen=300, nheads=4)
    inp = generate(w, seed=4)
    inp["D"] = None
    y, fs = _run(to_device(inp), algo="fused", with_final=False)
    ry, _ = _oracle(inp)
    assert fs is None and normwise_err(y, ry) <= TOL["bf16"]


# --------------------------------------------------------------------------
# Contiguous chunk ranges per CTA (at least as many head-pair sequences as
# CTAs): the CTA count is capped so that small problems cut sequences at
# every kind of place -- whole sequences only, one CTA for everything, a
# sequence split once, ranges shorter and longer than a sequence.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("grid", [1, 3, 5, 7, 8])
def test_fused_ranges(grid, monkeypatch):
    monkeypatch.setenv("SSD_FUSED_GRID", str(grid))
    # 2 batch rows x 2 groups x 2 head pairs (the second pair of a group has
    # one real head) = 8 sequences of 6 chunks, the last one ragged
    w = WORKLOADS["mamba2_2p7b"].with_(batch=2, seqlen=5 * 128 + 37, nheads=6, ngroups=2, has_init=True)
    inp = generate(w, seed=100 + grid)
    y, fs = _run(to_device(inp), algo="fused")
    _check(inp, y, fs, "bf16")


# --------------------------------------------------------------------------
# Sequence segments of the fused kernel: forced segment counts (the hand-off
# of the state between segments through the workspace), ragged splits.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("nseg", [2, 3, 5, 64])
@pytest.mark.parametrize("two_pass", ["0", "1"])
def test_fused_segments(nseg, two_pass, monkeypatch):
    """Segments chained through the workspace flags (two_pass 0) or computed
    first and combined (two_pass 1: fewer sequences than SMs)."""
    monkeypatch.setenv("SSD_FUSED_NSEG", str(nseg))
    monkeypatch.setenv("SSD_FUSED_TWOPASS", two_pass)
    w = WORKLOADS["mamba2_2p7b"].with_(batch=2, seqlen=5 * 128 + 37, nheads=6, ngroups=2, has_init=True)
    inp = generate(w, seed=nseg)
    y, fs = _run(to_device(inp), algo="fused")
    _check(inp, y, fs, "bf16")


# --------------------------------------------------------------------------
# The fused kernel at state sizes 64 and 16 (the 64-column kernel; at 16 the
# C/B columns past 16 load as zeros): the state kept on chip as rows
# (head, p) x 64 columns, split between the two head warpgroups; and at 256
# (one head per CTA, the warpgroups splitting its state rows n).
# --------------------------------------------------------------------------
@pytest.mark.parametrize("dstate", [16, 64, 256])
@pytest.mark.parametrize("init", [False, True])
@pytest.mark.parametrize("over", FUSED, ids=[str(f) for f in FUSED])
def test_fused_small_states_vs_oracle(over, init, dstate):
    w = WORKLOADS["mamba2_2p7b"].with_(has_init=init, dstate=dstate, **over)
    inp = generate(w, seed=37 + dstate)
    y, fs = _run(to_device(inp), algo="fused")
    _check(inp, y, fs, "bf16")


@pytest.mark.parametrize("dstate", [16, 64, 256])
@pytest.mark.parametrize("grid", [1, 3, 7])
def test_fused_small_states_ranges(grid, dstate, monkeypatch):
    """Contiguous chunk ranges with state hand-offs between CTAs."""
    monkeypatch.setenv("SSD_FUSED_GRID", str(grid))
    w = WORKLOADS["mamba2_2p7b"].with_(batch=2, seqlen=5 * 128 + 37, nheads=6, ngroups=2, has_init=True,
                                     dstate=dstate)
    inp = generate(w, seed=200 + grid)
    y, fs = _run(to_device(inp), algo="fused")
    _check(inp, y, fs, "bf16")


@pytest.mark.parametrize("dstate", [16, 64, 256])
def test_fused_small_states_segments(dstate, monkeypatch):
    """Segments chained through the workspace flags (no two-pass schedule at
    these state sizes)."""
    monkeypatch.setenv("SSD_FUSED_NSEG", "3")
    w = WORKLOADS["mamba2_2p7b"].with_(batch=2, seqlen=5 * 128 + 37, nheads=6, ngroups=2, has_init=True,
                                     dstate=dstate)
    inp = generate(w, seed=300 + dstate)
    y, fs = _run(to_device(inp), algo="fused")
    _check(inp, y, fs, "bf16")


@pytest.mark.parametrize("dstate", [16, 64, 256])
def test_fused_small_states_match_chunked(dstate):
    w = WORKLOADS["mamba2_2p7b"].with_(batch=2, seqlen=640, nheads=6, has_init=True, dstate=dstate)
    d = to_device(generate(w, seed=41))
    y1, f1 = _run(d, algo="fused")
    y2, f2 = _run(d, algo="chunked")
    assert normwise_err(y1, y2) < 1e-2 and normwise_err(f1, f2) < 1e-2


@pytest.mark.parametrize("dstate", [16, 64, 128, 256])
def test_fused_repeat_is_bitwise_stable(dstate):
    """The fused kernel has no atomics in its data path: repeated calls on the
    same inputs must agree bit for bit.  A race between the warps that stage
    one y tile (or any other hand-off inside a CTA) shows up here as a chunk
    that differs from one call to the next."""
    w = WORKLOADS["nsweep_128"].with_(batch=4, seqlen=2048, nheads=32, dstate=dstate)
    inp = generate(w, seed=500 + dstate)
    d = to_device(inp)
    y0, f0 = _run(d, algo="fused")
    for _ in range(7):
        y, fs = _run(d, algo="fused")
        assert torch.equal(y, y0) and torch.equal(fs, f0)
    _check(inp, y0, f0, "bf16")
