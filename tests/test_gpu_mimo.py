"""GPU parity of the retrieval-rank (MIMO) forward pass against the fp64 oracle.

Page "状态空间模型的对角等价：检索秩与选择性扩展新解", section "从 MIMO 到
HybridMamba", read as: per token R value channels with their own x, B and C
share the token's decay; the update writes all R values; each rank reads its
own output from the updated state.  The library runs this as the fused kernel
over rows (token, rank).  Bar: normwise ‖out − ref‖∞ / ‖ref‖∞ ≤ 2e-2 for y and
final_state (bf16 io, fp32 accumulation); outputs pre-filled with NaN.
"""
import ctypes

import pytest
import torch

import oracle
import ssd_scan_fwd_b300 as ssd
from ssd_scan_fwd_b300 import _lib
from ssd_scan_fwd_b300.inputs import WORKLOADS, generate_mimo
from tests._util import TOL, normwise_err, to_device

pytestmark = pytest.mark.gpu


def _run(d, init=True):
    x = d["x"]
    B, L, R, H, P = x.shape
    N = d["Bm"].shape[4]
    y = torch.full_like(x, float("nan"))
    fs = torch.full((B, H, P, N), float("nan"), device=x.device)
    y, fs = ssd.ssd_fwd_mimo(x, d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], d["init_state"] if init else None,
                             y=y, final_state=fs)
    torch.cuda.synchronize()
    return y, fs


def _check(inp, y, fs):
    ry, rf = oracle.ssd_recurrent_mimo(inp["x"], inp["dt"], inp["A"], inp["Bm"], inp["Cm"], inp["D"],
                                       inp["init_state"])
    ey, ef = normwise_err(y, ry), normwise_err(fs, rf)
    assert ey <= TOL["bf16"], f"y normwise error {ey:.3e}"
    assert ef <= TOL["bf16"], f"final_state normwise error {ef:.3e}"
    return ey, ef


def _w(**kw):
    return WORKLOADS["mamba2_2p7b"].with_(**kw)


# several chunks of rows and a ragged tail at every rank (128 rows = 128 / R tokens)
@pytest.mark.parametrize("dstate", [16, 64, 128, 256])
@pytest.mark.parametrize("rank", [1, 2, 4, 8])
def test_mimo_vs_oracle(rank, dstate):
    w = _w(batch=2, seqlen=(5 * 128 + 37) // rank + 3, nheads=4, ngroups=2, has_init=True, dstate=dstate)
    inp = generate_mimo(w, rank, seed=10 * rank + dstate)
    y, fs = _run(to_device(inp))
    _check(inp, y, fs)


@pytest.mark.parametrize("rank", [2, 8])
def test_mimo_no_init_no_d(rank):
    w = _w(batch=1, seqlen=301, nheads=6, ngroups=3, dstate=128)
    inp = generate_mimo(w, rank, seed=70 + rank)
    inp["D"] = None
    d = to_device(inp)
    y, fs = ssd.ssd_fwd_mimo(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"])
    torch.cuda.synchronize()
    _check(inp, y, fs)


def test_mimo_rank1_equals_siso_bitwise():
    """R = 1 is the SISO problem: the same kernel on the same rows, bit for bit."""
    w = _w(batch=2, seqlen=777, nheads=8, ngroups=2, has_init=True)
    inp = generate_mimo(w, 1, seed=5)
    d = to_device(inp)
    y1, f1 = _run(d)
    sq = lambda t: t.squeeze(2)  # noqa: E731
    y0, f0 = ssd.ssd_fwd(sq(d["x"]), d["dt"], d["A"], sq(d["Bm"]), sq(d["Cm"]), d["D"], d["init_state"],
                         algo="fused")
    torch.cuda.synchronize()
    assert torch.equal(y1.squeeze(2), y0) and torch.equal(f1, f0)


@pytest.mark.parametrize("grid", [1, 3, 7])
@pytest.mark.parametrize("rank", [2, 4])
def test_mimo_ranges(grid, rank, monkeypatch):
    """Contiguous chunk ranges with state hand-offs between CTAs."""
    monkeypatch.setenv("SSD_FUSED_GRID", str(grid))
    w = _w(batch=2, seqlen=(5 * 128 + 37) // rank, nheads=6, ngroups=2, has_init=True)
    inp = generate_mimo(w, rank, seed=100 + grid)
    y, fs = _run(to_device(inp))
    _check(inp, y, fs)


@pytest.mark.parametrize("dstate", [64, 128, 256])
def test_mimo_segments(dstate, monkeypatch):
    """Segments chained through the workspace flags."""
    monkeypatch.setenv("SSD_FUSED_NSEG", "3")
    w = _w(batch=2, seqlen=(5 * 128 + 37) // 4, nheads=6, ngroups=2, has_init=True, dstate=dstate)
    inp = generate_mimo(w, 4, seed=300 + dstate)
    y, fs = _run(to_device(inp))
    _check(inp, y, fs)


def test_mimo_equals_superposed_siso_runs():
    """The state is linear in the written values: with zero init, running
    rank r alone (the other ranks' x zeroed) and summing the final states
    over r gives the MIMO final state (up to bf16/fp32 rounding)."""
    rank = 4
    w = _w(batch=1, seqlen=200, nheads=4, dstate=64)
    inp = generate_mimo(w, rank, seed=9)
    d = to_device(inp)
    _, f_all = _run(d, init=False)
    acc = torch.zeros_like(f_all)
    for r in range(rank):
        x1 = torch.zeros_like(d["x"])
        x1[:, :, r] = d["x"][:, :, r]
        _, f1 = ssd.ssd_fwd_mimo(x1, d["dt"], d["A"], d["Bm"], d["Cm"], d["D"])
        acc += f1
    torch.cuda.synchronize()
    assert normwise_err(acc, f_all) < 1e-4


def test_mimo_empty_and_workspace():
    w = _w(batch=2, seqlen=0, nheads=4, has_init=True)
    d = to_device(generate_mimo(w, 2, seed=1))
    y, fs = _run(d)
    assert y.numel() == 0 and torch.equal(fs, d["init_state"])
    # the fused kernel's workspace (status word, hand-off flags and states of
    # the plan over L * R rows; never the two-pass schedule); none or too
    # little given -> error
    m = _lib.SsdFwdMimoArgs()
    w = _w(batch=2, seqlen=300, nheads=4)
    d = to_device(generate_mimo(w, 4, seed=2))
    rows = lambda t: t.view(2, 1200, *t.shape[3:])  # noqa: E731
    y = torch.empty_like(d["x"])
    fs = torch.empty(2, 4, 64, 128, device="cuda")
    m.base = ssd.make_args(rows(d["x"]), torch.empty(2, 1200, 4, device="cuda"), d["A"], rows(d["Bm"]),
                           rows(d["Cm"]), d["D"], None, rows(y), fs)
    m.base.seqlen = 300
    m.base.dt = d["dt"].data_ptr()
    m.rank = 4
    L = _lib.lib()
    got = L.ssd_fwd_mimo_workspace_size(ctypes.byref(m))
    assert 256 <= got < 1 << 20
    ws = torch.empty(got, dtype=torch.uint8, device="cuda")
    m.base.workspace = ws.data_ptr()
    m.base.workspace_bytes = got - 1
    assert L.ssd_fwd_mimo(ctypes.byref(m), None) == _lib.SSD_ERR_WORKSPACE
    m.base.workspace_bytes = got
    assert L.ssd_fwd_mimo(ctypes.byref(m), None) == _lib.SSD_OK
    torch.cuda.synchronize()
    m.base.workspace = None
    assert L.ssd_fwd_mimo(ctypes.byref(m), None) == _lib.SSD_ERR_WORKSPACE
    m.base.batch = 0
    assert L.ssd_fwd_mimo(ctypes.byref(m), None) == _lib.SSD_OK


def test_mimo_rejects_bad_rank_and_shapes():
    w = _w(batch=1, seqlen=64, nheads=2)
    d = to_device(generate_mimo(w, 3, seed=3))
    with pytest.raises(RuntimeError, match="rank"):
        ssd.ssd_fwd_mimo(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"])
    d = to_device(generate_mimo(w, 2, seed=3))
    with pytest.raises(ValueError):
        ssd.ssd_fwd_mimo(d["x"], d["dt"][:, :32], d["A"], d["Bm"], d["Cm"], d["D"])
