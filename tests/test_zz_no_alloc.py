"""The allocation-free entry point, ssd_fwd_noalloc, through the C ABI.

Some callers cannot allocate device memory themselves (their memory is owned
by a host framework's pool, or a cudaMalloc in their loop could synchronise
the device).  ssd_fwd_noalloc serves them with the fused kernel and a fixed
scratch array inside the library.  This file is named to be collected last,
so that a run stopping at the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import oracle
import ssd_scan_fwd_b300 as ssd
from ssd_scan_fwd_b300 import _lib
from ssd_scan_fwd_b300.inputs import WORKLOADS, generate
from tests._util import TOL, normwise_err, poison_like, to_device

pytestmark = pytest.mark.gpu


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _noalloc(d):
    y = poison_like(d["x"])
    B, _, H, P = d["x"].shape
    fs = torch.full((B, H, P, d["Bm"].shape[3]), float("nan"), device="cuda")
    args = ssd.make_args(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], d["init_state"], y, fs)
    _lib.check(_lib.lib().ssd_fwd_noalloc(ctypes.byref(args), _stream()), "ssd_fwd_noalloc")
    torch.cuda.synchronize()
    return y, fs


def test_no_alloc_matches_ssd_fwd_on_two_calls():
    # 8 head-pair sequences of 6 chunks: the same plan as ssd_fwd (one whole
    # sequence per CTA), so the outputs are bitwise equal
    w = WORKLOADS["mamba2_2p7b"].with_(batch=2, seqlen=700, nheads=8, has_init=True)
    inp = generate(w, seed=123)
    d = to_device(inp)
    y_ref, f_ref = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], d["init_state"])
    torch.cuda.synchronize()
    ry, rf = oracle.ssd_recurrent(inp["x"], inp["dt"], inp["A"], inp["Bm"], inp["Cm"], inp["D"], inp["init_state"])
    for _ in range(2):
        y, fs = _noalloc(d)
        assert normwise_err(y, y_ref) <= TOL["bf16"]
        assert normwise_err(fs, f_ref) <= TOL["bf16"]
        assert torch.equal(y, y_ref) and torch.equal(fs, f_ref)
        assert normwise_err(y, ry) <= TOL["bf16"] and normwise_err(fs, rf) <= TOL["bf16"]
        assert _lib.lib().ssd_fwd_noalloc_status(_stream()) == _lib.SSD_OK


@pytest.mark.parametrize("case", ["ranges_fall_back", "two_pass_fewer_segments"])
def test_no_alloc_schedules_past_the_scratch_size(case, monkeypatch):
    """Problems whose usual hand-off states do not fit in the fixed 1 MiB:
    (a) 40 sequences on 3 CTAs would use contiguous ranges with 40 heads x 2
    rows x 32 KB = 2.5 MiB of hand-off states, so every sequence runs whole on
    one CTA instead; (b) one head pair over 64 chunks runs two passes, whose
    segment states (two heads x 64 KB per segment) allow at most 7 segments
    in 1 MiB.  Both against the oracle."""
    if case == "ranges_fall_back":
        monkeypatch.setenv("SSD_FUSED_GRID", "3")
        w = WORKLOADS["mamba2_2p7b"].with_(batch=2, seqlen=5 * 128 + 37, nheads=40, has_init=True)
    else:
        w = WORKLOADS["mamba2_2p7b"].with_(batch=1, seqlen=8192, nheads=2, has_init=True)
    inp = generate(w, seed=321)
    y, fs = _noalloc(to_device(inp))
    ry, rf = oracle.ssd_recurrent(inp["x"], inp["dt"], inp["A"], inp["Bm"], inp["Cm"], inp["D"], inp["init_state"])
    assert normwise_err(y, ry) <= TOL["bf16"]
    assert normwise_err(fs, rf) <= TOL["bf16"]


def test_no_alloc_timeout_is_reported(monkeypatch):
    """A bounded wait that gives up inside ssd_fwd_noalloc is reported by
    ssd_fwd_noalloc_status (hand-off flags never raised: a test knob), and
    the next call on the same context is clean."""
    w = WORKLOADS["mamba2_2p7b"].with_(batch=2, seqlen=5 * 128 + 37, nheads=6, ngroups=2, has_init=True)
    inp = generate(w, seed=322)
    d = to_device(inp)
    monkeypatch.setenv("SSD_FUSED_GRID", "3")
    monkeypatch.setenv("SSD_FUSED_TIMEOUT_MS", "50")
    monkeypatch.setenv("SSD_FUSED_TEST_NO_FLAGS", "1")
    _noalloc(d)
    assert _lib.lib().ssd_fwd_noalloc_status(_stream()) == _lib.SSD_ERR_TIMEOUT
    monkeypatch.delenv("SSD_FUSED_TEST_NO_FLAGS")
    monkeypatch.delenv("SSD_FUSED_TIMEOUT_MS")
    y, fs = _noalloc(d)
    assert _lib.lib().ssd_fwd_noalloc_status(_stream()) == _lib.SSD_OK
    ry, rf = oracle.ssd_recurrent(inp["x"], inp["dt"], inp["A"], inp["Bm"], inp["Cm"], inp["D"], inp["init_state"])
    assert normwise_err(y, ry) <= TOL["bf16"] and normwise_err(fs, rf) <= TOL["bf16"]


def test_no_alloc_rejects_unsupported_problem():
    w = WORKLOADS["tiny_fp32"]
    d = to_device(generate(w))
    y = torch.empty_like(d["x"])
    args = ssd.make_args(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], None, y, None)
    s = _lib.lib().ssd_fwd_noalloc(ctypes.byref(args), None)
    assert s == _lib.SSD_ERR_UNSUPPORTED
    assert b"fused" in _lib.lib().ssd_last_error_message()
