"""Failure detection of the fused kernel, on the GPU without a fault: its
device-side waits are bounded.  With the hand-off flags never raised (a test
knob) the units that wait on them run out of time, the kernel stops and
records SSD_ERR_TIMEOUT in the workspace, ssd_workspace_status() reports it,
and the CUDA context stays usable for the next call.
"""
import ctypes
import time

import pytest
import torch

import oracle
import ssd_scan_fwd_b300 as ssd
from ssd_scan_fwd_b300 import _lib
from ssd_scan_fwd_b300.inputs import WORKLOADS, generate
from tests._util import TOL, normwise_err, to_device

pytestmark = pytest.mark.gpu


def _status(ws):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return _lib.lib().ssd_workspace_status(ctypes.c_void_p(ws.data_ptr()), stream)


def test_wait_runs_out_and_is_reported(monkeypatch):
    # 8 head-pair sequences of 6 chunks on 3 CTAs: the tail pieces of two
    # sequences wait for states handed over by another CTA
    w = WORKLOADS["mamba2_2p7b"].with_(batch=2, seqlen=5 * 128 + 37, nheads=6, ngroups=2, has_init=True)
    inp = generate(w, seed=9000)
    d = to_device(inp)
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")

    monkeypatch.setenv("SSD_FUSED_GRID", "3")
    monkeypatch.setenv("SSD_FUSED_TIMEOUT_MS", "50")
    monkeypatch.setenv("SSD_FUSED_TEST_NO_FLAGS", "1")
    t0 = time.time()
    ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], d["init_state"], algo="fused", workspace=ws)
    assert _status(ws) == _lib.SSD_ERR_TIMEOUT
    assert time.time() - t0 < 10.0

    # the same context, the knobs gone: a normal call is correct and clean
    monkeypatch.delenv("SSD_FUSED_TEST_NO_FLAGS")
    monkeypatch.delenv("SSD_FUSED_TIMEOUT_MS")
    y, fs = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], d["init_state"], algo="fused",
                        workspace=ws)
    assert _status(ws) == _lib.SSD_OK
    ry, rf = oracle.ssd_recurrent(inp["x"], inp["dt"], inp["A"], inp["Bm"], inp["Cm"], inp["D"], inp["init_state"])
    assert normwise_err(y, ry) <= TOL["bf16"] and normwise_err(fs, rf) <= TOL["bf16"]


def test_status_of_a_clean_call():
    w = WORKLOADS["mamba2_2p7b"].with_(batch=1, seqlen=300, nheads=4)
    d = to_device(generate(w, seed=9001))
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], None, algo="fused", workspace=ws)
    assert _status(ws) == _lib.SSD_OK


def test_check_status_raises_on_timeout(monkeypatch):
    """ssd_fwd(..., check_status=True) turns a bounded wait that gave up into
    an SsdError carrying SSD_ERR_TIMEOUT; the context stays usable."""
    w = WORKLOADS["mamba2_2p7b"].with_(batch=2, seqlen=5 * 128 + 37, nheads=6, ngroups=2, has_init=True)
    inp = generate(w, seed=9002)
    d = to_device(inp)
    monkeypatch.setenv("SSD_FUSED_GRID", "3")
    monkeypatch.setenv("SSD_FUSED_TIMEOUT_MS", "50")
    monkeypatch.setenv("SSD_FUSED_TEST_NO_FLAGS", "1")
    with pytest.raises(ssd.SsdError) as ei:
        ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], d["init_state"], algo="fused",
                    check_status=True)
    assert ei.value.status == _lib.SSD_ERR_TIMEOUT
    monkeypatch.delenv("SSD_FUSED_TEST_NO_FLAGS")
    monkeypatch.delenv("SSD_FUSED_TIMEOUT_MS")
    y, fs = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], d["init_state"], algo="fused",
                        check_status=True)
    ry, rf = oracle.ssd_recurrent(inp["x"], inp["dt"], inp["A"], inp["Bm"], inp["Cm"], inp["D"], inp["init_state"])
    assert normwise_err(y, ry) <= TOL["bf16"] and normwise_err(fs, rf) <= TOL["bf16"]


def test_check_status_clean_on_chunked_path():
    """The chunked path keeps a status word too: a normal call reports SSD_OK."""
    w = WORKLOADS["nsweep_64"].with_(batch=1, seqlen=300, nheads=4)
    d = to_device(generate(w, seed=9003))
    y, fs = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], algo="chunked", check_status=True)
    assert torch.isfinite(y.float()).all()
