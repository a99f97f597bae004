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

import ssd_scan_fwd_b300 as ssd
from ssd_scan_fwd_b300 import _lib
from ssd_scan_fwd_b300.inputs import WORKLOADS, generate
from tests._util import TOL, normwise_err, poison_like, to_device

pytestmark = pytest.mark.gpu


def test_no_alloc_matches_ssd_fwd_on_two_calls():
    w = WORKLOADS["mamba2_2p7b"].with_(batch=2, seqlen=700, nheads=8, has_init=True)
    d = to_device(generate(w, seed=123))
    y_ref, f_ref = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], d["init_state"])
    torch.cuda.synchronize()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        y = poison_like(d["x"])
        fs = torch.full_like(f_ref, float("nan"))
        args = ssd.make_args(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], d["init_state"], y, fs)
        _lib.check(_lib.lib().ssd_fwd_noalloc(ctypes.byref(args), stream), "ssd_fwd_noalloc")
        torch.cuda.synchronize()
        assert normwise_err(y, y_ref) <= TOL["bf16"]
        assert normwise_err(fs, f_ref) <= TOL["bf16"]


def test_no_alloc_rejects_unsupported_problem():
    w = WORKLOADS["tiny_fp32"]
    d = to_device(generate(w))
    y = torch.empty_like(d["x"])
    args = ssd.make_args(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], None, y, None)
    s = _lib.lib().ssd_fwd_noalloc(ctypes.byref(args), None)
    assert s == _lib.SSD_ERR_UNSUPPORTED
    assert b"fused" in _lib.lib().ssd_last_error_message()
