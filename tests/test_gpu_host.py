"""GPU parity of ssd_fwd_host (host buffers, pipelined copies) against the
fp64 oracle and against ssd_fwd on device buffers."""
import pytest
import torch

import oracle
import ssd_scan_fwd_b300 as ssd
from ssd_scan_fwd_b300.inputs import WORKLOADS, generate
from tests._util import TOL, normwise_err, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wname,batch,seqlen,algo", [
    ("mamba2_2p7b", 5, 700, "auto"),     # 6 token segments of 128, the last one 60 tokens
    ("mamba2_130m", 2, 1000, "chunked"),
    ("mamba2_130m", 1, 2500, "auto"),    # 10 segments of 256 tokens (the last one 196)
    ("mamba2_2p7b", 3, 4096, "auto"),    # 16 segments of 256 tokens, exact
    ("tiny_fp32", 3, 300, "auto"),       # < 4 chunks: three groups of one batch row
    ("tiny_fp32", 9, 200, "chunked"),    # groups of 3, 3, 3 batch rows
])
def test_host_matches_oracle_and_device(wname, batch, seqlen, algo):
    w = WORKLOADS[wname].with_(batch=batch, seqlen=seqlen, nheads=min(WORKLOADS[wname].nheads, 8), has_init=True)
    inp = generate(w, seed=71)
    host = {k: (None if v is None else v.pin_memory()) for k, v in inp.items()}
    y, fs = ssd.ssd_fwd_host(host["x"], host["dt"], host["A"], host["Bm"], host["Cm"], host["D"],
                             host["init_state"], algo=algo)
    torch.cuda.synchronize()
    y_ref, h_ref = oracle.ssd_recurrent(inp["x"], inp["dt"], inp["A"], inp["Bm"], inp["Cm"], inp["D"],
                                        inp["init_state"])
    tol = TOL[w.io_dtype]
    assert normwise_err(y, y_ref) <= tol
    assert normwise_err(fs, h_ref) <= tol
    d = to_device(inp)
    y_dev, f_dev = ssd.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], d["init_state"], algo=algo)
    torch.cuda.synchronize()
    assert normwise_err(y, y_dev) <= tol
    assert normwise_err(fs, f_dev) <= tol


def test_host_empty_sequence_copies_the_state():
    w = WORKLOADS["tiny_fp32"].with_(batch=2, seqlen=0, has_init=True)
    inp = generate(w, seed=72)
    y, fs = ssd.ssd_fwd_host(inp["x"], inp["dt"], inp["A"], inp["Bm"], inp["Cm"], inp["D"], inp["init_state"])
    torch.cuda.synchronize()
    assert torch.equal(fs, inp["init_state"])


def test_host_without_init_state():
    """Segments chained through the device state buffers from a zero state."""
    w = WORKLOADS["mamba2_2p7b"].with_(batch=2, seqlen=1500, nheads=4)
    inp = generate(w, seed=73)
    host = {k: (None if v is None else v.pin_memory()) for k, v in inp.items()}
    y, fs = ssd.ssd_fwd_host(host["x"], host["dt"], host["A"], host["Bm"], host["Cm"], host["D"], None)
    torch.cuda.synchronize()
    y_ref, h_ref = oracle.ssd_recurrent(inp["x"], inp["dt"], inp["A"], inp["Bm"], inp["Cm"], inp["D"], None)
    assert normwise_err(y, y_ref) <= TOL["bf16"]
    assert normwise_err(fs, h_ref) <= TOL["bf16"]
