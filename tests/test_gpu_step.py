"""GPU parity of the recurrent step (ssd_step) against the fp64 oracle.

The oracle's sequential recurrence over one token, started from the given
state, is exactly one step; over L tokens it is L steps, so repeated calls of
ssd_step must also agree with the chunked forward pass on the same sequence.
"""
import pytest
import torch

import oracle
from ssd_scan_fwd_b300 import api
from ssd_scan_fwd_b300.inputs import Workload, generate

from tests._util import TOL, normwise_err, poison_like

pytestmark = pytest.mark.gpu

# (B, H, P, N, G, io): the vector path (N % 4 == 0) and the scalar one,
# grouped heads, the largest supported sizes, a single head.
CASES = [
    (3, 8, 64, 128, 2, "bf16"),
    (2, 4, 16, 16, 1, "f32"),
    (2, 6, 24, 30, 3, "f32"),
    (1, 2, 256, 256, 1, "bf16"),
    (4, 1, 1, 1, 1, "f32"),
    (2, 80, 64, 128, 1, "bf16"),
]


def _one_token(case, seed):
    B, H, P, N, G, io = case
    w = Workload(name="step", batch=B, seqlen=1, nheads=H, headdim=P, dstate=N, ngroups=G,
                 io_dtype=io, has_init=True, seed=seed)
    inp = generate(w)
    return w, inp


@pytest.mark.parametrize("case", CASES)
def test_step_matches_oracle(case):
    w, inp = _one_token(case, 5000 + CASES.index(case))
    y_ref, h_ref = oracle.ssd_recurrent(inp["x"], inp["dt"], inp["A"], inp["Bm"], inp["Cm"], inp["D"],
                                        inp["init_state"])
    d = {k: v.cuda() for k, v in inp.items() if v is not None}
    state = d["init_state"].clone()
    y = poison_like(d["x"][:, 0])
    api.ssd_step(d["x"][:, 0].contiguous(), d["dt"][:, 0].contiguous(), d["A"], d["Bm"][:, 0].contiguous(),
                 d["Cm"][:, 0].contiguous(), d["D"], state, y=y)
    torch.cuda.synchronize()
    # one step: the state is fp32 arithmetic on exact inputs; y is rounded to the io dtype
    assert normwise_err(state, h_ref) <= 1e-5
    assert normwise_err(y, y_ref[:, 0]) <= (1e-5 if w.io_dtype == "f32" else 8e-3)


def test_step_without_D():
    w, inp = _one_token((2, 4, 32, 64, 2, "f32"), 5100)
    y_ref, h_ref = oracle.ssd_recurrent(inp["x"], inp["dt"], inp["A"], inp["Bm"], inp["Cm"], None,
                                        inp["init_state"])
    d = {k: v.cuda() for k, v in inp.items() if v is not None}
    state = d["init_state"].clone()
    y = api.ssd_step(d["x"][:, 0].contiguous(), d["dt"][:, 0].contiguous(), d["A"], d["Bm"][:, 0].contiguous(),
                     d["Cm"][:, 0].contiguous(), None, state)
    torch.cuda.synchronize()
    assert normwise_err(state, h_ref) <= 1e-5
    assert normwise_err(y, y_ref[:, 0]) <= 1e-5


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_steps_reproduce_the_forward_pass(io):
    """L calls of ssd_step over a sequence give ssd_fwd's y and final state."""
    B, L, H, P, N, G = 2, 40, 4, 64, 128, 2
    w = Workload(name="seq", batch=B, seqlen=L, nheads=H, headdim=P, dstate=N, ngroups=G, io_dtype=io,
                 has_init=True, seed=5200)
    inp = generate(w)
    d = {k: v.cuda() for k, v in inp.items() if v is not None}
    y_fwd, h_fwd = api.ssd_fwd(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], d["init_state"])
    state = d["init_state"].clone()
    ys = []
    for t in range(L):
        ys.append(api.ssd_step(d["x"][:, t].contiguous(), d["dt"][:, t].contiguous(), d["A"],
                               d["Bm"][:, t].contiguous(), d["Cm"][:, t].contiguous(), d["D"], state))
    torch.cuda.synchronize()
    y_steps = torch.stack(ys, dim=1)
    y_ref, h_ref = oracle.ssd_recurrent(inp["x"], inp["dt"], inp["A"], inp["Bm"], inp["Cm"], inp["D"],
                                        inp["init_state"])
    tol = TOL[io]
    assert normwise_err(y_steps, y_ref) <= tol
    assert normwise_err(state, h_ref) <= tol
    assert normwise_err(y_steps, y_fwd) <= tol
    assert normwise_err(state, h_fwd) <= tol


def test_step_empty_batch():
    x = torch.empty(0, 4, 64, device="cuda")
    state = torch.empty(0, 4, 64, 128, device="cuda")
    y = api.ssd_step(x, torch.empty(0, 4, device="cuda"), torch.zeros(4, device="cuda"),
                     torch.empty(0, 1, 128, device="cuda"), torch.empty(0, 1, 128, device="cuda"), None, state)
    assert y.shape == (0, 4, 64)
