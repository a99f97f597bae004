"""Pins for the retrieval-rank (MIMO) oracle, oracle.ssd_recurrent_mimo.

Page "状态空间模型的对角等价：检索秩与选择性扩展新解", section "从 MIMO 到
HybridMamba": the retrieval rank is the number of independent value channels
written and read in parallel at a local interface, SSD-MIMO routes an
independent value per rank, and SISO is recovered exactly.  Reading (no
formula on the page): the R channels of a token share its decay, the update
writes all R values, each rank reads its own output from the updated state.
Pinned by: a hand-worked R = 2 example, R = 1 against the pinned SISO
oracle, superposition of R SISO runs (the state is linear in the inputs), and
invariance under permuting the ranks; two plausible mistakes written out here
(each rank decaying the state; each rank reading before the later ranks have
written) are rejected by the superposition pin.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_example_mimo_R2.json")


def _rand(rng, Bsz=2, L=23, R=3, H=4, P=3, G=2, N=5, h0=True):
    x = rng.standard_normal((Bsz, L, R, H, P))
    dt = np.log1p(np.exp(rng.standard_normal((Bsz, L, H)) - 1.0))
    A = -np.exp(rng.uniform(0.0, math.log(16.0), H))
    Bm = rng.standard_normal((Bsz, L, R, G, N)) / math.sqrt(N)
    Cm = rng.standard_normal((Bsz, L, R, G, N)) / math.sqrt(N)
    D = rng.standard_normal(H)
    s0 = 0.1 * rng.standard_normal((Bsz, H, P, N)) if h0 else None
    return x, dt, A, Bm, Cm, D, s0


def _rel(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


def test_hand_example_rank2():
    g = json.load(open(GOLDEN))
    inp = g["inputs"]
    x = np.array(inp["x"]).reshape(1, 2, 2, 1, 1)
    Bm = np.array(inp["B"]).reshape(1, 2, 2, 1, 1)
    Cm = np.array(inp["C"]).reshape(1, 2, 2, 1, 1)
    dt = np.array(inp["dt"]).reshape(1, 2, 1)
    A = np.array([inp["A"]])
    D = np.array([inp["D"]])
    for case in g["cases"]:
        h0 = np.full((1, 1, 1, 1), case["h0"])
        y, hT = oracle.ssd_recurrent_mimo(x, dt, A, Bm, Cm, D, h0)
        assert np.max(np.abs(y.reshape(2, 2) - np.array(case["y"]))) < 1e-14
        assert abs(hT.item() - case["final_state"]) < 1e-14


def test_rank1_is_siso():
    x, dt, A, Bm, Cm, D, h0 = _rand(np.random.default_rng(1), R=1)
    y, hT = oracle.ssd_recurrent_mimo(x, dt, A, Bm, Cm, D, h0)
    y1, h1 = oracle.ssd_recurrent(x[:, :, 0], dt, A, Bm[:, :, 0], Cm[:, :, 0], D, h0)
    assert _rel(y[:, :, 0], y1) < 1e-14 and _rel(hT, h1) < 1e-14


def _superposition(x, dt, A, Bm, Cm, D, h0):
    """y^(r') = Σ_r SISO(x^(r), B^(r), C^(r'), no skip, initial state only in
    the r = 0 term) + D x^(r'); final = Σ_r SISO finals."""
    R = x.shape[2]
    y = np.zeros_like(x)
    fin = 0.0
    for r in range(R):
        for rr in range(R):
            yr, fr = oracle.ssd_recurrent(x[:, :, r], dt, A, Bm[:, :, r], Cm[:, :, rr], None,
                                          h0 if r == 0 else None)
            y[:, :, rr] += yr
            if rr == 0:
                fin = fin + fr
    y += D[None, None, None, :, None] * x
    return y, fin


def test_superposition_of_siso_runs():
    args = _rand(np.random.default_rng(2), R=3)
    y, hT = oracle.ssd_recurrent_mimo(*args)
    ys, fs = _superposition(*args)
    assert _rel(y, ys) < 1e-12 and _rel(hT, fs) < 1e-12


def test_rank_permutation():
    x, dt, A, Bm, Cm, D, h0 = _rand(np.random.default_rng(3), R=4)
    perm = [2, 0, 3, 1]
    y, hT = oracle.ssd_recurrent_mimo(x, dt, A, Bm, Cm, D, h0)
    yp, hp = oracle.ssd_recurrent_mimo(x[:, :, perm], dt, A, Bm[:, :, perm], Cm[:, :, perm], D, h0)
    assert _rel(yp, y[:, :, perm]) < 1e-13 and _rel(hp, hT) < 1e-13


def _mistake(x, dt, A, Bm, Cm, D, h0, kind):
    """Plain numpy recurrence with a planted mistake (P x N state per head)."""
    Bsz, L, R, H, P = x.shape
    G, N = Bm.shape[3], Bm.shape[4]
    y = np.zeros_like(x)
    for b in range(Bsz):
        for h in range(H):
            g = h // (H // G)
            st = np.zeros((P, N)) if h0 is None else h0[b, h].copy()
            for t in range(L):
                a = math.exp(dt[b, t, h] * A[h])
                if kind == "decay_per_rank":
                    for r in range(R):
                        st = a * st + dt[b, t, h] * np.outer(x[b, t, r, h], Bm[b, t, r, g])
                    for r in range(R):
                        y[b, t, r, h] = st @ Cm[b, t, r, g] + D[h] * x[b, t, r, h]
                else:  # "read_before_later_ranks": rank r reads after its own write only
                    st = a * st
                    for r in range(R):
                        st = st + dt[b, t, h] * np.outer(x[b, t, r, h], Bm[b, t, r, g])
                        y[b, t, r, h] = st @ Cm[b, t, r, g] + D[h] * x[b, t, r, h]
    return y


@pytest.mark.parametrize("kind", ["decay_per_rank", "read_before_later_ranks"])
def test_superposition_rejects_planted_mistakes(kind):
    args = _rand(np.random.default_rng(4), Bsz=1, L=6, R=2, H=2, P=2, G=1, N=3)
    ys, _ = _superposition(*args)
    assert _rel(_mistake(*args, kind), ys) > 1e-3
