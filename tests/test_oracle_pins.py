"""Pins for the fp64 CPU oracle.

The oracle is only trusted once it agrees with something other than itself.
Each test below checks it against a fact fixed by the pages or by plain
mathematics, chosen so that a plausible slip (dropped term, wrong index,
swapped operand, wrong sign) fails at least one of them -- the last test plants
exactly those slips in copies of the oracle and checks that they are caught.

Pages (cited by title and section):
  [M3-02] "Mamba-3 深度剖析 - 02. SSM 基础回顾与演进 (Foundations of SSM)"
  [T2M]   "从Transformer到Mamba：状态空间模型（SSM）如何改变序列建模的未来"
  [TaS]   "Transformers are SSMs"
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_example_L4.json")


def _rand_problem(rng, Bsz=2, L=37, H=4, P=3, G=2, N=5, h0=True, D=True):
    x = rng.standard_normal((Bsz, L, H, P))
    dt = np.log1p(np.exp(rng.standard_normal((Bsz, L, H)) - 1.0))
    A = -np.exp(rng.uniform(0.0, math.log(16.0), H))
    Bm = rng.standard_normal((Bsz, L, G, N)) / math.sqrt(N)
    Cm = rng.standard_normal((Bsz, L, G, N)) / math.sqrt(N)
    Dv = rng.standard_normal(H) if D else None
    s0 = 0.1 * rng.standard_normal((Bsz, H, P, N)) if h0 else None
    return dict(x=x, dt=dt, A=A, Bm=Bm, Cm=Cm, D=Dv, h0=s0)


def _golden_problem(g):
    inp = g["inputs"]
    x = np.array(inp["x"]).reshape(1, 4, 1, 1)
    dt = np.array(inp["dt"]).reshape(1, 4, 1)
    A = np.array([inp["A"]])
    Bm = np.array(inp["B"]).reshape(1, 4, 1, 1)
    Cm = np.array(inp["C"]).reshape(1, 4, 1, 1)
    D = np.array([inp["D"]])
    return x, dt, A, Bm, Cm, D


def _relmax(a, b):
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# --------------------------------------------------------------------------
# T1  hand-worked example ([M3-02] §2.1.1, §2.1.2, §2.2.1)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("form", ["recurrent", "quadratic", "chunked1", "chunked3", "chunked4"])
def test_hand_example(form):
    g = json.load(open(GOLDEN))
    x, dt, A, Bm, Cm, D = _golden_problem(g)
    for case in g["cases"]:
        h0 = np.array([[[[case["h0"]]]]])
        if form == "recurrent":
            y, hT = oracle.ssd_recurrent(x, dt, A, Bm, Cm, D, h0)
        elif form == "quadratic":
            y, hT = oracle.ssd_quadratic(x, dt, A, Bm, Cm, D, h0)
        else:
            r = oracle.ssd_chunked(x, dt, A, Bm, Cm, D, h0, chunk=int(form[-1]))
            y, hT = r["y"], r["final_state"]
        np.testing.assert_allclose(y.reshape(4), case["y"], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(hT.reshape(()), case["final_state"], rtol=1e-13)


def test_hand_example_mask_matrix():
    """Columns of M from unit impulses through the recurrence ([TaS] §1.1:
    the recurrence computes the same lower-triangular matrix product)."""
    g = json.load(open(GOLDEN))
    x, dt, A, Bm, Cm, _ = _golden_problem(g)
    M = np.zeros((4, 4))
    for j in range(4):
        e = np.zeros_like(x)
        e[0, j, 0, 0] = 1.0
        y, _ = oracle.ssd_recurrent(e, dt, A, Bm, Cm, None, None)
        M[:, j] = y.reshape(4)
    np.testing.assert_allclose(M, np.array(g["mask_matrix_times_C_B_Delta"]["M"]),
                               rtol=1e-13, atol=1e-15)


# --------------------------------------------------------------------------
# T2  duality: recurrence == masked matrix form ([M3-02] §2.2.1; [T2M] §2.1)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_duality_recurrent_vs_quadratic(seed):
    p = _rand_problem(np.random.default_rng(seed))
    y1, h1 = oracle.ssd_recurrent(**p)
    y2, h2 = oracle.ssd_quadratic(**p)
    assert _relmax(y1, y2) < 1e-12
    assert _relmax(h1, h2) < 1e-12


# --------------------------------------------------------------------------
# Exact brute force: the mask form in rational arithmetic.  With A = -ln 2 and
# integer Δ, α = 2^-Δ is exact, so the matrix product of [M3-02] §2.2.1 can be
# evaluated with Fractions and compared with the fp64 recurrence.
# --------------------------------------------------------------------------
def test_exact_rational_mask_form():
    rng = np.random.default_rng(7)
    L, P, N = 6, 2, 3
    dts = [int(v) for v in rng.integers(0, 4, L)]
    xs = [[int(v) for v in rng.integers(-3, 4, P)] for _ in range(L)]
    Bs = [[int(v) for v in rng.integers(-2, 3, N)] for _ in range(L)]
    Cs = [[int(v) for v in rng.integers(-2, 3, N)] for _ in range(L)]
    Dh = Fraction(3, 4)
    h0 = [[Fraction(int(v), 8) for v in rng.integers(-4, 5, N)] for _ in range(P)]
    alpha = [Fraction(1, 2 ** d) for d in dts]

    def L_mask(i, j):
        if i < j:
            return Fraction(0)
        out = Fraction(1)
        for k in range(j + 1, i + 1):
            out *= alpha[k]
        return out

    y_exact = []
    for i in range(L):
        row = []
        for p in range(P):
            acc = Fraction(0)
            for j in range(i + 1):
                cb = sum(Fraction(Cs[i][n] * Bs[j][n]) for n in range(N))
                acc += L_mask(i, j) * cb * dts[j] * xs[j][p]
            dec = Fraction(1)
            for k in range(i + 1):
                dec *= alpha[k]
            acc += dec * sum(Cs[i][n] * h0[p][n] for n in range(N))
            acc += Dh * xs[i][p]
            row.append(acc)
        y_exact.append(row)

    x = np.array(xs, float).reshape(1, L, 1, P)
    dt = np.array(dts, float).reshape(1, L, 1)
    A = np.array([-math.log(2.0)])
    Bm = np.array(Bs, float).reshape(1, L, 1, N)
    Cm = np.array(Cs, float).reshape(1, L, 1, N)
    D = np.array([0.75])
    s0 = np.array([[float(v) for v in r] for r in h0]).reshape(1, 1, P, N)
    y, _ = oracle.ssd_recurrent(x, dt, A, Bm, Cm, D, s0)
    ref = np.array([[float(v) for v in r] for r in y_exact])
    np.testing.assert_allclose(y.reshape(L, P), ref, rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# T3  LTI closed form ([TaS] §1.1: y = (CB, CAB, CA²B, ...) * x).  With constant
# Δ, B, C the scan is a causal convolution with kernel K_k = Δ (C·B) α^k,
# computed here by numpy's convolution.  K_0 = Δ C·B pins that y_t sees x_t.
# --------------------------------------------------------------------------
def test_lti_convolution():
    rng = np.random.default_rng(3)
    L, P, N = 50, 4, 6
    delta, Aval = 0.37, -1.3
    b = rng.standard_normal(N)
    c = rng.standard_normal(N)
    x = rng.standard_normal((1, L, 1, P))
    dt = np.full((1, L, 1), delta)
    A = np.array([Aval])
    Bm = np.broadcast_to(b, (1, L, 1, N)).copy()
    Cm = np.broadcast_to(c, (1, L, 1, N)).copy()
    D = np.array([0.8])
    y, _ = oracle.ssd_recurrent(x, dt, A, Bm, Cm, D, None)
    alpha = math.exp(delta * Aval)
    K = delta * float(c @ b) * alpha ** np.arange(L)
    for p in range(P):
        ref = np.convolve(x[0, :, 0, p], K)[:L] + 0.8 * x[0, :, 0, p]
        np.testing.assert_allclose(y[0, :, 0, p], ref, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# T4  special cases of the gates ([M3-02] §2.1.2: α ∈ (0,1) forgets, α = 1
# remembers)
# --------------------------------------------------------------------------
def test_no_decay_is_prefix_sum():
    """A = 0 ⇒ α = 1 ⇒ h_t = h0 + Σ_{i≤t} Δ_i x_i B_iᵀ (numpy cumsum)."""
    p = _rand_problem(np.random.default_rng(4), Bsz=1, H=2, G=1)
    p["A"] = np.zeros_like(p["A"])
    y, hT = oracle.ssd_recurrent(**p)
    x, dt, Bm, Cm, D, h0 = p["x"], p["dt"], p["Bm"], p["Cm"], p["D"], p["h0"]
    upd = np.einsum("blh,blhp,bln->blhpn", dt, x, Bm[:, :, 0, :])
    states = np.cumsum(upd, axis=1) + h0[:, None]
    ref = np.einsum("bln,blhpn->blhp", Cm[:, :, 0, :], states) + D[None, None, :, None] * x
    assert _relmax(y, ref) < 1e-12
    assert _relmax(hT, states[:, -1]) < 1e-12


def test_zero_input_matrix_is_skip_plus_decayed_readout():
    """B = 0 ⇒ the state only decays: y_t = exp(A Σ_{k≤t} Δ_k) C_tᵀ h0 + D x_t."""
    p = _rand_problem(np.random.default_rng(5), Bsz=1, H=2, G=1)
    p["Bm"] = np.zeros_like(p["Bm"])
    y, hT = oracle.ssd_recurrent(**p)
    x, dt, A, Cm, D, h0 = p["x"], p["dt"], p["A"], p["Cm"], p["D"], p["h0"]
    dec = np.exp(np.cumsum(dt, axis=1) * A[None, None, :])  # [b,l,h]
    ref = dec[..., None] * np.einsum("bln,bhpn->blhp", Cm[:, :, 0, :], h0) + D[None, None, :, None] * x
    assert _relmax(y, ref) < 1e-12
    assert _relmax(hT, dec[:, -1, :, None, None] * h0) < 1e-12


def test_zero_x_and_no_init_gives_zero():
    p = _rand_problem(np.random.default_rng(6), h0=False)
    p["x"] = np.zeros_like(p["x"])
    y, hT = oracle.ssd_recurrent(**p)
    assert np.all(y == 0.0) and np.all(hT == 0.0)


# --------------------------------------------------------------------------
# T5  chunk-size invariance of the chunked decomposition (mask figure of
# [M3-02] §2.2.2: block decomposition is exact)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("Q", [1, 2, 3, 8, 16, 37, 64])
def test_chunked_equals_recurrent(Q):
    p = _rand_problem(np.random.default_rng(8), L=37)
    y1, h1 = oracle.ssd_recurrent(**p)
    r = oracle.ssd_chunked(**p, chunk=Q)
    assert _relmax(r["y"], y1) < 1e-12
    assert _relmax(r["final_state"], h1) < 1e-12


def test_chunked_intermediates_consistent():
    """The states entering chunk c equal the recurrence run on the first c·Q
    tokens; dA_cs is the in-chunk running sum of Δ·A."""
    p = _rand_problem(np.random.default_rng(9), L=40)
    Q = 16
    r = oracle.ssd_chunked(**p, chunk=Q)
    for c in range(3):
        t = c * Q
        if t == 0:
            ref = p["h0"]
        else:
            q = dict(p)
            q["x"], q["dt"] = p["x"][:, :t], p["dt"][:, :t]
            q["Bm"], q["Cm"] = p["Bm"][:, :t], p["Cm"][:, :t]
            _, ref = oracle.ssd_recurrent(**q)
        assert _relmax(r["states_in"][:, c], ref) < 1e-12
    dA = p["dt"] * p["A"][None, None, :]
    for c in range(3):
        seg = dA[:, c * Q:(c + 1) * Q, :]
        cs = np.cumsum(seg, axis=1).transpose(0, 2, 1)
        n = cs.shape[-1]
        np.testing.assert_allclose(r["dA_cs"][:, :, c, :n], cs, rtol=1e-13, atol=1e-13)
        if n < Q:  # padded tail: Δ = 0 keeps the sum constant
            np.testing.assert_allclose(r["dA_cs"][:, :, c, n:], cs[..., -1:].repeat(Q - n, -1))


# --------------------------------------------------------------------------
# T6  split / resume through the state
# --------------------------------------------------------------------------
def test_split_resume():
    p = _rand_problem(np.random.default_rng(10), L=41)
    y, hT = oracle.ssd_recurrent(**p)
    cut = 17
    a = {k: (v[:, :cut] if k in ("x", "dt", "Bm", "Cm") else v) for k, v in p.items()}
    b = {k: (v[:, cut:] if k in ("x", "dt", "Bm", "Cm") else v) for k, v in p.items()}
    ya, ha = oracle.ssd_recurrent(**a)
    b["h0"] = ha
    yb, hb = oracle.ssd_recurrent(**b)
    assert _relmax(np.concatenate([ya, yb], axis=1), y) < 1e-13
    assert _relmax(hb, hT) < 1e-13


# --------------------------------------------------------------------------
# T7  groups: G shared B/C groups == the same call with B/C expanded per head
# --------------------------------------------------------------------------
def test_group_expansion():
    p = _rand_problem(np.random.default_rng(11), H=6, G=3)
    y, hT = oracle.ssd_recurrent(**p)
    q = dict(p)
    q["Bm"] = np.repeat(p["Bm"], 2, axis=2)  # head h reads group h // (H/G)
    q["Cm"] = np.repeat(p["Cm"], 2, axis=2)
    y2, h2 = oracle.ssd_recurrent(**q)
    assert _relmax(y, y2) < 1e-14 and _relmax(hT, h2) < 1e-14


# --------------------------------------------------------------------------
# The per-(batch, head) helper used for spot checks equals the matching
# slices of the whole-problem recurrence: grouped B/C (G = 4, two heads per
# group, distinct values per group), a skip term D and an initial state that
# differ per head, so that a wrong group index, an unsliced D or an unsliced
# initial state changes the result.
# --------------------------------------------------------------------------
def test_recurrent_heads_equals_slices():
    p = _rand_problem(np.random.default_rng(13), Bsz=2, L=45, H=8, G=4, P=3, N=5)
    y, hT = oracle.ssd_recurrent(**p)
    inputs = dict(x=p["x"], dt=p["dt"], A=p["A"], Bm=p["Bm"], Cm=p["Cm"], D=p["D"], init_state=p["h0"])
    pairs = [(b, h) for b in range(2) for h in range(8)]
    got = oracle.ssd_recurrent_heads(inputs, pairs)
    assert sorted(got) == sorted(pairs)
    for (b, h), (yh, fh) in got.items():
        assert yh.shape == (45, 3) and fh.shape == (3, 5)
        assert _relmax(yh, y[b, :, h, :]) < 1e-14, (b, h)
        assert _relmax(fh, hT[b, h]) < 1e-14, (b, h)
    # without D and initial state
    inputs0 = dict(inputs, D=None, init_state=None)
    y0, h00 = oracle.ssd_recurrent(p["x"], p["dt"], p["A"], p["Bm"], p["Cm"])
    for (b, h), (yh, fh) in oracle.ssd_recurrent_heads(inputs0, [(1, 7), (0, 2)]).items():
        assert _relmax(yh, y0[b, :, h, :]) < 1e-14 and _relmax(fh, h00[b, h]) < 1e-14


# --------------------------------------------------------------------------
# T8  linearity in x (zero init) and superposition with the initial state
# --------------------------------------------------------------------------
def test_linearity_and_superposition():
    rng = np.random.default_rng(12)
    p = _rand_problem(rng, h0=False, D=True)
    x2 = rng.standard_normal(p["x"].shape)
    y1, _ = oracle.ssd_recurrent(**p)
    q = dict(p, x=x2)
    y2, _ = oracle.ssd_recurrent(**q)
    r = dict(p, x=2.5 * p["x"] - 0.5 * x2)
    y3, _ = oracle.ssd_recurrent(**r)
    assert _relmax(y3, 2.5 * y1 - 0.5 * y2) < 1e-12
    s0 = 0.1 * rng.standard_normal((p["x"].shape[0], p["x"].shape[2], p["x"].shape[3], p["Bm"].shape[3]))
    ya, _ = oracle.ssd_recurrent(**dict(p, h0=s0))
    yb, _ = oracle.ssd_recurrent(**dict(p, x=np.zeros_like(p["x"]), h0=s0))
    assert _relmax(ya, y1 + yb) < 1e-12


# --------------------------------------------------------------------------
# T9  semiseparable structure ([TaS] §1, §1.1): every strictly-lower block of
# the L×L matrix has rank ≤ N
# --------------------------------------------------------------------------
def test_semiseparable_rank():
    rng = np.random.default_rng(13)
    L, N = 24, 3
    dt = np.log1p(np.exp(rng.standard_normal((1, L, 1)) - 1.0))
    A = np.array([-0.7])
    Bm = rng.standard_normal((1, L, 1, N))
    Cm = rng.standard_normal((1, L, 1, N))
    M = np.zeros((L, L))
    for j in range(L):
        e = np.zeros((1, L, 1, 1))
        e[0, j, 0, 0] = 1.0
        y, _ = oracle.ssd_recurrent(e, dt, A, Bm, Cm, None, None)
        M[:, j] = y.reshape(L)
    assert np.allclose(np.triu(M, 1), 0.0)
    for k in range(1, L):
        s = np.linalg.svd(M[k:, :k], compute_uv=False)
        rank = int(np.sum(s > 1e-10 * s[0]))
        assert rank <= N
    # and the rank bound is attained (N is not larger than needed)
    s = np.linalg.svd(M[L // 2:, :L // 2], compute_uv=False)
    assert int(np.sum(s > 1e-10 * s[0])) == N


# --------------------------------------------------------------------------
# Planted mistakes: copies of the oracle with one slip each must fail a pin.
# --------------------------------------------------------------------------
def _passes_pins(run):
    g = json.load(open(GOLDEN))
    x, dt, A, Bm, Cm, D = _golden_problem(g)
    ok = True
    for case in g["cases"]:
        h0 = np.array([[[[case["h0"]]]]])
        y, hT = run(x, dt, A, Bm, Cm, D, h0)
        ok &= np.allclose(y.reshape(4), case["y"], rtol=1e-12)
        ok &= np.allclose(hT.reshape(()), case["final_state"], rtol=1e-12)
    p = _rand_problem(np.random.default_rng(0))
    y1, _ = run(**p)
    y2, _ = oracle.ssd_quadratic(**p)
    ok &= _relmax(y1, y2) < 1e-12
    return bool(ok)


def test_pins_accept_oracle():
    assert _passes_pins(oracle.ssd_recurrent)


@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5])
def test_pins_reject_planted_mistakes(mutant):
    assert not _passes_pins(oracle.mutant_recurrent(mutant))


# --------------------------------------------------------------------------
# Steps around the scan: Δ = softplus(dt + dt_bias) and the gate y · silu(z)
# (page "从 SSM 的长期记忆问题，到 Mamba 的选择性机制与硬件感知扫描": selective SSM
# and Mamba block paragraphs), pinned by closed forms on the hand example.
# --------------------------------------------------------------------------
GOLDEN_GATE = os.path.join(os.path.dirname(__file__), "golden", "hand_example_gate_L4.json")


def _gate_problem():
    g = json.load(open(GOLDEN))
    gg = json.load(open(GOLDEN_GATE))
    x, dt, A, Bm, Cm, D = _golden_problem(g)
    raw = np.array(gg["dt_raw"]).reshape(1, 4, 1)
    z = np.array(gg["z"]).reshape(1, 4, 1, 1)
    return gg, x, dt, raw, A, Bm, Cm, D, z


def test_softplus_delta_reproduces_hand_example():
    gg, x, dt, raw, A, Bm, Cm, D, _ = _gate_problem()
    d = oracle.delta(raw, np.array([gg["dt_bias"]]), dt_softplus=True)
    np.testing.assert_allclose(d, dt, rtol=1e-14)
    y, hT = oracle.ssd_fwd_ex(x, raw, A, Bm, Cm, D, None, dt_bias=np.array([gg["dt_bias"]]), dt_softplus=True)
    np.testing.assert_allclose(y.reshape(4), gg["y_ungated"], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(hT.reshape(()), gg["final_state"], rtol=1e-12)


def test_gate_closed_forms():
    gg, x, dt, raw, A, Bm, Cm, D, z = _gate_problem()
    np.testing.assert_allclose(oracle.silu(np.array(gg["z"])), gg["silu_z"], rtol=1e-14, atol=0)
    y, hT = oracle.ssd_fwd_ex(x, dt, A, Bm, Cm, D, None, z=z)
    np.testing.assert_allclose(y.reshape(4), gg["y_gated"], rtol=1e-12, atol=1e-14)
    # the gate touches y only, never the state
    np.testing.assert_allclose(hT.reshape(()), gg["final_state"], rtol=1e-12)


def test_softplus_limits_and_identity_without_options():
    v = np.array([-800.0, -40.0, 0.0, 40.0, 800.0])
    sp = oracle.softplus(v)
    assert sp[0] == 0.0 and abs(sp[1] - math.exp(-40.0)) < 1e-30
    assert sp[2] == math.log(2.0) and sp[3] == 40.0 + math.log1p(math.exp(-40.0)) and sp[4] == 800.0
    rng = np.random.default_rng(17)
    p = _rand_problem(rng)
    y0, h0 = oracle.ssd_recurrent(p["x"], p["dt"], p["A"], p["Bm"], p["Cm"], p["D"], p["h0"])
    y1, h1 = oracle.ssd_fwd_ex(p["x"], p["dt"], p["A"], p["Bm"], p["Cm"], p["D"], p["h0"])
    assert np.array_equal(y0, y1) and np.array_equal(h0, h1)
    # a bias without softplus is a plain shift of Δ
    b = rng.uniform(0.0, 0.5, p["A"].shape[0])
    y2, _ = oracle.ssd_fwd_ex(p["x"], p["dt"], p["A"], p["Bm"], p["Cm"], p["D"], p["h0"], dt_bias=b)
    y3, _ = oracle.ssd_recurrent(p["x"], p["dt"] + b[None, None, :], p["A"], p["Bm"], p["Cm"], p["D"], p["h0"])
    np.testing.assert_allclose(y2, y3, rtol=1e-15, atol=0)


def test_gate_sign_mistake_is_caught():
    """A gate written with σ(−z) instead of σ(z) fails the closed-form pin."""
    gg, x, dt, raw, A, Bm, Cm, D, z = _gate_problem()
    y, _ = oracle.ssd_recurrent(x, dt, A, Bm, Cm, D, None)
    zf = np.array(gg["z"]).reshape(1, 4, 1, 1)
    wrong = y * (zf / (1.0 + np.exp(zf)))
    assert not np.allclose(wrong.reshape(4), gg["y_gated"], rtol=1e-6)
