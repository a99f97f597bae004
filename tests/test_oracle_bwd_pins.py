"""Pins of the backward oracle (oracle.ssd_recurrent_bwd) to things other
than itself:

* central finite differences of the forward oracle, which is pinned on its
  own (tests/test_oracle_pins.py), for every input, at tiny sizes;
* torch.autograd through a recurrence written here with torch ops (fp64),
  at sizes where finite differences would be slow;
* special cases with closed forms (one token; A = 0, where the state is a
  prefix sum and the decay term of dΔ vanishes);
* three planted mistakes in copies of the oracle, each rejected.

The scalar differentiated is  Σ dy ⊙ y + Σ dfinal ⊙ final_state.
"""
import numpy as np
import pytest
import torch

import oracle

NAMES = {"x": "dx", "dt": "ddt", "A": "dA", "Bm": "dBm", "Cm": "dCm", "D": "dD", "h0": "dinit"}


def _case(B, L, H, P, G, N, seed, with_d=True, with_h0=True, with_dfinal=True):
    rng = np.random.default_rng(seed)
    inp = dict(
        x=rng.normal(size=(B, L, H, P)),
        dt=rng.uniform(0.05, 1.0, size=(B, L, H)),
        A=-rng.uniform(0.1, 2.0, size=H),
        Bm=rng.normal(size=(B, L, G, N)),
        Cm=rng.normal(size=(B, L, G, N)),
        D=rng.normal(size=H) if with_d else None,
        h0=rng.normal(size=(B, H, P, N)) if with_h0 else None,
    )
    dy = rng.normal(size=(B, L, H, P))
    dfinal = rng.normal(size=(B, H, P, N)) if with_dfinal else None
    return inp, dy, dfinal


def _loss(inp, dy, dfinal):
    y, hT = oracle.ssd_recurrent(inp["x"], inp["dt"], inp["A"], inp["Bm"], inp["Cm"], inp["D"], inp["h0"])
    s = float((y * dy).sum())
    if dfinal is not None:
        s += float((hT * dfinal).sum())
    return s


def _finite_differences(inp, dy, dfinal, eps=1e-6):
    fd = {}
    for k in NAMES:
        if inp[k] is None:
            continue
        arr = inp[k]
        g = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            a = arr.copy()
            a[idx] += eps
            lp = _loss(dict(inp, **{k: a}), dy, dfinal)
            a[idx] -= 2 * eps
            lm = _loss(dict(inp, **{k: a}), dy, dfinal)
            g[idx] = (lp - lm) / (2 * eps)
        fd[k] = g
    return fd


def _rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


def _grads(fn, inp, dy, dfinal):
    return fn(inp["x"], inp["dt"], inp["A"], inp["Bm"], inp["Cm"], inp["D"], inp["h0"], dy=dy, dfinal=dfinal)


SHAPES = [
    # B, L, H, P, G, N
    (1, 1, 1, 1, 1, 1),
    (2, 7, 4, 3, 2, 5),    # sqrt(L) spans of 3 tokens, the last one short
    (1, 10, 2, 2, 1, 3),   # four spans of 4, 4, 2 tokens
    (2, 5, 3, 2, 3, 2),    # one head per group
]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
@pytest.mark.parametrize("opts", [(True, True, True), (False, False, False), (True, False, True)],
                         ids=["D,h0,dfinal", "none", "D,dfinal"])
def test_bwd_matches_finite_differences(shape, opts):
    inp, dy, dfinal = _case(*shape, seed=sum(shape), with_d=opts[0], with_h0=opts[1], with_dfinal=opts[2])
    g = _grads(oracle.ssd_recurrent_bwd, inp, dy, dfinal)
    fd = _finite_differences(inp, dy, dfinal)
    for k, v in fd.items():
        assert _rel(g[NAMES[k]], v) <= 1e-7, (k, _rel(g[NAMES[k]], v))


def _torch_recurrence(x, dt, A, Bm, Cm, D, h0):
    """The recurrence h_t = exp(Δ_t A) h_{t-1} + Δ_t x_t B_tᵀ, y_t = h_t C_t + D x_t
    with torch ops, heads expanded from their groups (h -> h // (H/G))."""
    B, L, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    idx = torch.arange(H) // (H // G)
    Bh, Ch = Bm[:, :, idx, :], Cm[:, :, idx, :]          # [B, L, H, N]
    h = h0.clone() if h0 is not None else torch.zeros(B, H, P, N, dtype=x.dtype)
    ys = []
    for t in range(L):
        alpha = torch.exp(dt[:, t, :] * A[None, :])     # [B, H]
        h = alpha[:, :, None, None] * h + (dt[:, t, :, None, None] * x[:, t, :, :, None]) * Bh[:, t, :, None, :]
        y = torch.einsum("bhpn,bhn->bhp", h, Ch[:, t])
        if D is not None:
            y = y + D[None, :, None] * x[:, t]
        ys.append(y)
    return torch.stack(ys, dim=1), h


@pytest.mark.parametrize("shape", [(2, 33, 4, 4, 2, 6), (1, 64, 2, 8, 1, 8), (3, 17, 6, 2, 3, 4)])
def test_bwd_matches_autograd(shape):
    inp, dy, dfinal = _case(*shape, seed=7 + shape[1])
    g = _grads(oracle.ssd_recurrent_bwd, inp, dy, dfinal)
    tin = {k: (torch.tensor(v, dtype=torch.float64, requires_grad=True) if v is not None else None)
           for k, v in inp.items()}
    y, hT = _torch_recurrence(tin["x"], tin["dt"], tin["A"], tin["Bm"], tin["Cm"], tin["D"], tin["h0"])
    s = (y * torch.tensor(dy)).sum() + (hT * torch.tensor(dfinal)).sum()
    s.backward()
    for k, name in NAMES.items():
        ref = tin[k].grad.numpy()
        assert _rel(g[name], ref) <= 1e-11, (k, _rel(g[name], ref))


def test_bwd_one_token_closed_form():
    """L = 1, one head, P = N = 1:  h = α h0 + Δ x b,  y = h c + D x."""
    x, dt, a, b, c, d, h0, dy, dh = 0.7, 0.4, -1.3, -0.6, 1.9, 0.25, 0.8, 1.1, -0.45
    alpha = np.exp(dt * a)
    h = alpha * h0 + dt * x * b
    G = dy * c + dh                      # ∂/∂h of dy·y + dh·h
    inp = dict(x=np.full((1, 1, 1, 1), x), dt=np.full((1, 1, 1), dt), A=np.array([a]),
               Bm=np.full((1, 1, 1, 1), b), Cm=np.full((1, 1, 1, 1), c), D=np.array([d]),
               h0=np.full((1, 1, 1, 1), h0))
    g = _grads(oracle.ssd_recurrent_bwd, inp, np.full((1, 1, 1, 1), dy), np.full((1, 1, 1, 1), dh))
    expect = dict(dx=d * dy + G * dt * b, ddt=G * (x * b + a * alpha * h0), dA=G * dt * alpha * h0,
                  dBm=G * dt * x, dCm=dy * h, dD=dy * x, dinit=G * alpha)
    for k, v in expect.items():
        assert np.allclose(g[k].ravel()[0], v, rtol=1e-14, atol=1e-14), (k, g[k], v)


def test_bwd_prefix_sum_case():
    """A = 0: α = 1, h_t = h0 + Σ_{s≤t} Δ_s x_s B_sᵀ.  Then G_t = dfinal + Σ_{s≥t} dy_s C_sᵀ,
    dx_t = D dy_t + Δ_t G_t B_t, and dΔ_t = x_t·(G_t B_t) (no decay term)."""
    inp, dy, dfinal = _case(1, 9, 2, 3, 1, 4, seed=3)
    inp["A"] = np.zeros(2)
    g = _grads(oracle.ssd_recurrent_bwd, inp, dy, dfinal)
    Bm, Cm = inp["Bm"][0, :, 0], inp["Cm"][0, :, 0]
    for h in range(2):
        for t in range(9):
            Gt = dfinal[0, h] + sum(np.outer(dy[0, s, h], Cm[s]) for s in range(t, 9))
            u = Gt @ Bm[t]
            assert np.allclose(g["dx"][0, t, h], inp["D"][h] * dy[0, t, h] + inp["dt"][0, t, h] * u, rtol=1e-12)
            assert np.isclose(g["ddt"][0, t, h], inp["x"][0, t, h] @ u, rtol=1e-12)


@pytest.mark.parametrize("mutant", [1, 2, 3])
def test_bwd_pins_reject_planted_mistakes(mutant):
    inp, dy, dfinal = _case(2, 7, 4, 3, 2, 5, seed=11)
    bad = _grads(oracle.mutant_recurrent_bwd(mutant), inp, dy, dfinal)
    fd = _finite_differences(inp, dy, dfinal)
    worst = max(_rel(bad[NAMES[k]], v) for k, v in fd.items())
    assert worst > 1e-3, f"planted mistake {mutant} not caught (worst rel err {worst:.2e})"
