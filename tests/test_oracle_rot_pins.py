"""Pins of the complex-decay oracle (oracle.ssd_recurrent_rot):
α_t = e^{Δ_t A}(cos θ_t + i sin θ_t), h_t = α_t h_{t-1} + Δ_t x_t B_tᵀ,
y_t = Re(h_t) C_t + D x_t.

* θ = 0 is the real recurrence (pinned on its own in test_oracle_pins.py);
* the parity task of the Foundations page (§2.3): rotating by π on every 1
  bit makes Re(h) the parity of the bits so far;
* closed forms of the impulse response (pure and damped rotation), including
  the imaginary part of the state, which fixes the sign of the rotation;
* the LTI case (constant Δ, θ, B, C) as a causal convolution with kernel
  Re(α^k) Δ (B·C), computed with numpy.convolve;
* split / resume through the complex state; linearity in x.
"""
import numpy as np
import pytest

import oracle


def _rand(B, L, H, P, G, N, seed):
    rng = np.random.default_rng(seed)
    return dict(x=rng.normal(size=(B, L, H, P)), dt=rng.uniform(0.05, 1.0, size=(B, L, H)),
                theta=rng.uniform(-np.pi, np.pi, size=(B, L, H)), A=-rng.uniform(0.1, 2.0, size=H),
                Bm=rng.normal(size=(B, L, G, N)), Cm=rng.normal(size=(B, L, G, N)), D=rng.normal(size=H))


def _run(d, h0=None):
    return oracle.ssd_recurrent_rot(d["x"], d["dt"], d["theta"], d["A"], d["Bm"], d["Cm"], d["D"], h0)


def test_zero_angle_is_the_real_recurrence():
    d = _rand(2, 13, 4, 3, 2, 5, seed=1)
    h0 = np.random.default_rng(2).normal(size=(2, 4, 3, 5))
    y0, hT = oracle.ssd_recurrent(d["x"], d["dt"], d["A"], d["Bm"], d["Cm"], d["D"], h0)
    y1, (hr, hi) = _run(dict(d, theta=np.zeros_like(d["theta"])), (h0, np.zeros_like(h0)))
    assert np.abs(y1 - y0).max() <= 1e-12 * np.abs(y0).max()
    assert np.abs(hr - hT).max() <= 1e-12 * np.abs(hT).max()
    assert np.abs(hi).max() == 0.0


def test_parity_task():
    """B = 0, A = 0, h0 = 1, θ_t = π·bit_t, C = 1: y_t = (−1)^(Σ_{s≤t} bit_s)."""
    bits = np.array([1, 0, 1, 1, 0, 0, 1, 0, 1, 1, 1, 0, 0, 1], dtype=np.float64)
    L = bits.size
    d = dict(x=np.zeros((1, L, 1, 1)), dt=np.ones((1, L, 1)), theta=(np.pi * bits).reshape(1, L, 1),
             A=np.zeros(1), Bm=np.zeros((1, L, 1, 1)), Cm=np.ones((1, L, 1, 1)), D=None)
    y, _ = _run(d, (np.ones((1, 1, 1, 1)), np.zeros((1, 1, 1, 1))))
    expect = (-1.0) ** np.cumsum(bits)
    assert np.allclose(y.ravel(), expect, atol=1e-14)


@pytest.mark.parametrize("a,theta", [(0.0, 0.7), (-0.3, 2.1), (-1.2, -0.4)])
def test_impulse_response_closed_form(a, theta):
    """x = impulse at t=0, Δ = 1, B = C = 1: h_t = e^{a t} e^{iθ t}."""
    L = 25
    x = np.zeros((1, L, 1, 1))
    x[0, 0, 0, 0] = 1.0
    d = dict(x=x, dt=np.ones((1, L, 1)), theta=np.full((1, L, 1), theta), A=np.array([a]),
             Bm=np.ones((1, L, 1, 1)), Cm=np.ones((1, L, 1, 1)), D=None)
    y, (hr, hi) = _run(d)
    t = np.arange(L)
    assert np.allclose(y.ravel(), np.exp(a * t) * np.cos(theta * t), rtol=1e-13, atol=1e-15)
    assert np.isclose(hr.ravel()[0], np.exp(a * (L - 1)) * np.cos(theta * (L - 1)), rtol=1e-13, atol=1e-15)
    assert np.isclose(hi.ravel()[0], np.exp(a * (L - 1)) * np.sin(theta * (L - 1)), rtol=1e-13, atol=1e-15)


def test_lti_case_is_a_convolution():
    rng = np.random.default_rng(5)
    L, P, N = 40, 3, 4
    delta, a, theta = 0.6, -0.5, 1.3
    b, c = rng.normal(size=N), rng.normal(size=N)
    x = rng.normal(size=(1, L, 1, P))
    d = dict(x=x, dt=np.full((1, L, 1), delta), theta=np.full((1, L, 1), theta), A=np.array([a]),
             Bm=np.broadcast_to(b, (1, L, 1, N)).copy(), Cm=np.broadcast_to(c, (1, L, 1, N)).copy(), D=None)
    y, _ = _run(d)
    alpha = np.exp(delta * a) * np.exp(1j * theta)
    kern = np.real(alpha ** np.arange(L)) * delta * float(b @ c)
    for p in range(P):
        ref = np.convolve(x[0, :, 0, p], kern)[:L]
        assert np.allclose(y[0, :, 0, p], ref, rtol=1e-12, atol=1e-13)


def test_split_and_resume_through_the_complex_state():
    d = _rand(2, 30, 4, 3, 2, 5, seed=8)
    y, (hr, hi) = _run(d)
    cut = 17
    first = {k: (v[:, :cut] if k in ("x", "dt", "theta", "Bm", "Cm") else v) for k, v in d.items()}
    second = {k: (v[:, cut:] if k in ("x", "dt", "theta", "Bm", "Cm") else v) for k, v in d.items()}
    y1, h1 = _run(first)
    y2, (hr2, hi2) = _run(second, h1)
    assert np.allclose(np.concatenate([y1, y2], axis=1), y, rtol=1e-12, atol=1e-12)
    assert np.allclose(hr2, hr, rtol=1e-12, atol=1e-12) and np.allclose(hi2, hi, rtol=1e-12, atol=1e-12)


def test_linear_in_x():
    d = _rand(1, 20, 2, 2, 1, 3, seed=9)
    x2 = np.random.default_rng(10).normal(size=d["x"].shape)
    ya, _ = _run(d)
    yb, _ = _run(dict(d, x=x2))
    yc, _ = _run(dict(d, x=2.0 * d["x"] - 3.0 * x2))
    assert np.allclose(yc, 2.0 * ya - 3.0 * yb, rtol=1e-12, atol=1e-12)
