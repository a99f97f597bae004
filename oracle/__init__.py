"""fp64 CPU oracle for the SSD selective-scan forward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference legs may import this package.  The
product path (the CUDA library and its Python binding) never imports, links or
calls it, and the oracle imports nothing from the product.

The arithmetic lives in ``ssd_oracle.c`` (plain loops, fp64, OpenMP over
(batch, head)); this module only compiles it with gcc on first use and
marshals numpy arrays.  Three forms are exposed:

* :func:`ssd_recurrent` -- the sequential recurrence, the primary oracle
  ("Mamba-3 深度剖析 - 02 (Foundations of SSM)", §2.1.2 boxed recurrence,
  plus the skip term D of §2.1.1);
* :func:`ssd_quadratic` -- the masked matrix form Y = (L ⊙ C Bᵀ) X of §2.2.1
  (diagnostic, O(L²));
* :func:`ssd_chunked` -- the chunked decomposition, returning the per-chunk
  intermediates (in-chunk log-decay sums, chunk states, states entering each
  chunk) that the per-step CUDA kernels are checked against;
* :func:`ssd_fwd_ex` -- the recurrence with Δ = softplus(dt + dt_bias) and the
  output gate y · silu(z) around it (the Mamba block steps of the page
  "从 SSM 的长期记忆问题，到 Mamba 的选择性机制与硬件感知扫描").

Parity pins: every form is pinned by tests in ``tests/test_oracle_pins.py``
(hand-worked example, duality, exact rational brute force, LTI convolution,
special cases, chunk-size invariance, split/resume, linearity, semiseparable
rank).  Parity unpinned: the head-to-group order (heads split into G
contiguous groups) -- the pages print no example that fixes it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libssd_oracle.so")
_lock = threading.Lock()
_lib = None

_dbl_p = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def build(force: bool = False, mutant: int = 0, bwd_mutant: int = 0) -> str:
    """Compile ssd_oracle.c into a shared library with gcc (no fast-math).
    ``mutant`` / ``bwd_mutant`` > 0 build a copy with a planted mistake in
    the forward / backward recurrence (pin tests only)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if mutant:
        path = os.path.join(_BUILD_DIR, f"libssd_oracle_mutant{mutant}.so")
    elif bwd_mutant:
        path = os.path.join(_BUILD_DIR, f"libssd_oracle_bwd_mutant{bwd_mutant}.so")
    else:
        path = _LIB_PATH
    if force or not os.path.exists(path) or (os.path.getmtime(path) < os.path.getmtime(_SRC)):
        tmp = path + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared",
               f"-DORACLE_MUTANT={int(mutant)}", f"-DORACLE_BWD_MUTANT={int(bwd_mutant)}",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, path)
    return path


def _bind(lib):
    common = [_i64] * 6
    lib.oracle_ssd_recurrent.argtypes = common + [_dbl_p] * 9
    lib.oracle_ssd_recurrent.restype = ctypes.c_int
    lib.oracle_ssd_quadratic.argtypes = common + [_dbl_p] * 9
    lib.oracle_ssd_quadratic.restype = ctypes.c_int
    lib.oracle_ssd_chunked.argtypes = common + [_i64] + [_dbl_p] * 12
    lib.oracle_ssd_chunked.restype = ctypes.c_int
    lib.oracle_ssd_recurrent_bwd.argtypes = common + [_dbl_p] * 16
    lib.oracle_ssd_recurrent_bwd.restype = ctypes.c_int
    lib.oracle_ssd_recurrent_rot.argtypes = common + [_dbl_p] * 12
    lib.oracle_ssd_recurrent_rot.restype = ctypes.c_int
    lib.oracle_ssd_recurrent_mimo.argtypes = [_i64] * 7 + [_dbl_p] * 9
    lib.oracle_ssd_recurrent_mimo.restype = ctypes.c_int
    lib.oracle_set_threads.argtypes = [ctypes.c_int]
    lib.oracle_set_threads.restype = None
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = ctypes.c_int
    return lib


def mutant_recurrent(mutant: int):
    """The recurrence from a copy of the oracle with planted mistake ``mutant``
    (see ORACLE_MUTANT in ssd_oracle.c).  Used only to show that the pins
    reject such mistakes."""
    lib = _bind(ctypes.CDLL(build(mutant=mutant)))

    def run(x, dt, A, Bm, Cm, D=None, h0=None):
        (x, dt, A, Bm, Cm, D, h0), dims = _prep(x, dt, A, Bm, Cm, D, h0)
        Bsz, L, H, P, G, N = dims
        y = np.empty((Bsz, L, H, P), np.float64)
        hT = np.empty((Bsz, H, P, N), np.float64)
        rc = lib.oracle_ssd_recurrent(*dims, _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm),
                                      _ptr(D), _ptr(h0), _ptr(y), _ptr(hT))
        if rc:
            raise ValueError(f"mutant oracle failed ({rc})")
        return y, hT

    return run


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def set_threads(n: int) -> None:
    """Number of OpenMP threads the oracle uses (0 = OpenMP default)."""
    _load().oracle_set_threads(int(n))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor -> numpy (values are upcast exactly)
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dbl_p)


def _dims(x, Bm):
    Bsz, L, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    return Bsz, L, H, P, G, N


def _prep(x, dt, A, Bm, Cm, D, h0):
    x, dt, A, Bm, Cm, D, h0 = (_f64(v) for v in (x, dt, A, Bm, Cm, D, h0))
    Bsz, L, H, P, G, N = _dims(x, Bm)
    assert dt.shape == (Bsz, L, H) and A.shape == (H,)
    assert Bm.shape == (Bsz, L, G, N) and Cm.shape == (Bsz, L, G, N)
    assert D is None or D.shape == (H,)
    assert h0 is None or h0.shape == (Bsz, H, P, N)
    return (x, dt, A, Bm, Cm, D, h0), (Bsz, L, H, P, G, N)


def ssd_recurrent(x, dt, A, Bm, Cm, D=None, h0=None):
    """Sequential recurrence.  Returns (y [B,L,H,P], final_state [B,H,P,N]) in fp64."""
    (x, dt, A, Bm, Cm, D, h0), dims = _prep(x, dt, A, Bm, Cm, D, h0)
    Bsz, L, H, P, G, N = dims
    y = np.empty((Bsz, L, H, P), np.float64)
    hT = np.empty((Bsz, H, P, N), np.float64)
    rc = _load().oracle_ssd_recurrent(*dims, _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm),
                                      _ptr(D), _ptr(h0), _ptr(y), _ptr(hT))
    if rc:
        raise ValueError(f"oracle_ssd_recurrent failed ({rc})")
    return y, hT


def _bwd(lib, x, dt, A, Bm, Cm, D, h0, dy, dhT):
    (x, dt, A, Bm, Cm, D, h0), dims = _prep(x, dt, A, Bm, Cm, D, h0)
    Bsz, L, H, P, G, N = dims
    dy = _f64(dy)
    dhT = _f64(dhT)
    assert dy.shape == (Bsz, L, H, P)
    assert dhT is None or dhT.shape == (Bsz, H, P, N)
    out = {
        "dx": np.empty((Bsz, L, H, P), np.float64),
        "ddt": np.empty((Bsz, L, H), np.float64),
        "dA": np.empty((H,), np.float64),
        "dBm": np.empty((Bsz, L, G, N), np.float64),
        "dCm": np.empty((Bsz, L, G, N), np.float64),
        "dD": np.empty((H,), np.float64),
        "dinit": np.empty((Bsz, H, P, N), np.float64),
    }
    rc = lib.oracle_ssd_recurrent_bwd(*dims, _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm),
                                      _ptr(D), _ptr(h0), _ptr(dy), _ptr(dhT), _ptr(out["dx"]),
                                      _ptr(out["ddt"]), _ptr(out["dA"]), _ptr(out["dBm"]),
                                      _ptr(out["dCm"]), _ptr(out["dD"]), _ptr(out["dinit"]))
    if rc:
        raise ValueError(f"oracle_ssd_recurrent_bwd failed ({rc})")
    return out


def ssd_recurrent_bwd(x, dt, A, Bm, Cm, D=None, h0=None, dy=None, dfinal=None):
    """Gradient of  Σ dy ⊙ y + Σ dfinal ⊙ final_state  through the recurrence
    (reverse mode, states recomputed from every sqrt(L)-th one).  Returns a
    dict of fp64 arrays: dx [B,L,H,P], ddt [B,L,H] (w.r.t. Δ), dA [H],
    dBm, dCm [B,L,G,N], dD [H], dinit [B,H,P,N]."""
    return _bwd(_load(), x, dt, A, Bm, Cm, D, h0, dy, dfinal)


def mutant_recurrent_bwd(mutant: int):
    """ssd_recurrent_bwd from a copy of the oracle with planted backward
    mistake ``mutant`` (see ORACLE_BWD_MUTANT in ssd_oracle.c); pin tests only."""
    lib = _bind(ctypes.CDLL(build(bwd_mutant=mutant)))

    def run(x, dt, A, Bm, Cm, D=None, h0=None, dy=None, dfinal=None):
        return _bwd(lib, x, dt, A, Bm, Cm, D, h0, dy, dfinal)

    return run


def ssd_recurrent_rot(x, dt, theta, A, Bm, Cm, D=None, h0=None):
    """The recurrence with a complex (rotational) decay
    α_t = e^{Δ_t A}(cos θ_t + i sin θ_t): complex state, y_t = Re(h_t) C_t + D x_t.
    theta [B,L,H]; h0 None or a pair (re, im) of [B,H,P,N].  Returns
    (y [B,L,H,P], (final_re, final_im)) in fp64."""
    h0_re, h0_im = (None, None) if h0 is None else h0
    (x, dt, A, Bm, Cm, D, h0_re), dims = _prep(x, dt, A, Bm, Cm, D, h0_re)
    Bsz, L, H, P, G, N = dims
    theta = _f64(theta)
    h0_im = _f64(h0_im)
    assert theta.shape == (Bsz, L, H)
    assert h0_im is None or h0_im.shape == (Bsz, H, P, N)
    y = np.empty((Bsz, L, H, P), np.float64)
    hr = np.empty((Bsz, H, P, N), np.float64)
    hi = np.empty((Bsz, H, P, N), np.float64)
    rc = _load().oracle_ssd_recurrent_rot(*dims, _ptr(x), _ptr(dt), _ptr(theta), _ptr(A), _ptr(Bm), _ptr(Cm),
                                          _ptr(D), _ptr(h0_re), _ptr(h0_im), _ptr(y), _ptr(hr), _ptr(hi))
    if rc:
        raise ValueError(f"oracle_ssd_recurrent_rot failed ({rc})")
    return y, (hr, hi)


def ssd_quadratic(x, dt, A, Bm, Cm, D=None, h0=None):
    """Masked matrix (quadratic) form.  Returns (y, final_state) in fp64."""
    (x, dt, A, Bm, Cm, D, h0), dims = _prep(x, dt, A, Bm, Cm, D, h0)
    Bsz, L, H, P, G, N = dims
    y = np.empty((Bsz, L, H, P), np.float64)
    hT = np.empty((Bsz, H, P, N), np.float64)
    rc = _load().oracle_ssd_quadratic(*dims, _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm),
                                      _ptr(D), _ptr(h0), _ptr(y), _ptr(hT))
    if rc:
        raise ValueError(f"oracle_ssd_quadratic failed ({rc})")
    return y, hT


def ssd_chunked(x, dt, A, Bm, Cm, D=None, h0=None, chunk: int = 64):
    """Chunked form.  Returns a dict with y, final_state and the intermediates
    dA_cs [B,H,nc,Q], chunk_states [B,nc,H,P,N], states_in [B,nc,H,P,N] (fp64)."""
    (x, dt, A, Bm, Cm, D, h0), dims = _prep(x, dt, A, Bm, Cm, D, h0)
    Bsz, L, H, P, G, N = dims
    Q = int(chunk)
    nc = (L + Q - 1) // Q
    out = {
        "dA_cs": np.empty((Bsz, H, nc, Q), np.float64),
        "chunk_states": np.empty((Bsz, nc, H, P, N), np.float64),
        "states_in": np.empty((Bsz, nc, H, P, N), np.float64),
        "y": np.empty((Bsz, L, H, P), np.float64),
        "final_state": np.empty((Bsz, H, P, N), np.float64),
    }
    rc = _load().oracle_ssd_chunked(*dims, Q, _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm),
                                    _ptr(D), _ptr(h0), _ptr(out["dA_cs"]),
                                    _ptr(out["chunk_states"]), _ptr(out["states_in"]),
                                    _ptr(out["y"]), _ptr(out["final_state"]))
    if rc:
        raise ValueError(f"oracle_ssd_chunked failed ({rc})")
    return out


def ssd_recurrent_mimo(x, dt, A, Bm, Cm, D=None, h0=None):
    """Retrieval rank R (MIMO; page "状态空间模型的对角等价：检索秩与选择性扩展新解",
    section "从 MIMO 到 HybridMamba", read as: R channels per token share the
    decay, the update writes all R values, each rank reads its own output):
        h_t = α_t h_{t-1} + Δ_t Σ_r x_t^(r) B_t^(r)ᵀ,   y_t^(r) = h_t C_t^(r) + D x_t^(r).
    x [B,L,R,H,P], dt [B,L,H], A [H], Bm/Cm [B,L,R,G,N], D [H], h0 [B,H,P,N].
    Returns (y [B,L,R,H,P], final_state [B,H,P,N]) in fp64."""
    x, dt, A, Bm, Cm, D, h0 = (_f64(v) for v in (x, dt, A, Bm, Cm, D, h0))
    Bsz, L, R, H, P = x.shape
    G, N = Bm.shape[3], Bm.shape[4]
    assert dt.shape == (Bsz, L, H) and A.shape == (H,)
    assert Bm.shape == (Bsz, L, R, G, N) and Cm.shape == (Bsz, L, R, G, N)
    assert D is None or D.shape == (H,)
    assert h0 is None or h0.shape == (Bsz, H, P, N)
    y = np.empty((Bsz, L, R, H, P), np.float64)
    hT = np.empty((Bsz, H, P, N), np.float64)
    rc = _load().oracle_ssd_recurrent_mimo(Bsz, L, R, H, P, G, N, _ptr(x), _ptr(dt), _ptr(A), _ptr(Bm), _ptr(Cm),
                                           _ptr(D), _ptr(h0), _ptr(y), _ptr(hT))
    if rc:
        raise ValueError(f"oracle_ssd_recurrent_mimo failed ({rc})")
    return y, hT


def ssd_recurrent_heads(inputs, pairs):
    """Recurrence for selected (batch, head) pairs only, for spot checks of
    large problems.  ``inputs`` holds x, dt, A, Bm, Cm, D, init_state (any of
    the last two may be None).  Returns {(b, h): (y [L,P], final [P,N])}."""
    x, Bm = inputs["x"], inputs["Bm"]
    H = x.shape[2]
    G = Bm.shape[2]
    hpg = H // G
    res = {}
    for b, h in pairs:
        g = h // hpg
        D = inputs.get("D")
        h0 = inputs.get("init_state")
        y, hT = ssd_recurrent(
            x[b:b + 1, :, h:h + 1, :], inputs["dt"][b:b + 1, :, h:h + 1],
            inputs["A"][h:h + 1], Bm[b:b + 1, :, g:g + 1, :], inputs["Cm"][b:b + 1, :, g:g + 1, :],
            None if D is None else D[h:h + 1],
            None if h0 is None else h0[b:b + 1, h:h + 1])
        res[(b, h)] = (y[0, :, 0, :], hT[0, 0])
    return res


# ---------------------------------------------------------------------------
# The steps either side of the scan in a Mamba block (page "从 SSM 的长期记忆问题，
# 到 Mamba 的选择性机制与硬件感知扫描", the paragraphs on the selective SSM and
# on the Mamba block): Δ is produced from a per-head parameter plus the
# input-dependent part through τ_Δ, and the scan's output is gated.  Readings
# (the page names τ_Δ and "gating" without formulas): τ_Δ = softplus, the
# gate is y ← y · silu(z) = y · z / (1 + e^{−z}).
# ---------------------------------------------------------------------------
def softplus(v):
    """log(1 + e^v) in fp64 (numpy's logaddexp, exact to rounding for every v)."""
    return np.logaddexp(0.0, np.asarray(v, np.float64))


def silu(z):
    """z · σ(z) = z / (1 + e^{−z}) in fp64."""
    z = np.asarray(z, np.float64)
    return z / (1.0 + np.exp(-z))


def delta(dt, dt_bias=None, dt_softplus=False):
    """Δ = τ_Δ(dt + dt_bias): dt [B,L,H], dt_bias [H] or None."""
    d = _f64(dt)
    if dt_bias is not None:
        d = d + _f64(dt_bias)[None, None, :]
    return softplus(d) if dt_softplus else d


def ssd_fwd_ex(x, dt, A, Bm, Cm, D=None, h0=None, dt_bias=None, dt_softplus=False, z=None):
    """The recurrence on Δ = τ_Δ(dt + dt_bias), then y ← y · silu(z) when z is
    given.  Returns (y [B,L,H,P], final_state [B,H,P,N]) in fp64."""
    y, hT = ssd_recurrent(x, delta(dt, dt_bias, dt_softplus), A, Bm, Cm, D, h0)
    if z is not None:
        y = y * silu(_f64(z))
    return y, hT
