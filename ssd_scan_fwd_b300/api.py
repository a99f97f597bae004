"""Python binding of the SSD forward library.

Thin wrappers: validate torch tensors, allocate outputs and workspace with
torch on the tensors' device, pass raw pointers and the current CUDA stream
to the C ABI.  Every step of the scan runs in the library's CUDA kernels.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib

_IO = {torch.float32: _lib.SSD_DTYPE_F32, torch.bfloat16: _lib.SSD_DTYPE_BF16}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_tensor(name, t, dtype=None, shape=None, device=None):
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def make_args(x, dt, A, Bm, Cm, D=None, init_state=None, y=None, final_state=None, *,
              algo: str = "auto", chunk_size: int = 0) -> _lib.SsdFwdArgs:
    """Build the C argument struct after checking shapes, dtypes and devices."""
    if x.dim() != 4 or Bm.dim() != 4:
        raise ValueError("x must be [B,L,H,P] and Bm/Cm [B,L,G,N]")
    B, L, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    if x.dtype not in _IO:
        raise TypeError(f"x must be float32 or bfloat16, got {x.dtype}")
    dev = x.device
    _check_tensor("x", x, x.dtype, (B, L, H, P), dev)
    _check_tensor("dt", dt, torch.float32, (B, L, H), dev)
    _check_tensor("A", A, torch.float32, (H,), dev)
    _check_tensor("Bm", Bm, x.dtype, (B, L, G, N), dev)
    _check_tensor("Cm", Cm, x.dtype, (B, L, G, N), dev)
    _check_tensor("D", D, torch.float32, (H,), dev)
    _check_tensor("init_state", init_state, torch.float32, (B, H, P, N), dev)
    _check_tensor("y", y, x.dtype, (B, L, H, P), dev)
    _check_tensor("final_state", final_state, torch.float32, (B, H, P, N), dev)
    if algo not in _lib.ALGOS:
        raise ValueError(f"algo must be one of {list(_lib.ALGOS)}")
    a = _lib.SsdFwdArgs()
    a.batch, a.seqlen, a.nheads, a.headdim, a.ngroups, a.dstate = B, L, H, P, G, N
    a.io_dtype = _IO[x.dtype]
    a.algo = _lib.ALGOS[algo]
    a.chunk_size = int(chunk_size)
    a.x, a.dt, a.A, a.Bm, a.Cm = (t.data_ptr() for t in (x, dt, A, Bm, Cm))
    a.D = None if D is None else D.data_ptr()
    a.init_state = None if init_state is None else init_state.data_ptr()
    a.y = None if y is None else y.data_ptr()
    a.final_state = None if final_state is None else final_state.data_ptr()
    return a


def _stream_handle(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def workspace_size(args: _lib.SsdFwdArgs) -> int:
    n = _lib.lib().ssd_fwd_workspace_size(ctypes.byref(args))
    if n == ctypes.c_size_t(-1).value:
        raise _lib.SsdError(_lib.SSD_ERR_UNSUPPORTED, "ssd_fwd_workspace_size")
    return int(n)


def _check_device_status(workspace, device, where):
    """Raise SsdError when the call that used `workspace` recorded a device-side
    status other than SSD_OK (a bounded wait that gave up).  Synchronises the
    device's current stream."""
    if workspace is None:
        return
    s = _lib.lib().ssd_workspace_status(ctypes.c_void_p(workspace.data_ptr()), _stream_handle(device))
    _lib.check(s, where)


def ssd_fwd(x, dt, A, Bm, Cm, D=None, init_state=None, *, return_final_state: bool = True,
            algo: str = "auto", chunk_size: int = 0, y=None, final_state=None, workspace=None,
            check_status: bool = False):
    """SSD selective-scan forward pass on the GPU.

    x [B,L,H,P] (fp32/bf16), dt [B,L,H] fp32 (Δ ≥ 0), A [H] fp32 (≤ 0),
    Bm/Cm [B,L,G,N] (x's dtype), D [H] fp32 or None, init_state [B,H,P,N] fp32
    or None.  Returns (y, final_state) -- final_state is None when not asked
    for.  Outputs/workspace may be passed in to avoid allocation.
    algo: "auto" (the fused kernel where it applies: bf16, P=64, N=128),
    "fused" or "chunked".  chunk_size (chunked path): 32, 64 or 128; 0 picks
    128 where the tensor-core chunk kernels apply (bf16, P=64, N in
    {16, 64, 128, 256}), else 64.
    check_status: synchronise after the call and raise SsdError if one of its
    kernels' bounded device-side waits gave up (SSD_ERR_TIMEOUT: the outputs
    are then unspecified).  Off by default, as it costs a synchronisation.
    """
    if not x.is_cuda:
        raise ValueError("ssd_fwd runs on CUDA tensors only")
    B, L, H, P = x.shape
    N = Bm.shape[3]
    if y is None:
        y = torch.empty_like(x)
    if final_state is None and return_final_state:
        final_state = torch.empty(B, H, P, N, dtype=torch.float32, device=x.device)
    args = make_args(x, dt, A, Bm, Cm, D, init_state, y, final_state, algo=algo, chunk_size=chunk_size)
    need = workspace_size(args)
    if need > 0:
        if workspace is None or workspace.numel() * workspace.element_size() < need:
            workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
        args.workspace = workspace.data_ptr()
        args.workspace_bytes = workspace.numel() * workspace.element_size()
    _lib.check(_lib.lib().ssd_fwd(ctypes.byref(args), _stream_handle(x.device)), "ssd_fwd")
    if check_status and need > 0:
        _check_device_status(workspace, x.device, "ssd_fwd")
    return y, final_state


def ssd_fwd_ex(x, dt, A, Bm, Cm, D=None, init_state=None, *, dt_bias=None, dt_softplus: bool = False,
               z=None, return_final_state: bool = True, algo: str = "auto", chunk_size: int = 0,
               y=None, final_state=None, workspace=None, check_status: bool = False):
    """ssd_fwd with the steps around the scan in a Mamba block: Δ =
    softplus(dt + dt_bias) (or dt + dt_bias without softplus) and the output
    gate y · silu(z).  dt is the raw [B,L,H] fp32 input, dt_bias [H] fp32 or
    None, z [B,L,H,P] in x's dtype or None.  Returns (y, final_state)."""
    if not x.is_cuda:
        raise ValueError("ssd_fwd_ex runs on CUDA tensors only")
    B, L, H, P = x.shape
    N = Bm.shape[3]
    _check_tensor("dt_bias", dt_bias, torch.float32, (H,), x.device)
    _check_tensor("z", z, x.dtype, (B, L, H, P), x.device)
    if y is None:
        y = torch.empty_like(x)
    if final_state is None and return_final_state:
        final_state = torch.empty(B, H, P, N, dtype=torch.float32, device=x.device)
    ex = _lib.SsdFwdExArgs()
    ex.base = make_args(x, dt, A, Bm, Cm, D, init_state, y, final_state, algo=algo, chunk_size=chunk_size)
    ex.dt_bias = None if dt_bias is None else dt_bias.data_ptr()
    ex.dt_softplus = 1 if dt_softplus else 0
    ex.reserved = 0
    ex.z = None if z is None else z.data_ptr()
    need = workspace_size(ex.base)
    if need > 0:
        if workspace is None or workspace.numel() * workspace.element_size() < need:
            workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
        ex.base.workspace = workspace.data_ptr()
        ex.base.workspace_bytes = workspace.numel() * workspace.element_size()
    _lib.check(_lib.lib().ssd_fwd_ex(ctypes.byref(ex), _stream_handle(x.device)), "ssd_fwd_ex")
    if check_status and need > 0:
        _check_device_status(workspace, x.device, "ssd_fwd_ex")
    return y, final_state


def ssd_fwd_host(x, dt, A, Bm, Cm, D=None, init_state=None, *, device=None, algo: str = "auto",
                 chunk_size: int = 0, y=None, final_state=None, workspace=None, return_final_state: bool = True):
    """The forward pass on host (CPU) tensors: the library copies them to the
    GPU, runs the pass and copies y and final_state back, overlapping the
    copies of one group of batch rows with the compute of another.  Pinned
    CPU tensors let the copies overlap.  Returns (y, final_state) as CPU
    tensors, ready once the device's current stream is synchronised."""
    if x.is_cuda:
        raise ValueError("ssd_fwd_host takes host (CPU) tensors")
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    B, L, H, P = x.shape
    N = Bm.shape[3]
    if y is None:
        y = torch.empty(x.shape, dtype=x.dtype).pin_memory()
    if final_state is None and return_final_state:
        final_state = torch.empty(B, H, P, N, dtype=torch.float32).pin_memory()
    args = make_args(x, dt, A, Bm, Cm, D, init_state, y, final_state, algo=algo, chunk_size=chunk_size)
    need = _lib.lib().ssd_fwd_host_workspace_size(ctypes.byref(args))
    if need == ctypes.c_size_t(-1).value:
        raise _lib.SsdError(_lib.SSD_ERR_UNSUPPORTED, "ssd_fwd_host_workspace_size")
    if need > 0:
        if workspace is None or workspace.numel() * workspace.element_size() < need:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        args.workspace = workspace.data_ptr()
        args.workspace_bytes = workspace.numel() * workspace.element_size()
    _lib.check(_lib.lib().ssd_fwd_host(ctypes.byref(args), _stream_handle(dev)), "ssd_fwd_host")
    return y, final_state


# ---------------------------------------------------------------------------
# The four steps of the chunked path, one call each.
# ---------------------------------------------------------------------------
def _step_args(x, dt, A, Bm, Cm, D, init_state, y, final_state):
    return make_args(x, dt, A, Bm, Cm, D, init_state, y, final_state)


def chunk_cumsum(x, dt, A, Bm, Cm, chunk: int):
    """Returns (dA_cs, dt_chunked), both [B,H,nc,chunk] fp32."""
    B, L, H, _ = x.shape
    nc = (L + chunk - 1) // chunk
    dA = torch.empty(B, H, nc, chunk, dtype=torch.float32, device=x.device)
    dtc = torch.empty_like(dA)
    a = _step_args(x, dt, A, Bm, Cm, None, None, None, None)
    _lib.check(_lib.lib().ssd_chunk_cumsum(ctypes.byref(a), chunk, _ptr(dA), _ptr(dtc),
                                           _stream_handle(x.device)), "ssd_chunk_cumsum")
    return dA, dtc


def chunk_state(x, dt, A, Bm, Cm, dA_cs, dt_chunked, chunk: int):
    """Returns the chunk states [B,nc,H,P,N] fp32."""
    B, L, H, P = x.shape
    N = Bm.shape[3]
    nc = (L + chunk - 1) // chunk
    st = torch.empty(B, nc, H, P, N, dtype=torch.float32, device=x.device)
    a = _step_args(x, dt, A, Bm, Cm, None, None, None, None)
    _lib.check(_lib.lib().ssd_chunk_state(ctypes.byref(a), chunk, _ptr(dA_cs), _ptr(dt_chunked),
                                          _ptr(st), _stream_handle(x.device)), "ssd_chunk_state")
    return st


def state_passing(x, dt, A, Bm, Cm, dA_cs, states, chunk: int, init_state=None, final_state=None):
    """In place: states[c] becomes the state entering chunk c; writes final_state."""
    a = _step_args(x, dt, A, Bm, Cm, None, init_state, None, final_state)
    _lib.check(_lib.lib().ssd_state_passing(ctypes.byref(a), chunk, _ptr(dA_cs), _ptr(states),
                                            _stream_handle(x.device)), "ssd_state_passing")
    return states


def chunk_scan(x, dt, A, Bm, Cm, D, dA_cs, dt_chunked, states, chunk: int, y=None):
    """Returns y [B,L,H,P] in x's dtype."""
    if y is None:
        y = torch.empty_like(x)
    a = _step_args(x, dt, A, Bm, Cm, D, None, y, None)
    _lib.check(_lib.lib().ssd_chunk_scan(ctypes.byref(a), chunk, _ptr(dA_cs), _ptr(dt_chunked),
                                         _ptr(states), _stream_handle(x.device)), "ssd_chunk_scan")
    return y


# ---------------------------------------------------------------------------
# Recurrent step (inference): one token per (batch row, head), state in place.
# ---------------------------------------------------------------------------
def make_step_args(x, dt, A, Bm, Cm, D, state, y) -> _lib.SsdStepArgs:
    """Build the C argument struct of ssd_step after checking the tensors."""
    if x.dim() != 3 or Bm.dim() != 3:
        raise ValueError("x must be [B,H,P] and Bm/Cm [B,G,N]")
    B, H, P = x.shape
    G, N = Bm.shape[1], Bm.shape[2]
    if x.dtype not in _IO:
        raise TypeError(f"x must be float32 or bfloat16, got {x.dtype}")
    dev = x.device
    _check_tensor("x", x, x.dtype, (B, H, P), dev)
    _check_tensor("dt", dt, torch.float32, (B, H), dev)
    _check_tensor("A", A, torch.float32, (H,), dev)
    _check_tensor("Bm", Bm, x.dtype, (B, G, N), dev)
    _check_tensor("Cm", Cm, x.dtype, (B, G, N), dev)
    _check_tensor("D", D, torch.float32, (H,), dev)
    _check_tensor("state", state, torch.float32, (B, H, P, N), dev)
    _check_tensor("y", y, x.dtype, (B, H, P), dev)
    a = _lib.SsdStepArgs()
    a.batch, a.nheads, a.headdim, a.ngroups, a.dstate = B, H, P, G, N
    a.io_dtype = _IO[x.dtype]
    a.reserved = 0
    a.x, a.dt, a.A, a.Bm, a.Cm, a.state, a.y = (t.data_ptr() for t in (x, dt, A, Bm, Cm, state, y))
    a.D = None if D is None else D.data_ptr()
    return a


def ssd_step(x, dt, A, Bm, Cm, D, state, *, y=None):
    """One recurrent step on the GPU: updates `state` [B,H,P,N] fp32 in place
    and returns y [B,H,P] (x's dtype).  x [B,H,P], dt [B,H] fp32, A [H] fp32,
    Bm/Cm [B,G,N] (x's dtype), D [H] fp32 or None."""
    if not x.is_cuda:
        raise ValueError("ssd_step runs on CUDA tensors only")
    if y is None:
        y = torch.empty_like(x)
    args = make_step_args(x, dt, A, Bm, Cm, D, state, y)
    _lib.check(_lib.lib().ssd_step(ctypes.byref(args), _stream_handle(x.device)), "ssd_step")
    return y


def ssd_bwd(x, dt, A, Bm, Cm, D=None, init_state=None, *, dy, dfinal=None, workspace=None,
            chunk_size: int = 0):
    """Gradients of  Σ dy ⊙ y + Σ dfinal ⊙ final_state  through ssd_fwd (same
    inputs; dt is Δ).  dy [B,L,H,P] in x's dtype, dfinal [B,H,P,N] fp32 or
    None.  Returns a dict: dx [B,L,H,P] and dBm, dCm [B,L,G,N] in x's dtype;
    ddt [B,L,H], dA [H], dD [H] (None when D is None), dinit [B,H,P,N] fp32.
    chunk_size: 0 (default: 128 on the tensor-core path, else 64), 64, or 128
    (bf16, headdim 64, dstate 128)."""
    if not x.is_cuda:
        raise ValueError("ssd_bwd runs on CUDA tensors only")
    B, L, H, P = x.shape
    G, N = Bm.shape[2], Bm.shape[3]
    dev = x.device
    _check_tensor("dy", dy, x.dtype, (B, L, H, P), dev)
    _check_tensor("dfinal", dfinal, torch.float32, (B, H, P, N), dev)
    out = {
        "dx": torch.empty_like(x),
        "ddt": torch.empty(B, L, H, dtype=torch.float32, device=dev),
        "dA": torch.empty(H, dtype=torch.float32, device=dev),
        "dBm": torch.empty_like(Bm),
        "dCm": torch.empty_like(Cm),
        "dD": None if D is None else torch.empty(H, dtype=torch.float32, device=dev),
        "dinit": torch.empty(B, H, P, N, dtype=torch.float32, device=dev),
    }
    a = _lib.SsdBwdArgs()
    a.fwd = make_args(x, dt, A, Bm, Cm, D, init_state, chunk_size=chunk_size)
    a.dy = dy.data_ptr()
    a.dfinal = None if dfinal is None else dfinal.data_ptr()
    for k in ("dx", "ddt", "dA", "dBm", "dCm", "dD", "dinit"):
        setattr(a, k, None if out[k] is None else out[k].data_ptr())
    lib = _lib.lib()
    need = lib.ssd_bwd_workspace_size(ctypes.byref(a))
    if need == ctypes.c_size_t(-1).value:
        _lib.check(lib.ssd_bwd(ctypes.byref(a), _stream_handle(dev)), "ssd_bwd")
    if need > 0:
        if workspace is None or workspace.numel() * workspace.element_size() < need:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        a.fwd.workspace = workspace.data_ptr()
        a.fwd.workspace_bytes = workspace.numel() * workspace.element_size()
    _lib.check(lib.ssd_bwd(ctypes.byref(a), _stream_handle(dev)), "ssd_bwd")
    return out


def ssd_fwd_rot(x, dt, theta, A, Bm, Cm, D=None, init_state=None, *, return_final_state: bool = True,
                chunk_size: int = 0, algo: str = "auto", y=None, workspace=None):
    """The forward pass with the complex (rotational) decay
    α_t = exp(Δ_t A)(cos θ_t + i sin θ_t): complex state, y_t = Re(h_t) C_t + D x_t.
    theta [B,L,H] fp32; init_state None or a pair (re, im) of [B,H,P,N] fp32
    tensors (either may be None).  Returns (y, (final_re, final_im)) -- the
    pair is None when not asked for.  algo "auto" runs the fused kernel (state
    on chip) for bf16, P=64, N=128 at chunk_size 0 or 128 and the chunked path
    otherwise; "fused" or "chunked" force one.  chunk_size (chunked path): 32,
    64 or 128; 0 picks 128 where the tensor-core chunk kernels apply (bf16,
    P=64, N in {16, 64, 128, 256}), else 64."""
    if not x.is_cuda:
        raise ValueError("ssd_fwd_rot runs on CUDA tensors only")
    B, L, H, P = x.shape
    N = Bm.shape[3]
    dev = x.device
    _check_tensor("theta", theta, torch.float32, (B, L, H), dev)
    init_re, init_im = (None, None) if init_state is None else init_state
    _check_tensor("init_state_im", init_im, torch.float32, (B, H, P, N), dev)
    if y is None:
        y = torch.empty_like(x)
    fr = fi = None
    if return_final_state:
        fr = torch.empty(B, H, P, N, dtype=torch.float32, device=dev)
        fi = torch.empty(B, H, P, N, dtype=torch.float32, device=dev)
    a = _lib.SsdFwdRotArgs()
    a.base = make_args(x, dt, A, Bm, Cm, D, init_re, y, fr, algo=algo, chunk_size=chunk_size)
    a.theta = theta.data_ptr()
    a.init_state_im = None if init_im is None else init_im.data_ptr()
    a.final_state_im = None if fi is None else fi.data_ptr()
    lib = _lib.lib()
    need = lib.ssd_fwd_rot_workspace_size(ctypes.byref(a))
    if need == ctypes.c_size_t(-1).value:
        _lib.check(lib.ssd_fwd_rot(ctypes.byref(a), _stream_handle(dev)), "ssd_fwd_rot")
    if need > 0:
        if workspace is None or workspace.numel() * workspace.element_size() < need:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        a.base.workspace = workspace.data_ptr()
        a.base.workspace_bytes = workspace.numel() * workspace.element_size()
    _lib.check(lib.ssd_fwd_rot(ctypes.byref(a), _stream_handle(dev)), "ssd_fwd_rot")
    return y, (None if fr is None else (fr, fi))


def ssd_fwd_mimo(x, dt, A, Bm, Cm, D=None, init_state=None, *, return_final_state: bool = True, y=None,
                 final_state=None, workspace=None):
    """The forward pass with retrieval rank R (MIMO): per token R ranks with
    their own x, B, C share the token's decay; the update writes all R values
    and each rank reads its own output (y_t^(r) = h_t C_t^(r) + D x_t^(r)).
    x [B,L,R,H,P] bf16, dt [B,L,H] fp32 (one Δ per token), A [H], Bm/Cm
    [B,L,R,G,N] bf16, D [H] or None, init_state [B,H,P,N] fp32 or None.
    R in {1, 2, 4, 8}; headdim 64, dstate 16, 64, 128 or 256 (fused kernel).
    Returns (y [B,L,R,H,P], final_state)."""
    if not x.is_cuda:
        raise ValueError("ssd_fwd_mimo runs on CUDA tensors only")
    if x.dim() != 5 or Bm.dim() != 5:
        raise ValueError("x must be [B,L,R,H,P] and Bm/Cm [B,L,R,G,N]")
    B, L, R, H, P = x.shape
    G, N = Bm.shape[3], Bm.shape[4]
    dev = x.device
    _check_tensor("dt", dt, torch.float32, (B, L, H), dev)
    _check_tensor("Bm", Bm, torch.bfloat16, (B, L, R, G, N), dev)
    _check_tensor("Cm", Cm, torch.bfloat16, (B, L, R, G, N), dev)
    if y is None:
        y = torch.empty_like(x)
    _check_tensor("y", y, torch.bfloat16, tuple(x.shape), dev)
    if final_state is None and return_final_state:
        final_state = torch.empty(B, H, P, N, dtype=torch.float32, device=dev)
    _check_tensor("x", x, torch.bfloat16, (B, L, R, H, P), dev)
    _check_tensor("A", A, torch.float32, (H,), dev)
    _check_tensor("D", D, torch.float32, (H,), dev)
    _check_tensor("init_state", init_state, torch.float32, (B, H, P, N), dev)
    _check_tensor("final_state", final_state, torch.float32, (B, H, P, N), dev)
    args = _lib.SsdFwdMimoArgs()
    a = args.base
    a.batch, a.seqlen, a.nheads, a.headdim, a.ngroups, a.dstate = B, L, H, P, G, N
    a.io_dtype = _IO[x.dtype]
    a.algo = _lib.ALGOS["auto"]
    a.chunk_size = 0
    a.x, a.dt, a.A, a.Bm, a.Cm, a.y = (t.data_ptr() for t in (x, dt, A, Bm, Cm, y))
    a.D = None if D is None else D.data_ptr()
    a.init_state = None if init_state is None else init_state.data_ptr()
    a.final_state = None if final_state is None else final_state.data_ptr()
    args.rank = R
    lib = _lib.lib()
    need = lib.ssd_fwd_mimo_workspace_size(ctypes.byref(args))
    if need == ctypes.c_size_t(-1).value:
        _lib.check(lib.ssd_fwd_mimo(ctypes.byref(args), _stream_handle(dev)), "ssd_fwd_mimo")
    if need > 0:
        if workspace is None or workspace.numel() * workspace.element_size() < need:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        args.base.workspace = workspace.data_ptr()
        args.base.workspace_bytes = workspace.numel() * workspace.element_size()
    _lib.check(lib.ssd_fwd_mimo(ctypes.byref(args), _stream_handle(dev)), "ssd_fwd_mimo")
    return y, final_state
