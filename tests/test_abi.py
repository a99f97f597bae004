"""Host-side checks of the C ABI (no GPU needed).

The library must load, export every function include/ssd.h declares, and
reject bad arguments on the host before anything is launched.  Fake device
pointers are used where a call must fail validation before touching CUDA.
"""
import ctypes
import re

import pytest

from ssd_scan_fwd_b300 import _lib


def _declared_functions():
    text = open(_lib.HEADER_PATH).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(ssd_[a-z0-9_]+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_expected_entry_points():
    names = _declared_functions()
    for n in ["ssd_fwd", "ssd_fwd_workspace_size", "ssd_status_string", "ssd_chunk_cumsum",
              "ssd_chunk_state", "ssd_state_passing", "ssd_chunk_scan"]:
        assert n in names


def test_library_exports_every_declared_symbol():
    L = ctypes.CDLL(_lib.LIB_PATH)
    for n in _declared_functions():
        assert hasattr(L, n), n
    assert set(_declared_functions()) == set(_lib.SIGNATURES)


def test_abi_version_and_status_strings():
    L = _lib.lib()
    assert L.ssd_abi_version() == 1
    for s in range(6):
        assert L.ssd_status_string(s).decode().startswith("SSD_")
    assert b"unknown" in L.ssd_status_string(99)


def test_args_struct_layout_matches_header(tmp_path):
    """The ctypes struct must have the C struct's size and field offsets
    (checked by compiling a probe against include/ssd.h with gcc)."""
    import os
    import subprocess
    fields = [f for f, _ in _lib.SsdFwdArgs._fields_]
    src = tmp_path / "probe.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "ssd.h"\nint main(void){\n'
                   '  printf("%zu\\n", sizeof(ssd_fwd_args));\n' +
                   "".join(f'  printf("%zu\\n", offsetof(ssd_fwd_args, {f}));\n' for f in fields) +
                   "  return 0;\n}\n")
    exe = tmp_path / "probe"
    inc = os.path.dirname(_lib.HEADER_PATH)
    subprocess.run(["gcc", "-I", inc, str(src), "-o", str(exe)], check=True)
    out = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert out[0] == ctypes.sizeof(_lib.SsdFwdArgs)
    assert out[1:] == [getattr(_lib.SsdFwdArgs, f).offset for f in fields]


FAKE = 1 << 40  # an aligned address that is never dereferenced


def _args(B=2, L=100, H=4, P=64, G=2, N=128, io=1, algo=1, chunk=64, fake=True):
    a = _lib.SsdFwdArgs()
    a.batch, a.seqlen, a.nheads, a.headdim, a.ngroups, a.dstate = B, L, H, P, G, N
    a.io_dtype, a.algo, a.chunk_size = io, algo, chunk
    if fake:
        base = FAKE
        for name in ["x", "dt", "A", "Bm", "Cm", "D", "init_state", "y", "final_state"]:
            setattr(a, name, base)
            base += 1 << 32
    return a


def _fwd(a):
    L = _lib.lib()
    return L.ssd_fwd(ctypes.byref(a), None), L.ssd_last_error_message().decode()


def test_workspace_size_chunked():
    a = _args(B=2, L=100, H=4, P=64, G=2, N=128, chunk=64)
    nc = 2
    cs = 2 * 4 * nc * 64 * 4
    st = 2 * nc * 4 * 64 * 128 * 4
    al = lambda v: (v + 255) // 256 * 256  # noqa: E731
    # a 256-byte status word first, then the in-chunk sums, Δ and the chunk states
    assert _lib.lib().ssd_fwd_workspace_size(ctypes.byref(a)) == 256 + 2 * al(cs) + al(st)


@pytest.mark.parametrize("N", [16, 64, 128, 256])
def test_workspace_size_chunked_default_chunk(N):
    """algo chunked, chunk_size 0: chunk 128 with bf16 copies of the entering
    states where the tensor-core chunk states and outputs apply (bf16,
    headdim 64), chunk 64 and fp32 states only otherwise."""
    al = lambda v: (v + 255) // 256 * 256  # noqa: E731
    size = lambda a: _lib.lib().ssd_fwd_workspace_size(ctypes.byref(a))  # noqa: E731

    def expect(Q, P, bf):
        nc = (300 + Q - 1) // Q
        st = 2 * nc * 4 * P * N
        return 256 + 2 * al(2 * 4 * nc * Q * 4) + al(st * 4) + (al(st * 2) if bf else 0)

    assert size(_args(B=2, L=300, H=4, P=64, G=2, N=N, io=1, algo=1, chunk=0)) == expect(128, 64, True)
    assert size(_args(B=2, L=300, H=4, P=64, G=2, N=N, io=1, algo=1, chunk=128)) == expect(128, 64, True)
    assert size(_args(B=2, L=300, H=4, P=64, G=2, N=N, io=1, algo=1, chunk=64)) == expect(64, 64, False)
    assert size(_args(B=2, L=300, H=4, P=64, G=2, N=N, io=0, algo=1, chunk=0)) == expect(64, 64, False)
    assert size(_args(B=2, L=300, H=4, P=32, G=2, N=N, io=1, algo=1, chunk=0)) == expect(64, 32, False)


@pytest.mark.parametrize("field,value,status", [
    ("ngroups", 3, _lib.SSD_ERR_INVALID_ARG),       # H % G != 0
    ("headdim", 0, _lib.SSD_ERR_INVALID_ARG),
    ("headdim", 512, _lib.SSD_ERR_UNSUPPORTED),
    ("dstate", 300, _lib.SSD_ERR_UNSUPPORTED),
    ("io_dtype", 7, _lib.SSD_ERR_INVALID_ARG),
    ("chunk_size", 48, _lib.SSD_ERR_UNSUPPORTED),
    ("algo", 9, _lib.SSD_ERR_INVALID_ARG),
    ("batch", -1, _lib.SSD_ERR_INVALID_ARG),
])
def test_bad_shapes_rejected(field, value, status):
    a = _args()
    setattr(a, field, value)
    s, msg = _fwd(a)
    assert s == status and msg
    assert _lib.lib().ssd_fwd_workspace_size(ctypes.byref(a)) == ctypes.c_size_t(-1).value


@pytest.mark.parametrize("field", ["x", "dt", "A", "Bm", "Cm", "y"])
def test_missing_required_pointer(field):
    a = _args()
    setattr(a, field, None)
    s, msg = _fwd(a)
    assert s == _lib.SSD_ERR_INVALID_ARG and field in msg


@pytest.mark.parametrize("field", ["x", "dt", "Bm", "D", "init_state", "final_state"])
def test_misaligned_pointer(field):
    a = _args()
    setattr(a, field, getattr(a, field) + 4)
    s, msg = _fwd(a)
    assert s == _lib.SSD_ERR_INVALID_ARG and "aligned" in msg


def test_output_overlapping_input_rejected():
    a = _args()
    a.y = a.x + 64
    s, msg = _fwd(a)
    assert s == _lib.SSD_ERR_INVALID_ARG and "overlaps" in msg


def test_in_place_state_allowed_by_validation():
    a = _args()
    a.final_state = a.init_state
    s, msg = _fwd(a)  # passes pointer checks, then stops at the missing workspace
    assert s == _lib.SSD_ERR_WORKSPACE


def test_workspace_missing_or_small():
    a = _args()
    s, _ = _fwd(a)
    assert s == _lib.SSD_ERR_WORKSPACE
    a.workspace = FAKE + (1 << 38)
    a.workspace_bytes = 1024
    s, msg = _fwd(a)
    assert s == _lib.SSD_ERR_WORKSPACE and "needed" in msg


def test_workspace_misaligned():
    a = _args()
    a.workspace = FAKE + (1 << 38) + 16
    a.workspace_bytes = 1 << 30
    s, msg = _fwd(a)
    assert s == _lib.SSD_ERR_INVALID_ARG and "256" in msg


def test_empty_batch_is_a_no_op():
    a = _args(B=0)
    s, _ = _fwd(a)
    assert s == _lib.SSD_OK


def test_fused_request_unsupported_for_fp32():
    a = _args(io=0, algo=2, chunk=0)
    s, msg = _fwd(a)
    assert s == _lib.SSD_ERR_UNSUPPORTED and "fused" in msg


def test_step_entry_points_validate():
    L = _lib.lib()
    a = _args()
    assert L.ssd_chunk_cumsum(ctypes.byref(a), 64, None, FAKE, None) == _lib.SSD_ERR_INVALID_ARG
    assert L.ssd_chunk_cumsum(ctypes.byref(a), 0, FAKE, FAKE, None) == _lib.SSD_ERR_INVALID_ARG
    assert L.ssd_chunk_state(ctypes.byref(a), 64, FAKE, FAKE, FAKE + 8, None) == _lib.SSD_ERR_INVALID_ARG
    assert L.ssd_state_passing(ctypes.byref(a), 96, FAKE, FAKE, None) == _lib.SSD_ERR_UNSUPPORTED
    assert L.ssd_chunk_scan(None, 64, FAKE, FAKE, FAKE, None) == _lib.SSD_ERR_INVALID_ARG


def test_step_struct_layout_matches_header(tmp_path):
    """ssd_step_args: the ctypes mirror has the C struct's size and offsets."""
    import os
    import subprocess
    fields = [f for f, _ in _lib.SsdStepArgs._fields_]
    src = tmp_path / "probe_step.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "ssd.h"\nint main(void){\n'
                   '  printf("%zu\\n", sizeof(ssd_step_args));\n' +
                   "".join(f'  printf("%zu\\n", offsetof(ssd_step_args, {f}));\n' for f in fields) +
                   "  return 0;\n}\n")
    exe = tmp_path / "probe_step"
    subprocess.run(["gcc", "-I", os.path.dirname(_lib.HEADER_PATH), str(src), "-o", str(exe)], check=True)
    out = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert out[0] == ctypes.sizeof(_lib.SsdStepArgs)
    assert out[1:] == [getattr(_lib.SsdStepArgs, f).offset for f in fields]


def _step_args(B=2, H=4, P=64, G=2, N=128, io=1, fake=True):
    a = _lib.SsdStepArgs()
    a.batch, a.nheads, a.headdim, a.ngroups, a.dstate = B, H, P, G, N
    a.io_dtype, a.reserved = io, 0
    if fake:
        base = FAKE
        for name in ["x", "dt", "A", "Bm", "Cm", "D", "state", "y"]:
            setattr(a, name, base)
            base += 1 << 32
    return a


def _step(a):
    L = _lib.lib()
    return L.ssd_step(ctypes.byref(a), None), L.ssd_last_error_message().decode()


@pytest.mark.parametrize("field,value,status", [
    ("ngroups", 3, _lib.SSD_ERR_INVALID_ARG),
    ("headdim", 0, _lib.SSD_ERR_INVALID_ARG),
    ("headdim", 257, _lib.SSD_ERR_UNSUPPORTED),
    ("dstate", 300, _lib.SSD_ERR_UNSUPPORTED),
    ("io_dtype", 5, _lib.SSD_ERR_INVALID_ARG),
    ("reserved", 1, _lib.SSD_ERR_INVALID_ARG),
    ("batch", -1, _lib.SSD_ERR_INVALID_ARG),
])
def test_step_bad_shapes_rejected(field, value, status):
    a = _step_args()
    setattr(a, field, value)
    s, msg = _step(a)
    assert s == status and msg


@pytest.mark.parametrize("field", ["x", "dt", "A", "Bm", "Cm", "state", "y"])
def test_step_missing_pointer(field):
    a = _step_args()
    setattr(a, field, None)
    s, _ = _step(a)
    assert s == _lib.SSD_ERR_INVALID_ARG


def test_step_misaligned_and_overlap():
    a = _step_args()
    a.state = FAKE + (7 << 32) + 4
    assert _step(a)[0] == _lib.SSD_ERR_INVALID_ARG
    a = _step_args()
    a.y = a.x
    s, msg = _step(a)
    assert s == _lib.SSD_ERR_INVALID_ARG and "overlaps" in msg
    a = _step_args()
    a.state = a.Bm
    s, msg = _step(a)
    assert s == _lib.SSD_ERR_INVALID_ARG and "overlaps" in msg


def test_step_empty_batch_is_a_no_op():
    a = _step_args(B=0, fake=False)
    assert _step(a)[0] == _lib.SSD_OK


def test_fwd_ex_struct_layout_matches_header(tmp_path):
    import os
    import subprocess
    fields = [f for f, _ in _lib.SsdFwdExArgs._fields_]
    src = tmp_path / "probe_ex.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "ssd.h"\nint main(void){\n'
                   '  printf("%zu\\n", sizeof(ssd_fwd_ex_args));\n' +
                   "".join(f'  printf("%zu\\n", offsetof(ssd_fwd_ex_args, {f}));\n' for f in fields) +
                   "  return 0;\n}\n")
    exe = tmp_path / "probe_ex"
    subprocess.run(["gcc", "-I", os.path.dirname(_lib.HEADER_PATH), str(src), "-o", str(exe)], check=True)
    out = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert out[0] == ctypes.sizeof(_lib.SsdFwdExArgs)
    assert out[1:] == [getattr(_lib.SsdFwdExArgs, f).offset for f in fields]


def _ex_args():
    ex = _lib.SsdFwdExArgs()
    ex.base = _args()
    ex.dt_bias = FAKE + (20 << 32)
    ex.z = FAKE + (21 << 32)
    ex.dt_softplus, ex.reserved = 1, 0
    return ex


def _fwd_ex(ex):
    L = _lib.lib()
    return L.ssd_fwd_ex(ctypes.byref(ex), None), L.ssd_last_error_message().decode()


def test_fwd_ex_validation():
    ex = _ex_args()
    ex.reserved = 3
    assert _fwd_ex(ex)[0] == _lib.SSD_ERR_INVALID_ARG
    ex = _ex_args()
    ex.dt_softplus = 2
    assert _fwd_ex(ex)[0] == _lib.SSD_ERR_INVALID_ARG
    ex = _ex_args()
    ex.z = ex.base.y  # gate operand overlapping the output
    s, msg = _fwd_ex(ex)
    assert s == _lib.SSD_ERR_INVALID_ARG and "overlaps" in msg
    ex = _ex_args()
    ex.dt_bias = FAKE + (20 << 32) + 4
    s, msg = _fwd_ex(ex)
    assert s == _lib.SSD_ERR_INVALID_ARG and "aligned" in msg
    ex = _ex_args()
    ex.base.headdim = 0
    assert _fwd_ex(ex)[0] == _lib.SSD_ERR_INVALID_ARG


def test_fwd_ex_workspace_equals_base():
    ex = _ex_args()
    L = _lib.lib()
    assert L.ssd_fwd_ex_workspace_size(ctypes.byref(ex)) == L.ssd_fwd_workspace_size(ctypes.byref(ex.base))


def test_host_workspace_size():
    L = _lib.lib()
    a = _args(B=4, L=1000, H=8, P=64, G=1, N=128, io=1, algo=0, chunk=0)
    n4 = L.ssd_fwd_host_workspace_size(ctypes.byref(a))
    assert 0 < n4 < (1 << 40)
    a.batch = 0
    assert L.ssd_fwd_host_workspace_size(ctypes.byref(a)) == 0
    a.batch, a.ngroups = 4, 3
    assert L.ssd_fwd_host_workspace_size(ctypes.byref(a)) == ctypes.c_size_t(-1).value


# ---------------------------------------------------------------- backward pass
def test_bwd_struct_layout_matches_header(tmp_path):
    import os
    import subprocess
    fields = [f for f, _ in _lib.SsdBwdArgs._fields_]
    src = tmp_path / "probe_bwd.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "ssd.h"\nint main(void){\n'
                   '  printf("%zu\\n", sizeof(ssd_bwd_args));\n' +
                   "".join(f'  printf("%zu\\n", offsetof(ssd_bwd_args, {f}));\n' for f in fields) +
                   "  return 0;\n}\n")
    exe = tmp_path / "probe_bwd"
    subprocess.run(["gcc", "-I", os.path.dirname(_lib.HEADER_PATH), str(src), "-o", str(exe)], check=True)
    out = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert out[0] == ctypes.sizeof(_lib.SsdBwdArgs)
    assert out[1:] == [getattr(_lib.SsdBwdArgs, f).offset for f in fields]


def _bwd_args(**kw):
    b = _lib.SsdBwdArgs()
    b.fwd = _args(**kw)
    b.fwd.y = None
    b.fwd.final_state = None
    base = FAKE + (40 << 32)
    for name in ["dy", "dfinal", "dx", "ddt", "dA", "dBm", "dCm", "dD", "dinit"]:
        setattr(b, name, base)
        base += 1 << 32
    return b


def _bwd(b):
    L = _lib.lib()
    return L.ssd_bwd(ctypes.byref(b), None), L.ssd_last_error_message().decode()


def test_bwd_workspace_size():
    al = lambda v: (v + 255) // 256 * 256  # noqa: E731

    def expect(Q, B=2, L=100, H=4, P=64, G=2, N=128):
        nc = (L + Q - 1) // Q
        cs = al(B * H * nc * Q * 4)
        st = al(B * nc * H * P * N * 4)
        bc = al(B * L * G * N * 4)
        # a 256-byte status word first; fp32 per-chunk states twice, or once
        # on the tensor-core path (chunk 128), whose state walks keep them on
        # chip and write only bf16 copies, plus a flag and an fp32 state per
        # walk and head for the walks' hand-offs (2 · B · G · ceil(H / G / 2)
        # walks of head pairs)
        if Q != 128:
            return 256 + 2 * cs + 2 * st + 2 * bc
        nw = 2 * (2 * B * G * ((H // G + 1) // 2))
        return 256 + 2 * cs + st + 2 * bc + al(nw * 4) + al(nw * P * N * 4)

    size = lambda b: _lib.lib().ssd_bwd_workspace_size(ctypes.byref(b))  # noqa: E731
    # bf16, headdim 64, dstate 128: chunk 0 picks the tensor-core chunk 128; 64 and 128 on request
    assert size(_bwd_args(B=2, L=100, H=4, P=64, G=2, N=128, chunk=0)) == expect(128)
    assert size(_bwd_args(B=2, L=100, H=4, P=64, G=2, N=128, chunk=64)) == expect(64)
    assert size(_bwd_args(B=2, L=300, H=4, P=64, G=2, N=128, chunk=128)) == expect(128, L=300)
    # other shapes and fp32: chunk 64 only
    assert size(_bwd_args(P=32, N=128, chunk=0)) == expect(64, P=32)
    assert size(_bwd_args(io=0, chunk=0)) == expect(64)
    for kw in (dict(io=0, chunk=128), dict(P=32, chunk=128), dict(N=64, chunk=128), dict(chunk=32),
               dict(P=256, N=16)):
        assert size(_bwd_args(**kw)) == ctypes.c_size_t(-1).value, kw


def test_bwd_validation():
    for kw in (dict(io=0, chunk=128), dict(P=32, chunk=128), dict(chunk=32)):
        assert _bwd(_bwd_args(**kw))[0] == _lib.SSD_ERR_UNSUPPORTED, kw
    b = _bwd_args(P=256, N=16)
    assert _bwd(b)[0] == _lib.SSD_ERR_UNSUPPORTED
    for field in ["dy", "dx", "ddt", "dA", "dBm", "dCm"]:
        b = _bwd_args()
        setattr(b, field, None)
        s, msg = _bwd(b)
        assert s == _lib.SSD_ERR_INVALID_ARG and "required" in msg, field
    b = _bwd_args()
    b.ddt = FAKE + (43 << 32) + 4
    s, msg = _bwd(b)
    assert s == _lib.SSD_ERR_INVALID_ARG and "aligned" in msg
    b = _bwd_args()
    b.dx = b.fwd.x  # gradient written over an input
    s, msg = _bwd(b)
    assert s == _lib.SSD_ERR_INVALID_ARG and "overlaps" in msg
    b = _bwd_args()
    b.dCm = b.dBm  # two outputs on the same memory
    s, msg = _bwd(b)
    assert s == _lib.SSD_ERR_INVALID_ARG and "overlaps" in msg
    b = _bwd_args()  # valid, but no workspace
    s, msg = _bwd(b)
    assert s == _lib.SSD_ERR_WORKSPACE


# ---------------------------------------------------------------- complex decay
def test_rot_struct_layout_matches_header(tmp_path):
    import os
    import subprocess
    fields = [f for f, _ in _lib.SsdFwdRotArgs._fields_]
    src = tmp_path / "probe_rot.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "ssd.h"\nint main(void){\n'
                   '  printf("%zu\\n", sizeof(ssd_fwd_rot_args));\n' +
                   "".join(f'  printf("%zu\\n", offsetof(ssd_fwd_rot_args, {f}));\n' for f in fields) +
                   "  return 0;\n}\n")
    exe = tmp_path / "probe_rot"
    subprocess.run(["gcc", "-I", os.path.dirname(_lib.HEADER_PATH), str(src), "-o", str(exe)], check=True)
    out = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert out[0] == ctypes.sizeof(_lib.SsdFwdRotArgs)
    assert out[1:] == [getattr(_lib.SsdFwdRotArgs, f).offset for f in fields]


def _rot_args(**kw):
    r = _lib.SsdFwdRotArgs()
    r.base = _args(**kw)
    r.theta = FAKE + (60 << 32)
    r.init_state_im = FAKE + (61 << 32)
    r.final_state_im = FAKE + (62 << 32)
    return r


def _rot(r):
    L = _lib.lib()
    return L.ssd_fwd_rot(ctypes.byref(r), None), L.ssd_last_error_message().decode()


def test_rot_workspace_and_validation():
    al = lambda v: (v + 255) // 256 * 256  # noqa: E731
    size = lambda r: _lib.lib().ssd_fwd_rot_workspace_size(ctypes.byref(r))  # noqa: E731
    # chunk 64 (explicit, or the default off the tensor-core shape): fp32 entering states only
    for kw in (dict(chunk=64), dict(chunk=0, io=0), dict(chunk=0, P=32)):
        P = kw.get("P", 64)
        r = _rot_args(B=2, L=100, H=4, G=2, N=128, **dict(dict(P=64), **kw))
        assert size(r) == 256 + 3 * al(2 * 4 * 2 * 64 * 4) + 2 * al(2 * 2 * 4 * P * 128 * 4), kw
    # bf16, headdim 64, dstate 128: chunk 0 is 128, with bf16 copies of both entering states
    for chunk in (0, 128):
        r = _rot_args(B=2, L=100, H=4, P=64, G=2, N=128, chunk=chunk)
        assert size(r) == 256 + 3 * al(2 * 4 * 1 * 128 * 4) + 2 * al(2 * 1 * 4 * 64 * 128 * 4) + \
            2 * al(2 * 1 * 4 * 64 * 128 * 2), chunk
    r = _rot_args()
    r.theta = None
    s, msg = _rot(r)
    assert s == _lib.SSD_ERR_INVALID_ARG and "theta" in msg
    r = _rot_args()
    r.theta = FAKE + (60 << 32) + 8
    assert _rot(r)[0] == _lib.SSD_ERR_INVALID_ARG
    r = _rot_args()
    r.final_state_im = r.base.final_state
    s, msg = _rot(r)
    assert s == _lib.SSD_ERR_INVALID_ARG and "overlaps" in msg
    r = _rot_args()
    r.final_state_im = r.theta
    s, msg = _rot(r)
    assert s == _lib.SSD_ERR_INVALID_ARG and "overlaps" in msg
    r = _rot_args()  # valid, no workspace
    assert _rot(r)[0] == _lib.SSD_ERR_WORKSPACE


# ---------------------------------------------------------------- retrieval rank
def test_mimo_struct_layout_matches_header(tmp_path):
    import os
    import subprocess
    fields = [f for f, _ in _lib.SsdFwdMimoArgs._fields_]
    src = tmp_path / "probe_mimo.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "ssd.h"\nint main(void){\n'
                   '  printf("%zu\\n", sizeof(ssd_fwd_mimo_args));\n' +
                   "".join(f'  printf("%zu\\n", offsetof(ssd_fwd_mimo_args, {f}));\n' for f in fields) +
                   "  return 0;\n}\n")
    exe = tmp_path / "probe_mimo"
    subprocess.run(["gcc", "-I", os.path.dirname(_lib.HEADER_PATH), str(src), "-o", str(exe)], check=True)
    out = [int(v) for v in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    assert out[0] == ctypes.sizeof(_lib.SsdFwdMimoArgs)
    assert out[1:] == [getattr(_lib.SsdFwdMimoArgs, f).offset for f in fields]


def _mimo_args(rank=4, **kw):
    m = _lib.SsdFwdMimoArgs()
    m.base = _args(**dict(dict(algo=0, chunk=0), **kw))
    m.rank = rank
    return m


def _mimo(m):
    L = _lib.lib()
    return L.ssd_fwd_mimo(ctypes.byref(m), None), L.ssd_last_error_message().decode()


def test_mimo_workspace_and_validation():
    size = lambda m: _lib.lib().ssd_fwd_mimo_workspace_size(ctypes.byref(m))  # noqa: E731
    bad = ctypes.c_size_t(-1).value
    # (the size of a valid problem depends on the device's SM count: checked
    # on the GPU, equal to the fused workspace of the problem of L * R rows)
    for R in (0, 3, 16, -1):
        m = _mimo_args(rank=R)
        s, msg = _mimo(m)
        assert s == _lib.SSD_ERR_UNSUPPORTED and "rank" in msg and size(m) == bad
    for kw in (dict(io=0), dict(P=32), dict(N=32), dict(chunk=64), dict(algo=1)):
        m = _mimo_args(**kw)
        s, msg = _mimo(m)
        assert s == _lib.SSD_ERR_UNSUPPORTED and "mimo" in msg and size(m) == bad, kw
    m = _mimo_args()
    m.base.dt = None
    assert _mimo(m)[0] == _lib.SSD_ERR_INVALID_ARG
    m = _mimo_args()
    m.base.y = m.base.x
    s, msg = _mimo(m)
    assert s == _lib.SSD_ERR_INVALID_ARG and "overlaps" in msg
    # (a valid problem, an empty batch and a missing workspace need the
    # driver's tensor-map encoder: checked on the GPU)


def test_rot_fused_request_unsupported():
    """algo FUSED on a problem the fused complex-decay kernel does not take
    (fp32 io, or dstate 64) is rejected before any launch, and the workspace
    query says so."""
    size = lambda r: _lib.lib().ssd_fwd_rot_workspace_size(ctypes.byref(r))  # noqa: E731
    for kw in (dict(io=0), dict(N=64), dict(P=32)):
        r = _rot_args(**dict(dict(B=2, L=100, H=4, P=64, G=2, N=128, chunk=0, algo=2), **kw))
        assert size(r) == ctypes.c_size_t(-1).value, kw
        s, msg = _rot(r)
        assert s == _lib.SSD_ERR_UNSUPPORTED and "fused" in msg, kw
