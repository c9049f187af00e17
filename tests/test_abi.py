"""The C ABI on the host (no GPU): the library loads, exports every entry point
that include/ss_scan.h declares, and rejects bad arguments before launching.
Only calls that fail validation are made, so nothing here touches a device."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

import selective_state_space_117_b300 as ss

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


def declared_functions():
    names = set()
    for f in os.listdir(HEADER_DIR):
        if f.endswith(".h"):
            src = open(os.path.join(HEADER_DIR, f)).read()
            names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(ss_\w+)\s*\(", src, flags=re.M))
    return sorted(names)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("ss_scan_fwd", "ss_scan_chunked", "ss_scan_chunked_workspace_bytes", "ss_state_update",
                 "ss_status_string", "ss_last_cuda_error"):
        assert want in names


def test_library_exports_every_declared_symbol():
    lib = ss.lib()
    out = subprocess.run(["nm", "-D", "--defined-only", ss.library_path()], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (ss_\w+)", out))
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in exported, name


def _dims(b=1, d=4, n=4, L=16, dt=ss.F32):
    return ss.Dims(b, d, n, L, dt)


P = 4096  # a fake, 256-byte aligned "device" address: never dereferenced, validation fails first


def _fwd(dims, **over):
    a = dict(u=P, delta=P, A=P, B=P, C=P, D=None, z=None, bias=None, y=P, last=None)
    a.update(over)
    return ss.lib().ss_scan_fwd(ctypes.byref(dims), a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"],
                                a["bias"], 1, a["y"], a["last"], None)


def _chunked(dims, chunk=8, ws=P, ws_bytes=1 << 30, **over):
    a = dict(u=P, delta=P, A=P, B=P, C=P, D=None, z=None, bias=None, y=P, last=None)
    a.update(over)
    return ss.lib().ss_scan_chunked(ctypes.byref(dims), a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"], a["z"],
                                    a["bias"], 1, a["y"], a["last"], chunk, ws, ws_bytes, None)


def _flagged(flags, **kw):
    d = _dims(**kw)
    d.flags = flags
    return d


def test_validation_status_codes():
    assert _fwd(_dims(dt=7)) == ss.SS_EDTYPE
    assert _fwd(_flagged(8)) == ss.SS_EINVAL                # unknown flag bit
    assert _fwd(_flagged(1 << 30)) == ss.SS_EINVAL
    assert _fwd(_dims(L=-1)) == ss.SS_EINVAL
    assert _fwd(_dims(n=65)) == ss.SS_EINVAL
    assert _fwd(_dims(b=70000)) == ss.SS_EINVAL
    assert _fwd(_dims(), u=None) == ss.SS_EINVAL
    assert _fwd(_dims(), y=None) == ss.SS_EINVAL
    assert _fwd(_dims(), B=None) == ss.SS_EINVAL
    assert _fwd(_dims(), u=P + 2) == ss.SS_EALIGN           # fp32 input at a 2-byte offset
    assert _fwd(_dims(dt=ss.BF16), u=P + 1) == ss.SS_EALIGN  # bf16 input at an odd address
    assert _fwd(_dims(), A=P + 1) == ss.SS_EALIGN
    assert _fwd(_dims(), y=P + 2) == ss.SS_EALIGN
    assert ss.lib().ss_scan_fwd(None, P, P, P, P, P, None, None, None, 1, P, None, None) == ss.SS_EINVAL
    # sizes of zero are valid no-ops and return before any launch
    assert _fwd(_dims(b=0), u=None, delta=None, y=None) == ss.SS_OK
    assert _fwd(_dims(d=0), u=None, delta=None, y=None, A=None) == ss.SS_OK


def test_schedule_flags():
    # every case fails on the host before any launch
    both = ss.FLAG_SCHED_THREAD | ss.FLAG_SCHED_WARP
    assert _fwd(_flagged(both)) == ss.SS_EINVAL
    # the warp schedule refuses what it cannot run: N > 16, L % 8 != 0 (either input weight)
    assert _fwd(_flagged(ss.FLAG_SCHED_WARP, n=17)) == ss.SS_EINVAL
    assert _fwd(_flagged(ss.FLAG_SCHED_WARP, L=12)) == ss.SS_EINVAL
    assert _fwd(_flagged(ss.FLAG_SCHED_WARP | ss.FLAG_ZOH, n=17)) == ss.SS_EINVAL
    assert _fwd(_flagged(ss.FLAG_SCHED_WARP | ss.FLAG_ZOH, L=20)) == ss.SS_EINVAL
    # schedule flags belong to ss_scan_fwd only
    assert _chunked(_flagged(ss.FLAG_SCHED_THREAD)) == ss.SS_EINVAL
    assert _chunked(_flagged(ss.FLAG_SCHED_WARP)) == ss.SS_EINVAL
    assert _bwd(_flagged(ss.FLAG_SCHED_WARP)) == ss.SS_EINVAL
    # zero sizes stay no-ops under either flag
    assert _fwd(_flagged(ss.FLAG_SCHED_WARP, b=0), u=None, delta=None, y=None) == ss.SS_OK
    with pytest.raises(ValueError):
        ss.scan_fwd(torch.zeros(1, 1, 8), torch.zeros(1, 1, 8), torch.zeros(1, 4), torch.zeros(1, 4, 8),
                    torch.zeros(1, 4, 8), schedule="lanes")


def _conv(dims, x=P, w=P, bias=None, out=P):
    return ss.lib().ss_causal_conv1d(ctypes.byref(dims), x, w, bias, 1, out, None)


def test_conv_validation():
    # every case fails (or returns) on the host before any launch
    assert _conv(_dims(dt=9)) == ss.SS_EDTYPE
    assert _conv(_dims(L=-1)) == ss.SS_EINVAL
    assert _conv(_flagged(ss.FLAG_ZOH)) == ss.SS_EINVAL          # no input weight to choose
    assert _conv(_flagged(ss.FLAG_SCHED_WARP)) == ss.SS_EINVAL
    assert _conv(_dims(), x=None) == ss.SS_EINVAL
    assert _conv(_dims(), w=P + 4) == ss.SS_EALIGN               # taps must be 16-byte aligned
    assert _conv(_dims(dt=ss.BF16), x=P + 1) == ss.SS_EALIGN
    assert _conv(_dims(L=0), x=None, w=None, out=None) == ss.SS_OK


def test_chunked_validation():
    assert _chunked(_dims(), chunk=0) == ss.SS_EINVAL
    assert _chunked(_dims(), ws=None) == ss.SS_EWORKSPACE
    assert _chunked(_dims(), ws=P + 16) == ss.SS_EWORKSPACE            # not 256-byte aligned
    need = ss.chunked_workspace_bytes(1, 4, 4, 16, 8)
    assert _chunked(_dims(), ws_bytes=need - 1) == ss.SS_EWORKSPACE
    assert _chunked(_dims(dt=3)) == ss.SS_EDTYPE


def test_workspace_bytes():
    # S: batch*dim*K floats, then H: batch*dim*K*N floats, each padded to 256 B, then the
    # channel order of the local pass: dim int32
    assert ss.chunked_workspace_bytes(1, 4, 4, 16, 8) == 256 + 256 + 4 * 4
    K = 65536 // 2048
    assert ss.chunked_workspace_bytes(1, 5120, 16, 65536, 2048) == 5120 * K * 4 + 5120 * K * 16 * 4 + 5120 * 4
    assert ss.chunked_workspace_bytes(1, 4, 4, 16, 0) == 0
    assert ss.chunked_workspace_bytes(2, 3, 5, 7, 3) == 256 + 512 + 3 * 4   # H: 360 B padded to 512


def _bwd(dims, ws=P, ws_bytes=1 << 40, **over):
    a = dict(h0=None, u=P, delta=P, A=P, B=P, C=P, D=None, z=None, bias=None, dy=P, dlast=None, du=P, ddelta=P,
             dA=P, dB=P, dC=P, dD=None, dz=None, dbias=None, dh0=None)
    a.update(over)
    return ss.lib().ss_scan_bwd(ctypes.byref(dims), a["h0"], a["u"], a["delta"], a["A"], a["B"], a["C"], a["D"],
                                a["z"], a["bias"], 1, a["dy"], a["dlast"], a["du"], a["ddelta"], a["dA"], a["dB"],
                                a["dC"], a["dD"], a["dz"], a["dbias"], a["dh0"], ws, ws_bytes, None)


def test_bwd_validation():
    bad = _dims()
    bad.flags = 2                                           # unknown discretisation bit
    assert _bwd(bad) == ss.SS_EINVAL
    assert _bwd(_dims(dt=5)) == ss.SS_EDTYPE
    assert _bwd(_dims(), dy=None) == ss.SS_EINVAL
    assert _bwd(_dims(), du=None) == ss.SS_EINVAL
    assert _bwd(_dims(), ddelta=None) == ss.SS_EINVAL
    assert _bwd(_dims(), dB=None) == ss.SS_EINVAL
    assert _bwd(_dims(), dA=None) == ss.SS_EINVAL
    assert _bwd(_dims(), dz=P) == ss.SS_EINVAL                # dz without a gate
    assert _bwd(_dims(), dA=P + 2) == ss.SS_EALIGN
    assert _bwd(_dims(), dh0=P + 1) == ss.SS_EALIGN
    assert _bwd(_dims(), ws=None) == ss.SS_EWORKSPACE
    assert _bwd(_dims(), ws=P + 16) == ss.SS_EWORKSPACE
    assert _bwd(_dims(), ws_bytes=ss.bwd_workspace_bytes(1, 4, 4, 16) - 1) == ss.SS_EWORKSPACE


def test_bwd_workspace_bytes():
    # S: batch*dim*K floats, then H and G: batch*dim*K*N floats each, the first two padded to 256 B
    assert ss.bwd_workspace_bytes(1, 4, 4, 16) == 256 + 256 + 1 * 4 * 1 * 4 * 4
    K = 65536 // 64
    assert ss.bwd_workspace_bytes(1, 5120, 16, 65536) == 5120 * K * 4 + 2 * 5120 * K * 16 * 4
    assert ss.bwd_workspace_bytes(2, 3, 5, 130) == 256 + 512 + 2 * 3 * 3 * 5 * 4   # K = 3


def test_state_update_validation():
    lib = ss.lib()
    d = _dims()
    call = lambda dims, st=P, u=P, A=P: lib.ss_state_update(ctypes.byref(dims), st, u, P, A, P, P, None, None, None,
                                                            1, P, None)
    assert call(_dims(dt=9)) == ss.SS_EDTYPE
    assert call(_dims(n=100)) == ss.SS_EINVAL
    assert call(d, st=None) == ss.SS_EINVAL
    assert call(d, u=None) == ss.SS_EINVAL
    assert call(d, st=P + 1) == ss.SS_EALIGN
    assert call(_dims(b=0)) == ss.SS_OK


def test_measure_ex2_validation():
    n = ctypes.c_uint64(0)
    f = ss.lib().ss_measure_ex2
    assert f(0, 16, P, ctypes.byref(n), None) == ss.SS_EINVAL
    assert f(4, 0, P, ctypes.byref(n), None) == ss.SS_EINVAL
    assert f(4, 16, None, ctypes.byref(n), None) == ss.SS_EINVAL
    assert f(4, 16, P, None, None) == ss.SS_EINVAL
    assert f(4, 16, P + 2, ctypes.byref(n), None) == ss.SS_EALIGN


def test_status_strings():
    for code in (0, -1, -2, -3, -4, -5, -6):
        s = ss.lib().ss_status_string(code).decode()
        assert s.startswith("SS_")
    assert "unknown" in ss.lib().ss_status_string(42).decode()
    assert ss.lib().ss_last_cuda_error() == 0


def test_binding_refuses_host_tensors():
    u = torch.zeros((1, 4, 16))
    with pytest.raises(ValueError, match="CUDA device only"):
        ss.scan_fwd(u, u, torch.zeros((4, 4)), torch.zeros((1, 4, 16)), torch.zeros((1, 4, 16)))
    with pytest.raises(ValueError, match="CUDA device only"):
        ss.state_update(torch.zeros((1, 4, 4)), u[:, :, 0], u[:, :, 0], torch.zeros((4, 4)), torch.zeros((1, 4)),
                        torch.zeros((1, 4)))
