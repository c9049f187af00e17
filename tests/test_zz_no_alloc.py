"""ss_scan_chunked_static: the chunked scan on a workspace the library owns.

Some callers cannot call cudaMalloc: code that runs inside a custom allocator or
memory pool, a plugin whose host owns every device allocation, or a service that
forbids allocation once it has started.  For them the library exports
ss_scan_chunked_static, which takes no workspace argument and uses a fixed
device array inside the library instead (SS_STATIC_WORKSPACE_BYTES).

The GPU test calls it through the C ABI twice in a row, on two problems of
different shapes and dtypes.  Each result must equal, bit for bit, what
ss_scan_chunked computes with a caller-provided workspace (the same kernels in
the same launch configuration), and must match the fp64 oracle under the parity
tolerances of tests/parity.py.  Because every call shares the array, anything
the first call left behind that the second call wrongly read would show up as a
mismatch.  The host test checks
that a problem too large for the array is refused before the device is touched.
"""
import ctypes

import pytest
import torch

import oracle
import selective_state_space_117_b300 as ss
from selective_state_space_117_b300 import inputs as I
from parity import check, host

STATIC_BYTES = 16 << 20  # SS_STATIC_WORKSPACE_BYTES in include/ss_scan.h


def _static_fn():
    f = ss.lib().ss_scan_chunked_static
    vp = ctypes.c_void_p
    f.argtypes = [ctypes.POINTER(ss.Dims), vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int, vp, vp, ctypes.c_int64, vp]
    f.restype = ctypes.c_int
    return f


def _ptr(t):
    return None if t is None else t.data_ptr()


def _call_static(p, chunk, y, hl):
    dims = ss.Dims(p.batch, p.dim, p.dstate, p.seqlen, p.in_dtype)
    return _static_fn()(ctypes.byref(dims), _ptr(p.u), _ptr(p.delta), _ptr(p.A), _ptr(p.B), _ptr(p.C), _ptr(p.D),
                        _ptr(p.z), _ptr(p.delta_bias), 1, _ptr(y), _ptr(hl), chunk,
                        torch.cuda.current_stream().cuda_stream)


def _problems():
    a = I.selective_problem("static_bf16", seed=11, batch=2, dim=384, dstate=16, seqlen=6144, dtype=torch.bfloat16,
                            bc_std=0.25, d_mode="ones", gate=True, device="cuda", gen_device="cpu")
    b = I.selective_problem("static_f32", seed=12, batch=1, dim=200, dstate=8, seqlen=3000, dtype=torch.float32,
                            bc_std=0.5, d_mode="normal", gate=False, device="cuda", gen_device="cpu")
    return [(a, 1024), (b, 256)]


@pytest.mark.gpu
def test_static_workspace_matches_caller_workspace_on_two_calls():
    for p, chunk in _problems():
        need = ss.chunked_workspace_bytes(p.batch, p.dim, p.dstate, p.seqlen, chunk)
        assert 0 < need <= STATIC_BYTES
        y_ref, h_ref = ss.scan_chunked(p.u, p.delta, p.A, p.B, p.C, D=p.D, z=p.z, delta_bias=p.delta_bias,
                                       chunk_len=chunk, return_last_state=True)
        y = torch.full_like(y_ref, float("nan"))
        hl = torch.full_like(h_ref, float("nan"))
        st = _call_static(p, chunk, y, hl)
        assert st == 0, ss.lib().ss_status_string(st).decode()
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref), f"{p.name}: y differs from ss_scan_chunked's"
        assert torch.equal(hl, h_ref), f"{p.name}: last_state differs from ss_scan_chunked's"
        bf = p.in_dtype == I.BF16
        n = p.batch * p.dim
        w = I.to_wire
        yr, hr = oracle.scan(w(p.u), w(p.delta), w(p.A), w(p.B), w(p.C), D=w(p.D), z=w(p.z),
                             delta_bias=w(p.delta_bias), dtype="bf16" if bf else "f32")
        check(host(y).reshape(n, p.seqlen), yr, bf, f"{p.name} static y vs oracle")
        check(host(hl).reshape(n, p.dstate), hr, bf, f"{p.name} static last_state vs oracle")


def test_static_workspace_refuses_oversized_problem():
    # 1 x 5120 channels, N = 64, L = 65536, chunk 64: about 1.4 GB of workspace.
    dims = ss.Dims(1, 5120, 64, 65536, ss.BF16)
    fake = 4096  # never dereferenced: the size check comes first
    st = _static_fn()(ctypes.byref(dims), fake, fake, fake, fake, fake, None, None, None, 1, fake, None, 64, None)
    assert st == ss.SS_EWORKSPACE
