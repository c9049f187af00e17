"""B300-native selective state space scan (Mamba S6).

Python binding of the C ABI in ``include/ss_scan.h`` (``libssscan.so``, built
in-tree by ``python -m selective_state_space_117_b300.build``).  The binding
only checks tensor shapes and dtypes, allocates outputs with PyTorch and
passes device pointers and the current CUDA stream to the library; every step
of the scan runs in the library's CUDA kernels.  There is no CPU path: when
the library is missing or a tensor is not on a CUDA device, calls raise.

Entry points (same names as the C ABI, without the ``ss_`` prefix):
  scan_fwd        full-sequence scan
  scan_chunked    full-sequence scan as local scan / carry / fix-up over chunks
  state_update    one decode step on a persistent (batch, dim, N) fp32 state
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

__all__ = ["scan_fwd", "scan_chunked", "scan_bwd", "bwd_workspace_bytes", "state_update", "causal_conv1d", "chunked_workspace_bytes", "device_status",
           "selftest_wait_timeout", "selective_scan", "measure_ex2",
           "SSError",
           "library_path",
           "F32", "BF16", "MAX_DSTATE", "LAUNCHES"]

_HERE = os.path.dirname(os.path.abspath(__file__))
# SS_LIBRARY=debug loads the debug build (device-side index checks, libssscan_debug.so).
_LIB_PATH = os.path.join(_HERE, "libssscan_debug.so" if os.environ.get("SS_LIBRARY") == "debug" else "libssscan.so")
_lib = None

F32, BF16 = 0, 1
MAX_DSTATE = 64
# Kernels launched per call (for launch accounting): chunked = channel order + local + carry + fix-up
# (the first two only when there is more than one chunk).
LAUNCHES = {"scan_fwd": 1, "scan_chunked": 4, "state_update": 1, "scan_bwd": 5}

SS_OK, SS_EINVAL, SS_EALIGN, SS_EDTYPE, SS_EWORKSPACE, SS_ECUDA, SS_ETIMEOUT, SS_EBOUNDS = 0, -1, -2, -3, -4, -5, -6, -7


class SSError(RuntimeError):
    """A non-zero ss_status returned by the library."""

    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


FLAG_ZOH = 1
FLAG_SCHED_THREAD, FLAG_SCHED_WARP = 2, 4
_SCHED = {None: 0, "thread": FLAG_SCHED_THREAD, "warp": FLAG_SCHED_WARP}


class Dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("dim", ctypes.c_int64), ("dstate", ctypes.c_int64),
                ("seqlen", ctypes.c_int64), ("in_dtype", ctypes.c_int32), ("flags", ctypes.c_int32)]


def library_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded libssscan.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise ImportError(f"{_LIB_PATH} is missing; build it with `python -m selective_state_space_117_b300.build`")
        L = ctypes.CDLL(_LIB_PATH)
        vp, i64 = ctypes.c_void_p, ctypes.c_int64
        dp = ctypes.POINTER(Dims)
        L.ss_scan_fwd.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int, vp, vp, vp]
        L.ss_scan_fwd.restype = ctypes.c_int
        L.ss_scan_chunked_workspace_bytes.argtypes = [dp, i64]
        L.ss_scan_chunked_workspace_bytes.restype = ctypes.c_size_t
        L.ss_scan_chunked.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int, vp, vp, i64, vp,
                                      ctypes.c_size_t, vp]
        L.ss_scan_chunked.restype = ctypes.c_int
        L.ss_scan_fwd_h0.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int, vp, vp, vp]
        L.ss_scan_fwd_h0.restype = ctypes.c_int
        L.ss_scan_chunked_h0.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int, vp, vp, i64, vp,
                                         ctypes.c_size_t, vp]
        L.ss_scan_chunked_h0.restype = ctypes.c_int
        L.ss_scan_chunked_phase.argtypes = [ctypes.c_int, dp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int, vp, vp,
                                            i64, vp, ctypes.c_size_t, vp]
        L.ss_scan_chunked_phase.restype = ctypes.c_int
        L.ss_state_update.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int, vp, vp]
        L.ss_state_update.restype = ctypes.c_int
        L.ss_status_string.argtypes = [ctypes.c_int]
        L.ss_status_string.restype = ctypes.c_char_p
        L.ss_last_cuda_error.argtypes = []
        L.ss_last_cuda_error.restype = ctypes.c_int
        L.ss_selftest_wait_timeout.argtypes = [vp]
        L.ss_selftest_wait_timeout.restype = ctypes.c_int
        L.ss_causal_conv1d.argtypes = [dp, vp, vp, vp, ctypes.c_int, vp, vp]
        L.ss_causal_conv1d.restype = ctypes.c_int
        L.ss_scan_bwd_workspace_bytes.argtypes = [dp]
        L.ss_scan_bwd_workspace_bytes.restype = ctypes.c_size_t
        L.ss_scan_bwd.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int, vp, vp, vp, vp, vp, vp, vp,
                                  vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
        L.ss_scan_bwd.restype = ctypes.c_int
        L.ss_device_status.argtypes = [ctypes.c_int]
        L.ss_device_status.restype = ctypes.c_int
        L.ss_measure_ex2.argtypes = [i64, ctypes.c_int, vp, ctypes.POINTER(ctypes.c_uint64), vp]
        L.ss_measure_ex2.restype = ctypes.c_int
        L.ss_selftest_bounds.argtypes = [vp]
        L.ss_selftest_bounds.restype = ctypes.c_int
        L.ss_debug_bounds_build.argtypes = []
        L.ss_debug_bounds_build.restype = ctypes.c_int
        _lib = L
    return _lib


def _check(status: int, what: str):
    if status != SS_OK:
        msg = lib().ss_status_string(status).decode()
        if status == SS_ECUDA:
            msg += f" (cudaError {lib().ss_last_cuda_error()})"
        raise SSError(status, f"{what}: {msg}")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


def _stream(device, stream):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"inputs must be float32 or bfloat16, got {t.dtype}")


def _need(t, name, shape, dtype, device):
    if t is None:
        return
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _scan_common(u, delta, A, B, C, D, z, delta_bias, y, last_state):
    if not isinstance(u, torch.Tensor) or u.dim() != 3:
        raise ValueError("u must be a (batch, dim, seqlen) tensor")
    if u.device.type != "cuda":
        raise ValueError("the selective scan runs on a CUDA device only; u is on " + str(u.device))
    batch, dim, L = u.shape
    if not isinstance(A, torch.Tensor) or A.dim() != 2:
        raise ValueError("A must be a (dim, dstate) tensor")
    N = A.shape[1]
    dev, dt = u.device, u.dtype
    code = _dtype_code(u)
    _need(u, "u", (batch, dim, L), dt, dev)
    _need(delta, "delta", (batch, dim, L), dt, dev)
    _need(A, "A", (dim, N), torch.float32, dev)
    _need(B, "B", (batch, N, L), dt, dev)
    _need(C, "C", (batch, N, L), dt, dev)
    _need(D, "D", (dim,), torch.float32, dev)
    _need(z, "z", (batch, dim, L), dt, dev)
    _need(delta_bias, "delta_bias", (dim,), torch.float32, dev)
    if y is None:
        y = torch.empty((batch, dim, L), dtype=torch.float32, device=dev)
    _need(y, "y", (batch, dim, L), torch.float32, dev)
    _need(last_state, "last_state", (batch, dim, N), torch.float32, dev)
    return Dims(batch, dim, N, L, code), y


def scan_fwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, *, y=None, last_state=None,
             return_last_state=False, h0=None, zoh=False, schedule=None, stream=None):
    """Full-sequence selective scan.  Returns y (fp32, (batch, dim, L)), or
    (y, last_state) when ``return_last_state`` or ``last_state`` is given.
    ``h0`` (fp32, (batch, dim, N)) starts the scan from that state (ss_scan_fwd_h0).
    ``zoh`` uses the zero-order-hold input weight (SS_FLAG_ZOH).  ``schedule``:
    None (the library picks), "thread" (one thread per channel) or "warp" (one
    warp per channel, lanes split time; SS_FLAG_SCHED_*)."""
    if schedule not in _SCHED:
        raise ValueError(f"schedule must be one of {sorted(k for k in _SCHED if k)} or None")
    dims, y = _scan_common(u, delta, A, B, C, D, z, delta_bias, y, last_state)
    dims.flags = (FLAG_ZOH if zoh else 0) | _SCHED[schedule]
    _need(h0, "h0", (dims.batch, dims.dim, dims.dstate), torch.float32, u.device)
    if return_last_state and last_state is None:
        last_state = torch.empty((dims.batch, dims.dim, dims.dstate), dtype=torch.float32, device=u.device)
    args = (_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias), int(bool(softplus)),
            _ptr(y), _ptr(last_state), _stream(u.device, stream))
    if h0 is None:
        _check(lib().ss_scan_fwd(ctypes.byref(dims), *args), "ss_scan_fwd")
    else:
        _check(lib().ss_scan_fwd_h0(ctypes.byref(dims), _ptr(h0), *args), "ss_scan_fwd_h0")
    return (y, last_state) if last_state is not None else y


def chunked_workspace_bytes(batch, dim, dstate, seqlen, chunk_len, dtype=F32) -> int:
    dims = Dims(batch, dim, dstate, seqlen, dtype)
    return int(lib().ss_scan_chunked_workspace_bytes(ctypes.byref(dims), int(chunk_len)))


PHASE_LOCAL, PHASE_CARRY, PHASE_FIXUP = 1, 2, 3


def scan_chunked(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, *, chunk_len=2048, y=None,
                 last_state=None, return_last_state=False, workspace=None, stream=None, phase=None, h0=None,
                 zoh=False):
    """Chunked selective scan (local scan, carry across chunks, fix-up).  Same
    result and return convention as ``scan_fwd``.  ``workspace`` is an optional
    uint8 CUDA tensor of at least ``chunked_workspace_bytes`` bytes.  With
    ``phase`` in (1, 2, 3) only that phase runs (ss_scan_chunked_phase); the
    three phases in order on one stream, sharing a workspace, are the full call."""
    dims, y = _scan_common(u, delta, A, B, C, D, z, delta_bias, y, last_state)
    dims.flags = FLAG_ZOH if zoh else 0
    if return_last_state and last_state is None:
        last_state = torch.empty((dims.batch, dims.dim, dims.dstate), dtype=torch.float32, device=u.device)
    need = int(lib().ss_scan_chunked_workspace_bytes(ctypes.byref(dims), int(chunk_len)))
    if workspace is None:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=u.device)
    if workspace.device != u.device or workspace.dtype != torch.uint8 or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous uint8 tensor on the inputs' device")
    _need(h0, "h0", (dims.batch, dims.dim, dims.dstate), torch.float32, u.device)
    if h0 is not None and phase is not None:
        raise ValueError("h0 is only supported for the whole chunked call (phase=None)")
    tail = (_ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z), _ptr(delta_bias),
            int(bool(softplus)), _ptr(y), _ptr(last_state), int(chunk_len), _ptr(workspace), workspace.numel(),
            _stream(u.device, stream))
    if h0 is not None:
        _check(lib().ss_scan_chunked_h0(ctypes.byref(dims), _ptr(h0), *tail), "ss_scan_chunked_h0")
    elif phase is None:
        _check(lib().ss_scan_chunked(ctypes.byref(dims), *tail), "ss_scan_chunked")
    else:
        _check(lib().ss_scan_chunked_phase(int(phase), ctypes.byref(dims), *tail), f"ss_scan_chunked_phase({phase})")
    return (y, last_state) if last_state is not None else y


def bwd_workspace_bytes(batch, dim, dstate, seqlen, dtype=F32) -> int:
    dims = Dims(batch, dim, dstate, seqlen, dtype)
    return int(lib().ss_scan_bwd_workspace_bytes(ctypes.byref(dims)))


def scan_bwd(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, *, dy, dlast=None, h0=None,
             want_dD=True, want_dbias=True, want_dh0=None, zoh=False, workspace=None, stream=None):
    """Backward pass of ``scan_fwd`` (ss_scan_bwd): the gradients of
    sum(dy * y) + sum(dlast * last_state) for the forward scan on the same inputs.

    dy is fp32 (batch, dim, L); dlast and h0 are fp32 (batch, dim, N) or None.
    Returns a dict of fp32 tensors: du, ddelta (like u), dz (like u, or None
    without z), dA (dim, N), dB, dC (batch, N, L), dD and ddelta_bias (dim,)
    (None unless ``want_dD`` / ``want_dbias``), dh0 (batch, dim, N) (computed
    when ``want_dh0``, by default when h0 is given).  ``workspace`` is an optional
    uint8 CUDA tensor of at least ``bwd_workspace_bytes`` bytes.  ``zoh``: the
    forward scan used the zero-order-hold input weight (SS_FLAG_ZOH)."""
    dims, _ = _scan_common(u, delta, A, B, C, D, z, delta_bias, dy, None)
    dims.flags = FLAG_ZOH if zoh else 0
    batch, dim, N, L = dims.batch, dims.dim, dims.dstate, dims.seqlen
    dev = u.device
    _need(dlast, "dlast", (batch, dim, N), torch.float32, dev)
    _need(h0, "h0", (batch, dim, N), torch.float32, dev)
    f32 = dict(dtype=torch.float32, device=dev)
    out = dict(du=torch.empty((batch, dim, L), **f32), ddelta=torch.empty((batch, dim, L), **f32),
               dz=torch.empty((batch, dim, L), **f32) if z is not None else None,
               dA=torch.empty((dim, N), **f32), dB=torch.empty((batch, N, L), **f32),
               dC=torch.empty((batch, N, L), **f32),
               dD=torch.empty((dim,), **f32) if want_dD else None,
               ddelta_bias=torch.empty((dim,), **f32) if want_dbias else None,
               dh0=torch.empty((batch, dim, N), **f32) if (want_dh0 if want_dh0 is not None else h0 is not None)
               else None)
    need = int(lib().ss_scan_bwd_workspace_bytes(ctypes.byref(dims)))
    if workspace is None:
        workspace = torch.empty((max(need, 1),), dtype=torch.uint8, device=dev)
    if workspace.device != dev or workspace.dtype != torch.uint8 or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous uint8 tensor on the inputs' device")
    st = lib().ss_scan_bwd(ctypes.byref(dims), _ptr(h0), _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
                           _ptr(z), _ptr(delta_bias), int(bool(softplus)), _ptr(dy), _ptr(dlast),
                           _ptr(out["du"]), _ptr(out["ddelta"]), _ptr(out["dA"]), _ptr(out["dB"]), _ptr(out["dC"]),
                           _ptr(out["dD"]), _ptr(out["dz"]), _ptr(out["ddelta_bias"]), _ptr(out["dh0"]),
                           _ptr(workspace), workspace.numel(), _stream(dev, stream))
    _check(st, "ss_scan_bwd")
    return out


class _SelectiveScan(torch.autograd.Function):
    """Forward: ss_scan_fwd (or ss_scan_chunked when chunk_len is given); backward:
    ss_scan_bwd with the cotangents of y and of the final state.  Gradients come back
    in fp32 from the library and are cast to each input's dtype."""

    @staticmethod
    def forward(ctx, u, delta, A, B, C, D, z, delta_bias, h0, softplus, zoh, chunk_len):
        kw = dict(D=D, z=z, delta_bias=delta_bias, softplus=softplus, zoh=zoh, return_last_state=True, h0=h0)
        if chunk_len is None:
            y, last = scan_fwd(u, delta, A, B, C, **kw)
        else:
            y, last = scan_chunked(u, delta, A, B, C, chunk_len=chunk_len, **kw)
        ctx.save_for_backward(u, delta, A, B, C, D, z, delta_bias, h0)
        ctx.softplus, ctx.zoh = softplus, zoh
        ctx.set_materialize_grads(False)
        return y, last

    @staticmethod
    def backward(ctx, dy, dlast):
        u, delta, A, B, C, D, z, delta_bias, h0 = ctx.saved_tensors
        if dy is None:
            dy = torch.zeros(u.shape, dtype=torch.float32, device=u.device)
        dy = dy.to(torch.float32).contiguous()
        if dlast is not None:
            dlast = dlast.to(torch.float32).contiguous()
        need = ctx.needs_input_grad
        g = scan_bwd(u, delta, A, B, C, D, z, delta_bias, ctx.softplus, dy=dy, dlast=dlast, h0=h0,
                     want_dD=D is not None and need[5], want_dbias=delta_bias is not None and need[7],
                     want_dh0=h0 is not None and need[8], zoh=ctx.zoh)
        cast = lambda t, like: None if t is None else t.to(like.dtype)
        return (cast(g["du"], u), cast(g["ddelta"], delta), g["dA"], cast(g["dB"], B), cast(g["dC"], C),
                g["dD"] if D is not None else None, cast(g["dz"], z) if z is not None else None,
                g["ddelta_bias"] if delta_bias is not None else None, g["dh0"] if h0 is not None else None,
                None, None, None)


def selective_scan(u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, *, h0=None, zoh=False,
                   chunk_len=None):
    """Differentiable selective scan: returns (y, last_state) like ``scan_fwd(...,
    return_last_state=True)`` (or ``scan_chunked`` with ``chunk_len``), starting from ``h0``
    (fp32 (batch, dim, N)) when given, and back-propagates through ``scan_bwd`` into every
    input that requires grad, h0 included.  Inputs as ``scan_fwd``; they must be contiguous
    CUDA tensors."""
    return _SelectiveScan.apply(u, delta, A, B, C, D, z, delta_bias, h0, bool(softplus), bool(zoh), chunk_len)


def state_update(state, u, delta, A, B, C, D=None, z=None, delta_bias=None, softplus=True, *, y=None,
                 zoh=False, stream=None):
    """One decode step.  state (batch, dim, N) fp32 is updated in place;
    u, delta, z are (batch, dim); B, C are (batch, N).  Returns y (batch, dim) fp32."""
    if not isinstance(u, torch.Tensor) or u.dim() != 2:
        raise ValueError("u must be a (batch, dim) tensor")
    if u.device.type != "cuda":
        raise ValueError("the selective scan runs on a CUDA device only; u is on " + str(u.device))
    batch, dim = u.shape
    N = A.shape[1]
    dev, dt = u.device, u.dtype
    code = _dtype_code(u)
    _need(state, "state", (batch, dim, N), torch.float32, dev)
    _need(delta, "delta", (batch, dim), dt, dev)
    _need(A, "A", (dim, N), torch.float32, dev)
    _need(B, "B", (batch, N), dt, dev)
    _need(C, "C", (batch, N), dt, dev)
    _need(D, "D", (dim,), torch.float32, dev)
    _need(z, "z", (batch, dim), dt, dev)
    _need(delta_bias, "delta_bias", (dim,), torch.float32, dev)
    if y is None:
        y = torch.empty((batch, dim), dtype=torch.float32, device=dev)
    _need(y, "y", (batch, dim), torch.float32, dev)
    dims = Dims(batch, dim, N, 1, code, FLAG_ZOH if zoh else 0)
    st = lib().ss_state_update(ctypes.byref(dims), _ptr(state), _ptr(u), _ptr(delta), _ptr(A), _ptr(B), _ptr(C),
                               _ptr(D), _ptr(z), _ptr(delta_bias), int(bool(softplus)), _ptr(y),
                               _stream(u.device, stream))
    _check(st, "ss_state_update")
    return y


def device_status(clear: bool = False) -> int:
    """Status word of the current device (ss_device_status): SS_OK, or SS_ETIMEOUT
    when a kernel's bounded wait gave up.  Synchronises the device first."""
    st = lib().ss_device_status(int(bool(clear)))
    if st not in (SS_OK, SS_ETIMEOUT, SS_EBOUNDS):
        _check(st, "ss_device_status")
    return st


def selftest_bounds(device=None, stream=None):
    """Launch the diagnostic index check of a span outside its array (ss_selftest_bounds): the
    debug build records SS_EBOUNDS, the normal build nothing; read it with device_status."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _check(lib().ss_selftest_bounds(_stream(dev, stream)), "ss_selftest_bounds")


def debug_bounds_build() -> bool:
    """Whether the loaded library is the debug build (SS_DEBUG_BOUNDS)."""
    return bool(lib().ss_debug_bounds_build())


def selftest_wait_timeout(device=None, stream=None):
    """Launch the diagnostic bounded wait that runs out (ss_selftest_wait_timeout) on
    ``device`` (default: the current CUDA device); read the outcome with device_status."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        _check(lib().ss_selftest_wait_timeout(_stream(dev, stream)), "ss_selftest_wait_timeout")


def measure_ex2(blocks: int, iters: int, *, sink=None, stream=None) -> int:
    """Launch the exp2 throughput kernel (ss_measure_ex2) on the current device and
    stream; returns the number of ex2.approx.ftz.f32 it computes.  Time the launch with
    CUDA events on the same stream."""
    dev = torch.device("cuda", torch.cuda.current_device())
    if sink is None:
        sink = torch.empty((blocks,), dtype=torch.float32, device=dev)
    n = ctypes.c_uint64(0)
    _check(lib().ss_measure_ex2(int(blocks), int(iters), sink.data_ptr(), ctypes.byref(n), _stream(dev, stream)),
           "ss_measure_ex2")
    return int(n.value)


def causal_conv1d(x, weight, bias=None, silu=True, *, out=None, stream=None):
    """Causal depthwise convolution of width 4 (weight[:, 3] on the current step),
    plus bias, then SiLU when ``silu`` (ss_causal_conv1d).  x (batch, dim, L) fp32
    or bf16; weight (dim, 4) fp32; bias (dim,) fp32.  Returns out, x's dtype."""
    if not isinstance(x, torch.Tensor) or x.dim() != 3:
        raise ValueError("x must be a (batch, dim, seqlen) tensor")
    if x.device.type != "cuda":
        raise ValueError("the convolution runs on a CUDA device only; x is on " + str(x.device))
    batch, dim, L = x.shape
    code = _dtype_code(x)
    _need(x, "x", (batch, dim, L), x.dtype, x.device)
    _need(weight, "weight", (dim, 4), torch.float32, x.device)
    _need(bias, "bias", (dim,), torch.float32, x.device)
    if out is None:
        out = torch.empty_like(x)
    _need(out, "out", (batch, dim, L), x.dtype, x.device)
    dims = Dims(batch, dim, 0, L, code)
    st = lib().ss_causal_conv1d(ctypes.byref(dims), _ptr(x), _ptr(weight), _ptr(bias), int(bool(silu)), _ptr(out),
                                _stream(x.device, stream))
    _check(st, "ss_causal_conv1d")
    return out
