"""GPU parity of the zero-order-hold discretisation (SS_FLAG_ZOH) against the
fp64 oracle, on every path: the forward scan under both schedules (one thread per
channel with TMA or ring staging, one warp per channel), the chunked scan (TMA and
ring local passes), and the decode step; plus Theorem 1 on the GPU."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import selective_state_space_117_b300 as ss
from selective_state_space_117_b300 import inputs as I
from parity import StreamCheck, check, host
from fullsize import compare_scans

pytestmark = pytest.mark.gpu
DEV = "cuda"


def problem(seed, batch, dim, N, L, dtype, spread=False):
    p = I.selective_problem("zoh", seed=seed, batch=batch, dim=dim, dstate=N, seqlen=L, dtype=dtype, bc_std=0.5,
                            d_mode="normal", gate=True, device=DEV, gen_device="cpu")
    g = torch.Generator().manual_seed(seed + 500)
    if spread:   # decay rates from -0.01 to -50: both branches of the hold weight
        n = torch.arange(N, dtype=torch.float32)
        row = -0.01 * torch.exp(n * (math.log(5000.0) / max(N - 1, 1)))
        p.A = row.unsqueeze(0).expand(dim, N).contiguous().to(DEV)
    else:
        p.A = (-torch.exp(torch.rand((dim, N), generator=g) * 3.0 - 1.5)).to(DEV)
    return p


def oracle_zoh(p, h0=None):
    w = I.to_wire
    return oracle.scan(w(p.u), w(p.delta), w(p.A), w(p.B), w(p.C), D=w(p.D), z=w(p.z), delta_bias=w(p.delta_bias),
                       dtype="bf16" if p.in_dtype == I.BF16 else "f32", h0=h0, zoh=True)


CASES = [
    # seed, batch, dim, N, L, dtype, spread
    (1, 2, 96, 16, 512, torch.float32, True),
    (2, 1, 130, 16, 1024, torch.bfloat16, True),
    (3, 2, 40, 5, 77, torch.float32, False),      # ring path (L % 8 != 0)
    (4, 1, 64, 64, 96, torch.bfloat16, True),
    (5, 1, 30, 5, 520, torch.float32, True),      # a last 512-step segment of 8 steps
]


@pytest.mark.parametrize("case", CASES, ids=[f"s{c[0]}d{c[2]}n{c[3]}L{c[4]}" for c in CASES])
@pytest.mark.parametrize("impl,chunk", [("fwd", None), ("fwd_thread", None), ("fwd_warp", None), ("chunked", 64),
                                        ("chunked", 7)])
def test_zoh_scan_matches_oracle(case, impl, chunk):
    seed, batch, dim, N, L, dtype, spread = case
    p = problem(seed, batch, dim, N, L, dtype, spread)
    kw = dict(D=p.D, z=p.z, delta_bias=p.delta_bias, return_last_state=True, zoh=True)
    if impl == "fwd_warp" and (L % 8 or N > 16):   # outside the warp schedule: refused on the host
        with pytest.raises(ss.SSError) as ei:
            ss.scan_fwd(p.u, p.delta, p.A, p.B, p.C, schedule="warp", **kw)
        assert ei.value.status == ss.SS_EINVAL
        return
    if impl.startswith("fwd"):
        y, hl = ss.scan_fwd(p.u, p.delta, p.A, p.B, p.C, schedule=impl[4:] or None, **kw)
    else:
        y, hl = ss.scan_chunked(p.u, p.delta, p.A, p.B, p.C, chunk_len=chunk, **kw)
    yr, hr = oracle_zoh(p.to("cpu"))
    bf = dtype == torch.bfloat16
    check(host(y).reshape(batch * dim, L), yr, bf, f"zoh/{impl} y")
    check(host(hl).reshape(batch * dim, N), hr, bf, f"zoh/{impl} state")


@pytest.mark.parametrize("impl", ["warp", "thread", "chunked"])
def test_zoh_initial_state(impl):
    """The zero-order hold started from a given state h0, on every forward path."""
    p = problem(31, 2, 24, 16, 264, torch.bfloat16, spread=True)
    g = torch.Generator().manual_seed(32)
    h0 = torch.randn((2, 24, 16), generator=g)
    kw = dict(D=p.D, z=p.z, delta_bias=p.delta_bias, return_last_state=True, zoh=True, h0=h0.to(DEV))
    if impl == "chunked":
        y, hl = ss.scan_chunked(p.u, p.delta, p.A, p.B, p.C, chunk_len=48, **kw)
    else:
        y, hl = ss.scan_fwd(p.u, p.delta, p.A, p.B, p.C, schedule=impl, **kw)
    yr, hr = oracle_zoh(p.to("cpu"), h0=h0.double().numpy().reshape(48, 16))
    check(host(y).reshape(48, 264), yr, True, f"zoh h0/{impl} y")
    check(host(hl).reshape(48, 16), hr, True, f"zoh h0/{impl} state")


@pytest.mark.parametrize("N", [1, 8, 16, 40])
def test_zoh_decode_matches_oracle(N):
    p = problem(20 + N, 3, 70, N, 12, torch.float32, spread=N > 1)
    st = torch.zeros((3, 70, N), device=DEV)
    sref = np.zeros((210, N))
    w = I.to_wire
    for t in range(12):
        col = lambda x: x[:, :, t].contiguous()
        y = ss.state_update(st, col(p.u), col(p.delta), p.A, col(p.B), col(p.C), D=p.D, z=col(p.z),
                            delta_bias=p.delta_bias, zoh=True)
        yr = oracle.state_update(sref, w(col(p.u)), w(col(p.delta)), w(p.A), w(col(p.B)), w(col(p.C)), D=w(p.D),
                                 z=w(col(p.z)), delta_bias=w(p.delta_bias), zoh=True)
        check(host(y).reshape(-1), yr, False, f"zoh decode step {t}")
    check(host(st).reshape(210, N), sref, False, "zoh decode state")


def test_zoh_theorem1_on_gpu():
    """N = 1, A = -1, B = C = 1, dt = softplus(g): the GPU scan is the gated RNN
    h_t = (1 - sigmoid(g_t)) h_{t-1} + sigmoid(g_t) x_t (Theorem 1 of azimuth.plus)."""
    g = torch.Generator().manual_seed(77)
    dim, L = 64, 256
    x = torch.randn((1, dim, L), generator=g)
    gate = torch.randn((1, dim, L), generator=g) * 2.0
    one = torch.ones((1, 1, L))
    A = -torch.ones((dim, 1))
    for impl in ("warp", "thread", "chunked"):
        kw = dict(return_last_state=True, zoh=True)
        args = (x.to(DEV), gate.to(DEV), A.to(DEV), one.to(DEV), one.to(DEV))
        y, _ = ss.scan_chunked(*args, chunk_len=64, **kw) if impl == "chunked" else ss.scan_fwd(*args, schedule=impl,
                                                                                               **kw)
        s = torch.sigmoid(gate.double())
        h = torch.zeros((1, dim), dtype=torch.float64)
        want = []
        for t in range(L):
            h = (1 - s[:, :, t]) * h + s[:, :, t] * x[:, :, t].double()
            want.append(h)
        want = torch.stack(want, dim=2)
        err = torch.max(torch.abs(y.double().cpu() - want) / torch.clamp(torch.abs(want), min=want.abs().mean()))
        assert err.item() <= 1e-4, (impl, err.item())


def test_zoh_two_faces_agree():
    """L decode steps with the hold weight == the ZOH scan."""
    p = problem(90, 2, 50, 16, 64, torch.float32, spread=True)
    yf, hf = ss.scan_fwd(p.u, p.delta, p.A, p.B, p.C, D=p.D, z=p.z, delta_bias=p.delta_bias, return_last_state=True,
                         zoh=True)
    st = torch.zeros((2, 50, 16), device=DEV)
    ys = [ss.state_update(st, p.u[:, :, t].contiguous(), p.delta[:, :, t].contiguous(), p.A,
                          p.B[:, :, t].contiguous(), p.C[:, :, t].contiguous(), D=p.D, z=p.z[:, :, t].contiguous(),
                          delta_bias=p.delta_bias, zoh=True) for t in range(64)]
    check(host(torch.stack(ys, dim=2)), host(yf), False, "zoh decode x L vs fwd")
    check(host(st), host(hf), False, "zoh decode state vs fwd")


def test_zoh_long_sequence_full():
    """The long-sequence workload (batch 1, D 5120, N 16, L 65536, bf16) with the hold weight
    through the chunked scan at chunk 2048, the benchmark's launch configuration: every
    element of y and every final state against the oracle's ZOH scan."""
    p = I.workload("mamba2p8b_long_bf16", device=DEV, gen_device="cuda")
    y, hl = ss.scan_chunked(p.u, p.delta, p.A, p.B, p.C, D=p.D, z=p.z, delta_bias=p.delta_bias, chunk_len=2048,
                            return_last_state=True, zoh=True)
    torch.cuda.synchronize()
    compare_scans(p, {"chunked2048": (y, hl)}, "zoh mamba2p8b_long", zoh=True)
    del y, hl, p
    torch.cuda.empty_cache()


def test_zoh_decode_stream_full_size():
    """256 sequential decode steps with the hold weight on the (256, 5120, 16) state of the
    decode workload: every step's y over all channels and the whole final state against the
    oracle's ZOH recurrence."""
    steps = 256
    st_in = I.decode_stream(seed=4, batch=256, dim=5120, dstate=16, steps=steps, device=DEV, gen_device="cuda")
    state = torch.zeros((256, 5120, 16), device=DEV)
    y = torch.empty((256, 5120), device=DEV)
    w = I.to_wire
    A, Dv, bias = w(st_in.A), w(st_in.D), w(st_in.delta_bias)
    sref = np.zeros((256 * 5120, 16))
    cy = StreamCheck("zoh decode_256x5120 y (256 steps, all channels)", True)
    for t in range(steps):
        ss.state_update(state, st_in.u[t], st_in.delta[t], st_in.A, st_in.B[t], st_in.C[t], D=st_in.D,
                        z=st_in.z[t], delta_bias=st_in.delta_bias, y=y, zoh=True)
        yg = host(y).reshape(-1)
        yr = oracle.state_update(sref, w(st_in.u[t]), w(st_in.delta[t]), A, w(st_in.B[t]), w(st_in.C[t]), D=Dv,
                                 z=w(st_in.z[t]), delta_bias=bias, dtype="bf16", zoh=True)
        cy.add(yg, yr)
    cy.finish()
    check(host(state).reshape(-1, 16), sref, True, "zoh decode_256x5120 final state (all channels)")
    del st_in, state
    torch.cuda.empty_cache()
