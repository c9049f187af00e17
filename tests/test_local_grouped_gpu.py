"""GPU checks of the chunked scan's local pass over channels grouped by decay speed.

That pass (used with the softplus on, N <= 16, 16-byte aligned rows and chunks of
whole 16-step tiles) skips a state for a tile only when its weight exp(A R) has
underflowed to exactly 0 in every channel of the warp, so its results cannot
depend on which channels share a warp.  The tests check that (a permutation of
the channels permutes the outputs bit for bit), the state counts that pad to the
next supported width, states that never decay or grow, both input weights, and
chunk lengths from one tile up, all against the oracle.
"""
from __future__ import annotations

import math

import pytest
import torch

import oracle
import selective_state_space_117_b300 as ss
from selective_state_space_117_b300 import inputs as I
from parity import check, host

pytestmark = pytest.mark.gpu
DEV = "cuda"


def problem(seed, batch, dim, N, L, dtype, zoh=False):
    p = I.selective_problem("grouped", seed=seed, batch=batch, dim=dim, dstate=N, seqlen=L, dtype=dtype,
                            bc_std=0.5, d_mode="normal", gate=True, device=DEV, gen_device="cpu")
    g = torch.Generator().manual_seed(seed + 77)
    # decay rates spread over channels and states, step sizes from 1e-3 to 1 over channels
    p.A = (-torch.exp(torch.rand((dim, N), generator=g) * 4.0 - 1.5)).to(DEV)
    p.delta_bias = torch.log(torch.expm1(torch.exp(torch.rand((dim,), generator=g) * math.log(1000.0) -
                                                   math.log(1000.0)))).to(DEV)
    p.extra["zoh"] = zoh
    return p


def run(p, chunk):
    return ss.scan_chunked(p.u, p.delta, p.A, p.B, p.C, D=p.D, z=p.z, delta_bias=p.delta_bias, chunk_len=chunk,
                           return_last_state=True, zoh=p.extra.get("zoh", False))


def against_oracle(p, y, hl, what):
    w = I.to_wire
    bf = p.in_dtype == I.BF16
    yr, hr = oracle.scan(w(p.u), w(p.delta), w(p.A), w(p.B), w(p.C), D=w(p.D), z=w(p.z), delta_bias=w(p.delta_bias),
                         dtype="bf16" if bf else "f32", zoh=p.extra.get("zoh", False))
    n = p.batch * p.dim
    check(host(y).reshape(n, p.seqlen), yr, bf, what + " y")
    check(host(hl).reshape(n, p.dstate), hr, bf, what + " last_state")


@pytest.mark.parametrize("zoh", [False, True], ids=["euler", "zoh"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_channel_order_does_not_change_results(dtype, zoh):
    """The same channels stored in another order give the same outputs, bit for bit, in the
    matching order (the grouping into warps changes, each channel's arithmetic does not)."""
    p = problem(5, 2, 200, 16, 2048, dtype, zoh)
    y, hl = run(p, 256)
    perm = torch.randperm(200, generator=torch.Generator().manual_seed(6)).to(DEV)
    q = I.Problem("grouped_perm", p.u[:, perm].contiguous(), p.delta[:, perm].contiguous(), p.A[perm].contiguous(),
                  p.B, p.C, p.D[perm].contiguous(), p.z[:, perm].contiguous(), p.delta_bias[perm].contiguous(),
                  True, 0, dict(p.extra))
    yq, hq = run(q, 256)
    torch.cuda.synchronize()
    assert torch.equal(yq, y[:, perm]) and torch.equal(hq, hl[:, perm])
    against_oracle(p, y, hl, f"grouped {dtype} zoh={zoh}")


@pytest.mark.parametrize("N", [1, 3, 5, 8, 13, 16])
@pytest.mark.parametrize("zoh", [False, True], ids=["euler", "zoh"])
def test_state_counts(N, zoh):
    p = problem(20 + N, 2, 96, N, 1024, torch.bfloat16, zoh)
    for chunk in (16, 128):
        y, hl = run(p, chunk)
        against_oracle(p, y, hl, f"grouped N={N} chunk={chunk} zoh={zoh}")


def test_states_that_never_decay():
    """A = 0 (never decays, the weight stays 1) and small positive A (grows) in a few channels:
    their warps can never stop early, and the other warps still may."""
    p = problem(40, 1, 160, 16, 3072, torch.float32)
    A = p.A.clone()
    A[3, 0] = 0.0
    A[70, 5] = 0.002
    A[150, :] = 0.0
    p.A = A
    for chunk in (512, 64):
        y, hl = run(p, chunk)
        against_oracle(p, y, hl, f"grouped non-decaying chunk={chunk}")


def test_fast_channels_stop_early():
    """Step sizes near 1 and decay rates near -10: most warps stop after a few tiles of every chunk."""
    p = problem(41, 1, 256, 16, 4096, torch.bfloat16)
    p.delta_bias = torch.full((256,), 1.0, device=DEV)
    p.A = torch.full((256, 16), -10.0, device=DEV)
    p.A[:32] = -0.5             # one slow group
    y, hl = run(p, 1024)
    against_oracle(p, y, hl, "grouped fast channels")
