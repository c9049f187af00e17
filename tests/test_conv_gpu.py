"""GPU parity of the causal depthwise convolution (ss_causal_conv1d) against the
fp64 oracle, and of the block's branch A (convolution -> SiLU -> selective scan)
against the composition of the two oracles."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import selective_state_space_117_b300 as ss
from selective_state_space_117_b300 import inputs as I
from parity import StreamCheckBf16Out, check, check_bf16_out, host

pytestmark = pytest.mark.gpu
DEV = "cuda"


def conv_case(seed, batch, dim, L, dtype, with_bias=True):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((batch, dim, L), generator=g).to(dtype)
    w = torch.randn((dim, 4), generator=g) * 0.5
    b = torch.randn((dim,), generator=g) * 0.3 if with_bias else None
    return x, w, b


CASES = [
    # seed, batch, dim, L, dtype, bias, silu
    (1, 2, 96, 2048, torch.bfloat16, True, True),
    (2, 1, 64, 8192 * 2 + 256, torch.bfloat16, True, True),      # several segments per row
    (3, 3, 17, 1000, torch.float32, False, True),                  # ragged tail, L % 8 == 0
    (4, 2, 5, 37, torch.float32, True, False),                     # L % 8 != 0: scalar path
    (5, 1, 33, 3, torch.bfloat16, True, True),                     # shorter than the filter
    (6, 1, 8, 8192 * 3 + 77, torch.float32, True, True),           # segments plus a ragged end
]


@pytest.mark.parametrize("case", CASES, ids=[f"s{c[0]}b{c[1]}d{c[2]}L{c[3]}" for c in CASES])
def test_conv1d_matches_oracle(case):
    seed, batch, dim, L, dtype, with_bias, silu_on = case
    x, w, b = conv_case(seed, batch, dim, L, dtype, with_bias)
    out = ss.causal_conv1d(x.to(DEV), w.to(DEV), None if b is None else b.to(DEV), silu=silu_on)
    torch.cuda.synchronize()
    ref = oracle.conv1d(I.to_wire(x), I.to_wire(w), I.to_wire(b), silu=silu_on,
                        dtype="bf16" if dtype == torch.bfloat16 else "f32")
    if dtype == torch.bfloat16:
        check_bf16_out(host(out), ref, "conv1d")
    else:
        check(host(out).reshape(-1, L), ref.reshape(-1, L), False, "conv1d")


def test_conv1d_unaligned_rows():
    """Rows starting one element past an allocation take the scalar path."""
    x, w, b = conv_case(7, 2, 12, 64, torch.bfloat16)
    flat = torch.empty(x.numel() + 1, dtype=torch.bfloat16, device=DEV)
    xs = flat[1:].view(x.shape)
    xs.copy_(x.to(DEV))
    out = ss.causal_conv1d(xs, w.to(DEV), b.to(DEV))
    ref = oracle.conv1d(I.to_wire(x), I.to_wire(w), I.to_wire(b), dtype="bf16")
    check_bf16_out(host(out), ref, "conv1d unaligned")


def test_branch_a_conv_then_scan():
    """Branch A of the block: u = silu(conv(x)), then the scan with the gate, against
    oracle.conv1d followed by oracle.scan on the same rounded u."""
    g = torch.Generator().manual_seed(9)
    batch, dim, N, L = 2, 128, 16, 1024
    x = torch.randn((batch, dim, L), generator=g).to(torch.bfloat16)
    w = torch.randn((dim, 4), generator=g) * 0.5
    cb = torch.randn((dim,), generator=g) * 0.2
    p = I.selective_problem("branch_a", seed=10, batch=batch, dim=dim, dstate=N, seqlen=L, dtype=torch.bfloat16,
                            bc_std=0.25, d_mode="ones", gate=True, device=DEV, gen_device="cpu")
    u = ss.causal_conv1d(x.to(DEV), w.to(DEV), cb.to(DEV))
    y, hl = ss.scan_fwd(u, p.delta, p.A, p.B, p.C, D=p.D, z=p.z, delta_bias=p.delta_bias, return_last_state=True)
    torch.cuda.synchronize()
    uref = oracle.conv1d(I.to_wire(x), I.to_wire(w), I.to_wire(cb), dtype="bf16")
    check_bf16_out(host(u), uref, "branch A conv")
    w_ = I.to_wire
    yr, hr = oracle.scan(w_(u), w_(p.delta), w_(p.A), w_(p.B), w_(p.C), D=w_(p.D), z=w_(p.z),
                         delta_bias=w_(p.delta_bias), dtype="bf16")
    check(host(y).reshape(batch * dim, L), yr, True, "branch A y")
    check(host(hl).reshape(batch * dim, N), hr, True, "branch A state")


def test_conv1d_full_size():
    """The benchmark's shape (batch 1, D 5120, L 65536, bf16 in and out, bias, SiLU) in its
    launch configuration: every output element against the oracle (blocks of 512 rows)."""
    g = torch.Generator(device=DEV).manual_seed(5)
    x = torch.randn((1, 5120, 65536), generator=g, device=DEV).to(torch.bfloat16)
    w = torch.randn((5120, 4), generator=g, device=DEV) * 0.5
    b = torch.randn((5120,), generator=g, device=DEV) * 0.1
    out = ss.causal_conv1d(x, w, b)
    torch.cuda.synchronize()
    chk = StreamCheckBf16Out("conv1d full size (all rows)")
    for d0 in range(0, 5120, 512):
        d1 = d0 + 512
        ref = oracle.conv1d(I.to_wire(x[:, d0:d1]), I.to_wire(w[d0:d1]), I.to_wire(b[d0:d1]), silu=True, dtype="bf16")
        chk.add(host(out[:, d0:d1]), ref)
    chk.finish()
    del x, out
    torch.cuda.empty_cache()
