"""Full-size comparisons of GPU outputs with the oracle, streamed over channel blocks.

The oracle computes every channel of the workload (channels are independent, so
it runs block by block over lists of flattened channel indices b * dim + d), and
each block of every GPU output is compared with it under the rules of
tests/parity.py (StreamCheck gives the outcome of a whole-array check).  Nothing
is sampled: every output element and every final state is compared.
"""
from __future__ import annotations

import numpy as np

import oracle
from selective_state_space_117_b300 import inputs as I
from parity import StreamCheck, host

BLOCK = 512


def wire_problem(p: I.Problem):
    """Host copies of every input in the oracle's wire format (made once per problem)."""
    w = I.to_wire
    return dict(u=w(p.u), delta=w(p.delta), z=w(p.z), B=w(p.B), C=w(p.C), A=w(p.A), D=w(p.D),
                delta_bias=w(p.delta_bias), softplus=p.softplus,
                dtype="bf16" if p.in_dtype == I.BF16 else "f32")


def oracle_blocks(p: I.Problem, zoh=False, block=BLOCK, wire=None):
    """(b, d0, d1, y_ref (d1 - d0, L), h_ref (d1 - d0, N)) over every channel block."""
    wp = wire or wire_problem(p)
    for b in range(p.batch):
        for d0 in range(0, p.dim, block):
            d1 = min(p.dim, d0 + block)
            chans = np.arange(b * p.dim + d0, b * p.dim + d1, dtype=np.int64)
            yr, hr = oracle.scan(wp["u"], wp["delta"], wp["A"], wp["B"], wp["C"], D=wp["D"], z=wp["z"],
                                 delta_bias=wp["delta_bias"], softplus=wp["softplus"], dtype=wp["dtype"],
                                 chans=chans, zoh=zoh)
            yield b, d0, d1, yr, hr


def compare_scans(p: I.Problem, outs: dict, label: str, zoh=False, block=BLOCK):
    """Every element of y and every final state of each GPU run in `outs` (name -> (y, last_state),
    device tensors (batch, dim, L) and (batch, dim, N)) against the oracle's scan of p."""
    bf = p.in_dtype == I.BF16
    chk = {n: (StreamCheck(f"{label}/{n} y", bf), StreamCheck(f"{label}/{n} last_state", bf)) for n in outs}
    for b, d0, d1, yr, hr in oracle_blocks(p, zoh=zoh, block=block):
        for n, (y, hl) in outs.items():
            chk[n][0].add(host(y[b, d0:d1]), yr)
            chk[n][1].add(host(hl[b, d0:d1]), hr)
    return {n: (cy.finish(), ch.finish()) for n, (cy, ch) in chk.items()}
