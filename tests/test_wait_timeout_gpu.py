"""The failure path of the bounded device-side waits, made to run out on purpose.

ss_selftest_wait_timeout launches one thread that waits, with the library's bounded
mbarrier wait, on a barrier that nothing ever arrives on.  The wait must give up,
record SS_ETIMEOUT in the device status word and return; the status word must read
back through ss_device_status, clear on request, and the device must stay usable (a
scan right after it still matches the oracle).  Nothing here faults or hangs: the
wait's limit ends it.
"""
from __future__ import annotations

import time

import pytest
import torch

import selective_state_space_117_b300 as ss
from selective_state_space_117_b300 import inputs as I
from parity import check, host
import oracle

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports():
    assert ss.device_status(clear=True) in (ss.SS_OK, ss.SS_ETIMEOUT)
    assert ss.device_status() == ss.SS_OK
    t0 = time.perf_counter()
    ss.selftest_wait_timeout()
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert ss.device_status() == ss.SS_ETIMEOUT          # recorded ...
    assert ss.device_status(clear=True) == ss.SS_ETIMEOUT
    assert ss.device_status() == ss.SS_OK                # ... and cleared
    # the limit is one second of the global timer
    assert 0.9 < waited < 10.0, f"the bounded wait gave up after {waited:.2f} s"
    print(f"bounded wait gave up after {waited:.3f} s")

    # the context is still usable: a small scan afterwards matches the oracle
    p = I.workload("tiny_fp32", device="cuda", gen_device="cpu")
    y, hl = ss.scan_fwd(p.u, p.delta, p.A, p.B, p.C, D=p.D, z=p.z, delta_bias=p.delta_bias,
                        return_last_state=True)
    w = I.to_wire
    yr, hr = oracle.scan(w(p.u), w(p.delta), w(p.A), w(p.B), w(p.C), D=w(p.D), z=w(p.z),
                         delta_bias=w(p.delta_bias))
    check(host(y).reshape(yr.shape), yr, False, "scan after the timeout")
    check(host(hl).reshape(hr.shape), hr, False, "state after the timeout")
    assert ss.device_status() == ss.SS_OK
