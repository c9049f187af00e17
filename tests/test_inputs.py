"""The seeded input generators: deterministic, with the stated shapes and distributions."""
import math

import torch

from selective_state_space_117_b300 import inputs as I


def test_tiny_workload_shapes_and_determinism():
    p = I.workload("tiny_fp32")
    q = I.workload("tiny_fp32")
    assert p.u.shape == (1, 16, 64) and p.B.shape == (1, 4, 64) and p.A.shape == (16, 4)
    assert p.z is None and p.u.dtype == torch.float32
    for a, b in ((p.u, q.u), (p.delta, q.delta), (p.B, q.B), (p.delta_bias, q.delta_bias), (p.D, q.D)):
        assert torch.equal(a, b)
    assert torch.equal(p.A[3], -torch.arange(1, 5, dtype=torch.float32))


def test_bias_is_inverse_softplus_of_uniform_step():
    p = I.workload("medium_fp32_gate")
    dt0 = torch.nn.functional.softplus(p.delta_bias.double())
    assert float(dt0.min()) >= 1e-3 - 1e-6 and float(dt0.max()) <= 1e-1 + 1e-6
    assert p.z is not None and torch.equal(p.D, torch.ones(256))
    assert abs(float(p.B.std()) - 0.25) < 0.01


def test_bf16_workload_and_lti():
    p = I.workload("mamba130m_layer_bf16", batch=1, dim=8, seqlen=32)
    assert p.u.dtype == torch.bfloat16 and p.A.dtype == torch.float32 and p.delta_bias.dtype == torch.float32
    assert torch.allclose(p.A[0], -torch.arange(1, 17, dtype=torch.float32))
    lti = I.lti_problem(batch=1, dim=4, seqlen=10)
    assert torch.equal(lti.B[:, :, 0], lti.B[:, :, 9]) and torch.equal(lti.delta[:, :, 0], lti.delta[:, :, 5])
    w = I.to_wire(p.u)
    assert w.dtype.name == "uint16" and w.shape == (1, 8, 32)


def test_decode_stream_small():
    s = I.decode_stream(batch=2, dim=3, dstate=4, steps=5)
    assert s.u.shape == (5, 2, 3) and s.B.shape == (5, 2, 4) and s.u.dtype == torch.bfloat16
    t = I.decode_stream(batch=2, dim=3, dstate=4, steps=5)
    assert torch.equal(s.z, t.z)
