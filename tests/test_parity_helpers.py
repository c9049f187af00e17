"""The streamed comparisons of tests/parity.py reach the same outcome as the
whole-array ones, whatever the split into blocks (no GPU needed)."""
import numpy as np
import pytest

from parity import (TOL_BF16, TOL_BF16_OUT, TOL_F32, StreamCheck, StreamCheckBf16Out, check, check_bf16_out,
                    err_bf16, err_f32, rel_unfloored)


def _cases(seed):
    rng = np.random.default_rng(seed)
    ref = rng.standard_normal(5000) * np.exp(rng.uniform(-6, 2, 5000))
    ref[::97] = 0.0
    return rng, ref


def _stream(cls_args, y, ref, rng, cls=StreamCheck):
    cuts = np.sort(rng.choice(np.arange(1, ref.size), size=6, replace=False))
    sc = cls(*cls_args)
    for yb, rb in zip(np.split(y, cuts), np.split(ref, cuts)):
        sc.add(yb, rb)
    return sc


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("bf16", [False, True])
def test_stream_check_matches_check(seed, bf16):
    rng, ref = _cases(seed)
    tol = TOL_BF16 if bf16 else TOL_F32
    r = np.sqrt(np.mean(ref * ref))
    for scale in (0.3, 0.9, 1.1, 3.0):
        # errors near the bound: some elements pass only through the rms floor
        noise = rng.standard_normal(ref.size)
        if bf16:
            y = ref + noise / np.max(np.abs(noise)) * tol * r * scale
            whole = err_bf16(y, ref) <= tol
        else:
            y = ref + noise * np.maximum(np.abs(ref), r) * tol * scale / 3.0
            whole = err_f32(y, ref) <= tol
        sc = _stream(("t", bf16), y, ref, rng)
        try:
            sc.finish()
            streamed = True
        except AssertionError:
            streamed = False
        assert streamed == whole, (scale, streamed, whole)


@pytest.mark.parametrize("seed", range(4))
def test_stream_check_bf16_out_matches(seed):
    rng, ref = _cases(100 + seed)
    r = np.sqrt(np.mean(ref * ref))
    for scale in (0.5, 0.99, 1.01, 2.0):
        noise = rng.uniform(-1, 1, ref.size)
        y = ref + noise * (TOL_BF16_OUT * np.abs(ref) + 1e-5 * r) * scale
        try:
            check_bf16_out(y, ref, "t")
            whole = True
        except AssertionError:
            whole = False
        sc = _stream(("t",), y, ref, rng, cls=StreamCheckBf16Out)
        try:
            sc.finish()
            streamed = True
        except AssertionError:
            streamed = False
        assert streamed == whole, (scale, streamed, whole)


def test_rel_unfloored_ignores_small_refs():
    ref = np.array([1.0, -2.0, 1e-9, 0.0])
    y = np.array([1.0 + 1e-6, -2.0, 1e-6, 1e-6])
    assert rel_unfloored(y, ref, 1e-3) == pytest.approx(1e-6)
    assert check(y[:2], ref[:2], False, "t") <= TOL_F32
