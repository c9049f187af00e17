"""Mutation check of the oracle pins (no GPU).

Each case below plants one plausible mistake in a private copy of the
oracle's C source (a dropped term, a wrong sign, a wrong or transposed index,
a swapped operand, a reordered step), compiles it with gcc into a temporary
directory and runs every pin against it.  A pin set that lets a mutant
through is too weak; each mutant must fail at least one pin.
"""
import os
import subprocess
import tempfile

import pytest

import oracle
from pins import PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "ss_oracle.c")

# (name, [(text to find, replacement), ...])  -- only the first occurrence is replaced
MUTANTS = [
    ("drop_delta_bias", [("double x = draw + bias;", "double x = draw;")]),
    ("no_softplus", [("double dt = softplus_flag ? sso_softplus(x) : x;", "double dt = x;")]),
    ("softplus_wrong_negative_branch", [("log1p(exp(-fabs(x)))", "log1p(exp(-x))")]),
    ("exp_sign_flipped", [("exp(dt * (double)A_row[n])", "exp(-dt * (double)A_row[n])")]),
    ("exp_missing_dt", [("exp(dt * (double)A_row[n])", "exp((double)A_row[n])")]),
    ("input_term_missing_dt", [("h[n] = Abar * h[n] + wdt * Bn * u;", "h[n] = Abar * h[n] + Bn * u;")]),
    ("B_C_swapped", [("double Bn = sso_widen(B, ", "double Bn = sso_widen(C, "),
                     ("double Cn = sso_widen(C, ", "double Cn = sso_widen(B, ")]),
    ("D_term_dropped", [("y += Dd * u;", "")]),
    ("gate_before_D", [("y += Dd * u;\n    if (has_z) y *= sso_silu(z);", "if (has_z) y *= sso_silu(z);\n    y += Dd * u;")]),
    ("sigmoid_not_silu", [("return z / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(-z));")]),
    ("silu_sign", [("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));")]),
    ("readout_before_update", [("h[n] = Abar * h[n] + wdt * Bn * u;\n        y += Cn * h[n];",
                                "y += Cn * h[n];\n        h[n] = Abar * h[n] + dt * Bn * u;")]),
    ("BC_time_off_by_one", [("B, C, b * dstate * seqlen + t, seqlen,", "B, C, b * dstate * seqlen + (t > 0 ? t - 1 : 0), seqlen,")]),
    ("A_row_wrong_channel", [("A + d * dstate, Dd,", "A + (d % 2) * dstate, Dd,")]),
    ("D_wrong_channel", [("double Dd = D ? (double)D[d] : 0.0;", "double Dd = D ? (double)D[0] : 0.0;")]),
    ("bias_wrong_channel", [("double bias = delta_bias ? (double)delta_bias[d] : 0.0;",
                             "double bias = delta_bias ? (double)delta_bias[0] : 0.0;")]),
    ("bf16_widen_shift", [("<< 16;", "<< 15;")]),
    ("h0_ignored", [("h[n] = h0 ? h0[i * dstate + n] : 0.0;", "h[n] = 0.0;")]),
    ("u_batch_channel_transposed", [("int64_t ix = c * seqlen + t;", "int64_t ix = (d * batch + b) * seqlen + t;")]),
    ("decode_BC_ignores_batch", [("B, C, b * dstate, 1,", "B, C, 0, 1,")]),
    ("decode_u_index", [("double uu = sso_widen(u, c, dtype);", "double uu = sso_widen(u, d, dtype);")]),
    ("zoh_times_A", [("return A != 0.0 ? expm1(dt * A) / A : dt;", "return A != 0.0 ? expm1(dt * A) * A : dt;")]),
    ("zoh_exp_not_expm1", [("return A != 0.0 ? expm1(dt * A) / A : dt;", "return A != 0.0 ? exp(dt * A) / A : dt;")]),
    ("zoh_limit_zero", [("return A != 0.0 ? expm1(dt * A) / A : dt;", "return A != 0.0 ? expm1(dt * A) / A : 0.0;")]),
    ("zoh_flag_ignored", [("double wdt = zoh ? sso_zoh_weight(dt, (double)A_row[n]) : dt;", "double wdt = dt;")]),
    ("conv_taps_reversed", [("(double)w[d * 4 + k] * sso_widen(x", "(double)w[d * 4 + 3 - k] * sso_widen(x")]),
    ("conv_not_causal", [("int64_t src = t - 3 + k;", "int64_t src = t - 2 + k;")]),
    ("conv_bias_dropped", [("double s = bias ? (double)bias[d] : 0.0;", "double s = 0.0;")]),
    ("conv_silu_ignored", [("out[c * seqlen + t] = silu_flag ? sso_silu(s) : s;", "out[c * seqlen + t] = s;")]),
    ("conv_wrong_channel_taps", [("(double)w[d * 4 + k]", "(double)w[(d % 2) * 4 + k]")]),
    # backward pass
    ("bwd_carry_without_decay", [("mu[n] = e * lam;", "mu[n] = lam;")]),
    ("bwd_lam_misses_readout", [("double lam = mu[n] + Cn * ds;", "double lam = mu[n];")]),
    ("bwd_dC_uses_previous_state", [("dCc[n * L + t] = ds * hc[n];", "dCc[n * L + t] = ds * hp[n];")]),
    ("bwd_dB_missing_weight", [("dBc[n * L + t] = lam * w * uu;", "dBc[n * L + t] = lam * uu;")]),
    ("bwd_du_missing_skip", [("double duv = Dd * ds, ddt = 0.0;", "double duv = 0.0, ddt = 0.0;")]),
    ("bwd_ddt_decay_sign", [("ddt += lam * (hp[n] * e * An +", "ddt += lam * (-hp[n] * e * An +")]),
    ("bwd_ddt_missing_input_term", [("ddt += lam * (hp[n] * e * An + Bn * uu * (zoh ? e : 1.0));",
                                     "ddt += lam * (hp[n] * e * An);")]),
    ("bwd_softplus_derivative_dropped", [("double dx = softplus_flag ? ddt * sso_sigmoid(x) : ddt;",
                                          "double dx = ddt;")]),
    ("bwd_dA_missing_dt", [("dAc[n] += lam * (hp[n] * e * dt +", "dAc[n] += lam * (hp[n] * e +")]),
    ("bwd_dA_uses_current_state", [("dAc[n] += lam * (hp[n] * e * dt", "dAc[n] += lam * (hc[n] * e * dt")]),
    ("bwd_zoh_ddt_weight", [("Bn * uu * (zoh ? e : 1.0)", "Bn * uu")]),
    ("bwd_zoh_dA_term_dropped", [("(zoh ? Bn * uu * sso_zoh_weight_dA(dt, An) : 0.0)", "0.0")]),
    ("bwd_zoh_dA_series", [("0.5 + y * (1.0 / 3.0", "0.5 + y * (1.0 / 2.0")]),
    ("bwd_zoh_dA_closed_form", [("return (dt * exp(y) - expm1(y) / A) / A;", "return (dt * exp(y) - expm1(y)) / A;")]),
    ("bwd_dz_silu_derivative", [("sg * (1.0 + zz * (1.0 - sg))", "sg")]),
    ("bwd_dz_without_skip", [("double s = Dd * uu;", "double s = 0.0;")]),
    ("bwd_ds_ignores_gate", [("ds = dy[i * L + t] * zz * sg;", "ds = dy[i * L + t];")]),
    ("bwd_dD_wrong_factor", [("dDc += ds * uu;", "dDc += ds;")]),
    ("bwd_dh0_not_decayed", [("if (dh0) dh0[i * N + n] = mu[n];", "if (dh0) dh0[i * N + n] = mu[n] / exp(dts[0] * (double)Ad[n]);")]),
    ("bwd_dlast_ignored", [("mu[n] = dlast ? dlast[i * N + n] : 0.0;", "mu[n] = 0.0;")]),
    ("bwd_dB_wrong_batch", [("if (dB) dB[b * N * L + k] += dBc[k];", "if (dB) dB[k] += dBc[k];")]),
    ("bwd_dbias_not_summed", [("dbc += dx;", "dbc = dx;")]),
]


def _mutate(src, edits):
    for find, repl in edits:
        assert find in src, f"mutation anchor not found: {find!r}"
        src = src.replace(find, repl, 1)
    return src


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, edits, source):
    mutated = _mutate(source, edits)
    assert mutated != source
    with tempfile.TemporaryDirectory() as td:
        c = os.path.join(td, "m.c")
        so = os.path.join(td, "libm.so")
        with open(c, "w") as f:
            f.write(mutated)
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", so, c, "-lm"])
        orc = oracle.Variant(so)
        caught = []
        for pin in PINS:
            try:
                pin(orc)
            except (AssertionError, ValueError, FloatingPointError) as e:   # noqa: PERF203
                caught.append(pin.__name__)
        assert caught, f"mutant {name} passed every pin"
