"""The oracle's pins must reject plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (a dropped term, a wrong
sign, a transposed index, the readout taken before the update, ...), builds it in a
temporary directory, and checks that at least one pin test fails against that build.
"""
import os
import subprocess

import pytest

from oracle import oracle
import tests.test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "ssm_oracle.c")

MUTANTS = {
    "drop_D_skip": ("if (D) acc += D[d] * x;\n      if (z_row)", "if (z_row)"),
    "A_sign": ("double abar = exp(dt * a);\n        double bx", "double abar = exp(-dt * a);\n        double bx"),
    "B_transposed": ("double bx = bbar_factor(dt, a, zoh) * B[((long)b * dstate + n) * seqlen + t] * x;",
                     "double bx = bbar_factor(dt, a, zoh) * B[((long)b * seqlen + t) * dstate + n] * x;"),
    "C_from_B": ("acc += C[((long)b * dstate + n) * seqlen + t] * h[n];",
                 "acc += B[((long)b * dstate + n) * seqlen + t] * h[n];"),
    "readout_before_update": ("h[n] = abar * h[n] + bx;\n        acc += C[((long)b * dstate + n) * seqlen + t] * h[n];",
                              "acc += C[((long)b * dstate + n) * seqlen + t] * h[n];\n        h[n] = abar * h[n] + bx;"),
    "bias_after_softplus": ("if (dt_bias) v += dt_bias[d];\n  if (use_softplus) v = softplus_f64(v);",
                            "if (use_softplus) v = softplus_f64(v);\n  if (dt_bias) v += dt_bias[d];"),
    "softplus_wrong_branch": ("if (x > 0.0) return x + log1p(exp(-x));", "if (x > 0.0) return log1p(exp(-x));"),
    "silu_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "bbar_missing_delta": ("if (!zoh || a == 0.0) return dt;", "if (!zoh || a == 0.0) return 1.0;"),
    "zoh_exp_not_expm1": ("return expm1(dt * a) / a;", "return exp(dt * a) / a;"),
    "zoh_missing_divide": ("return expm1(dt * a) / a;", "return expm1(dt * a);"),
    "zoh_limit_at_zero": ("if (!zoh || a == 0.0) return dt;", "if (!zoh) return dt;\n  if (a == 0.0) return 0.0;"),
    "zoh_ignored": ("if (!zoh || a == 0.0) return dt;\n  return", "if (1) return dt;\n  return"),
    "gate_additive": ("if (z_row) acc *= silu_f64(z_row[t]);", "if (z_row) acc += silu_f64(z_row[t]);"),
    "pair_combine_swapped": ("out_b[i] = ra * lb + rb;", "out_b[i] = la * rb + lb;"),
    "decode_no_state_decay": ("*s = abar * *s + bbar_factor(step, a, zoh) * B[(long)b * dstate + n] * x[ch];",
                              "*s = *s + bbar_factor(step, a, zoh) * B[(long)b * dstate + n] * x[ch];"),
    "conv_taps_reversed": ("acc += weight[(long)d * width + k] * v;", "acc += weight[(long)d * width + (width - 1 - k)] * v;"),
    "conv_off_by_one": ("int s = t - hw + k; /* input time index */", "int s = t - hw + k - 1; /* input time index */"),
    "conv_state_ignored": ("double v = s >= 0 ? xr[s] : (sr ? sr[hw + s] : 0.0);", "double v = s >= 0 ? xr[s] : 0.0;"),
    "conv_no_bias": ("double acc = bias ? bias[d] : 0.0;", "double acc = 0.0;"),
    "bwd_zoh_dc_ddelta": ("          dc_ddt = a;\n", "          dc_ddt = 1.0;\n"),
    "bwd_zoh_dc_da": ("dc_da = fabs(x) < 1e-3 ? dt * dt * (0.5 + x / 3.0 + x * x / 8.0 + x * x * x / 30.0) : (dt * a - c) / an;",
                      "dc_da = 0.0;"),
    "bwd_zoh_small_x_series": ("dt * dt * (0.5 + x / 3.0 + x * x / 8.0 + x * x * x / 30.0)", "dt * dt * (0.5 - x / 3.0)"),
    "bwd_no_carry": ("double lam = dy * C[((long)b * N + n) * L + t] + carry[n];",
                     "double lam = dy * C[((long)b * N + n) * L + t];"),
    "bwd_carry_without_decay": ("carry[n] = lam * a;", "carry[n] = lam;"),
    "bwd_dA_missing_state": ("dA[(long)d * N + n] += lam * (dt * a * hp + dc_da * bn * ur[t]);",
                             "dA[(long)d * N + n] += lam * (dt * a + dc_da * bn * ur[t]);"),
    "bwd_dC_previous_state": ("dC[((long)b * N + n) * L + t] += dy * hs[(t + 1) * N + n];",
                              "dC[((long)b * N + n) * L + t] += dy * hs[t * N + n];"),
    "bwd_softplus_grad": ("double dd = delta_softplus ? ddt / (1.0 + exp(-raw)) : ddt;",
                          "double dd = delta_softplus ? ddt / (1.0 + exp(raw)) : ddt;"),
    "bwd_dsilu": ("return sg * (1.0 + z * (1.0 - sg));", "return sg * (1.0 - sg);"),
    "h0_ignored": ("h[n] = h0 ? h0[ch * dstate + n] : 0.0;", "h[n] = 0.0;"),
}

PIN_TESTS = [getattr(pins, n) for n in dir(pins) if n.startswith("test_")]


def _arglists(fn):
    """Every keyword-argument combination of a test's parametrize marks (their product)."""
    arglists = [{}]
    for m in getattr(fn, "pytestmark", []):
        if m.name != "parametrize":
            continue
        names, values = m.args
        names = [n.strip() for n in names.split(",")] if isinstance(names, str) else list(names)
        combos = [dict(zip(names, v if len(names) > 1 else (v,))) for v in values]
        arglists = [{**a, **c} for a in arglists for c in combos]
    return arglists


def _run_pins():
    failures = 0
    for fn in PIN_TESTS:
        for kw in _arglists(fn):
            try:
                fn(**kw)
            except Exception:  # an assertion or a numerical error both count as a rejection
                failures += 1
    return failures


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mut = tmp_path / "mutant.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared", "-std=c99",
                    "-o", str(lib), str(mut), "-lm"], check=True)
    oracle.use_library(str(lib))
    try:
        assert _run_pins() > 0, f"no pin rejects the planted mistake {name}"
    finally:
        oracle.use_library(None)


def test_unmutated_oracle_passes_all_pins():
    assert _run_pins() == 0
