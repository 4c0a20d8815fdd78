"""Planted mistakes in the oracle must each fail at least one pin.

Each case rewrites one spot of ssm_oracle.c (a dropped term, a wrong sign, a wrong index, a swapped
operand ...), compiles that variant into a temporary directory and runs every pin against it. The real
oracle source is never modified.
"""
import os
import subprocess

import pytest

import oracle
from oracle_pins import ALL_PINS

MUTANTS = {
    "drop_input_term": ("h[n] = abar * h[n] + oracle_bbar_x(dt, A[n], ld(B, bc + n, is_f64), xt, disc);",
                        "h[n] = abar * h[n];"),
    "A_positive": ("A[n] = -exp(ld(A_log, d * N + n, is_f64));", "A[n] = exp(ld(A_log, d * N + n, is_f64));"),
    "A_log_transposed": ("A[n] = -exp(ld(A_log, d * N + n, is_f64));", "A[n] = -exp(ld(A_log, n * D + d, is_f64));"),
    "readout_before_update": (
        "                h[n] = abar * h[n] + oracle_bbar_x(dt, A[n], ld(B, bc + n, is_f64), xt, disc);\n"
        "                yt += ld(C, bc + n, is_f64) * h[n];",
        "                yt += ld(C, bc + n, is_f64) * h[n];\n"
        "                h[n] = abar * h[n] + oracle_bbar_x(dt, A[n], ld(B, bc + n, is_f64), xt, disc);"),
    "zoh_as_euler": ("if (disc == ORACLE_ZOH) {", "if (0) {"),
    "euler_as_zoh": ("    return dlt * b_n * x;\n}", "    return expm1(dlt * a_n) / a_n * b_n * x;\n}"),
    "zoh_missing_divide": ("return expm1(dlt * a_n) / a_n * b_n * x;", "return expm1(dlt * a_n) * b_n * x;"),
    "zoh_exp_not_expm1": ("return expm1(dlt * a_n) / a_n * b_n * x;", "return exp(dlt * a_n) / a_n * b_n * x;"),
    "B_from_C": ("oracle_bbar_x(dt, A[n], ld(B, bc + n, is_f64), xt, disc);",
                 "oracle_bbar_x(dt, A[n], ld(C, bc + n, is_f64), xt, disc);"),
    "BC_lag_one_step": ("int64_t bc = (b * L + t) * N;", "int64_t bc = (b * L + (t > 0 ? t - 1 : 0)) * N;"),
    "x_delta_swapped": ("double xt = ld(x, (b * L + t) * D + d, is_f64);",
                        "double xt = ld(delta, (b * L + t) * D + d, is_f64);"),
    "abar_without_A": ("double abar = exp(dt * A[n]);", "double abar = exp(-dt);"),
    "h0_ignored": ("h[n] = h0 ? h0[k * N + n] : 0.0;", "h[n] = 0.0;"),
    "step_drops_decay": ("double hn = abar * state[k * N + n] +", "double hn = state[k * N + n] +"),
    "step_reads_old_state": (
        "            state[k * N + n] = hn;\n            yt += ld(C_t, b * N + n, is_f64) * hn;",
        "            yt += ld(C_t, b * N + n, is_f64) * state[k * N + n];\n            state[k * N + n] = hn;"),
    "softplus_dropped": ("    if (!softplus) return v;\n", "    return v;\n"),
    "delta_bias_ignored": ("double v = raw + (bias ? bias[d] : 0.0);", "double v = raw;"),
    "skip_dropped": ("double out = yssm + (dskip ? dskip[d] * x : 0.0);", "double out = yssm;"),
    "gate_sigmoid_not_silu": ("out *= zv / (1.0 + exp(-zv));", "out *= 1.0 / (1.0 + exp(-zv));"),
    "gate_sign_flipped": ("out *= zv / (1.0 + exp(-zv));", "out *= zv / (1.0 + exp(zv));"),
    "bwd_hprev_is_h": ("double hprev = t > 0 ? H[(t - 1) * N + n]", "double hprev = t > 0 ? H[t * N + n]"),
    "bwd_adjoint_without_decay": ("mu[n] = abar * lam[n];", "mu[n] = lam[n];"),
    "bwd_zoh_dA_term_dropped": ("dA[n] += g_bbar * Bn * dt * dt * oracle_zoh_dA_factor(dt * A[n]);", ""),
    "bwd_zoh_series_wrong": ("0.5 + w * (1.0 / 3.0", "0.5 + w * (1.0 / 2.0"),
    "bwd_euler_ddelta_input_term": ("gdt += g_bbar * Bn;", ""),
    "bwd_zoh_ddelta_without_abar": ("gdt += g_bbar * abar * Bn;", "gdt += g_bbar * Bn;"),
    "bwd_dA_log_chain_sign": ("dA_log_out[k * N + n] = dA[n] * A[n];", "dA_log_out[k * N + n] = -dA[n] * A[n];"),
    "bwd_dfinal_ignored": ("mu[n] = dfinal ? dfinal[k * N + n] : 0.0;", "mu[n] = 0.0;"),
    "bwd_dC_uses_previous_state": ("dC_out[(k * L + t) * N + n] = dyt * H[t * N + n];",
                                   "dC_out[(k * L + t) * N + n] = dyt * hprev;"),
    "bwd_dx_missing_B": ("gx += lam[n] * bfac * Bn;", "gx += lam[n] * bfac;"),
    "bwd_dh0_undecayed": ("if (dh0_out) dh0_out[k * N + n] = mu[n];", "if (dh0_out) dh0_out[k * N + n] = lam[n];"),
    "ssd_decay_dropped": ("S[p * N + n] = abar * S[p * N + n] + coef", "S[p * N + n] = S[p * N + n] + coef"),
    "ssd_x_of_wrong_head": ("double xv = ld(x, ((b * L + t) * H + hh) * P + p, is_f64);",
                            "double xv = ld(x, ((b * L + t) * H + (hh + 1) % H) * P + p, is_f64);"),
    "ssd_delta_of_head_zero": ("double dt = ld(delta, (b * L + t) * H + hh, is_f64);",
                               "double dt = ld(delta, (b * L + t) * H, is_f64);"),
    "ssd_readout_uses_B": ("yv += ld(C, (b * L + t) * N + n, is_f64) * S[p * N + n];",
                           "yv += ld(B, (b * L + t) * N + n, is_f64) * S[p * N + n];"),
    "ssd_h0_ignored": ("for (int64_t i = 0; i < P * N; ++i) S[i] = h0 ? h0[k * P * N + i] : 0.0;",
                       "for (int64_t i = 0; i < P * N; ++i) S[i] = 0.0;"),
    "bwd_dy_lagged": ("double dyt = ld(dy, (b * L + t) * D + d, is_f64);",
                      "double dyt = ld(dy, (b * L + (t > 0 ? t - 1 : 0)) * D + d, is_f64);"),
    "channel_index_swapped": ("int64_t b = flat / D, d = flat % D;\n        double h[",
                              "int64_t d = flat / D, b = flat % D;\n        double h["),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new, 1)
    path = tmp_path / "mut.c"
    path.write_text(mutated)
    lib = str(tmp_path / f"liboracle_{name}.so")
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-o", lib, str(path), "-lm"], check=True)
    mut = oracle.Oracle(lib)
    caught = []
    for pin in ALL_PINS:
        try:
            pin(mut)
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"


def test_real_oracle_passes_every_pin(orc):
    for pin in ALL_PINS:
        pin(orc)
