"""Planted mistakes in the oracle must each fail at least one pin.

Each mutant is a copy of ``oracle/kda_oracle.c`` with one plausible slip
(built with gcc into a temporary directory, on the CPU).  A pin set that lets
a mutant through would not pin the oracle.
"""
import os

import pytest

import oracle
import oracle_pins

MUTANTS = {
    "no_decay": ("row[j] *= alpha;", "(void)alpha;"),
    "decay_sign": ("double alpha = exp(lambda[c]);", "double alpha = exp(-lambda[c]);"),
    "correction_sign": ("u[j] = beta * (v[j] - w);", "u[j] = beta * (v[j] + w);"),
    "missing_beta": ("u[j] = beta * (v[j] - w);", "u[j] = (v[j] - w);"),
    "transposed_state_read": ("w += S[(size_t)c * dv + j] * kh[c];", "w += S[(size_t)j * dv + c] * kh[c];"),
    "query_uses_key": ("acc += S[(size_t)c * dv + j] * qh[c];", "acc += S[(size_t)c * dv + j] * kh[c];"),
    "no_delta_correction": ("row[j] += kh[c] * u[j];", "row[j] += kh[c] * beta * v[j];"),
    "missing_scale": ("o[j] = scale * acc;", "o[j] = acc;"),
    "bias_outside_product": ("sigmoid(a * (g[c] + dt_bias[c]))", "sigmoid(a * g[c] + dt_bias[c])"),
    "A_log_not_exponentiated": ("double a = exp(A_log);", "double a = A_log;"),
    "norm_not_sqrt": ("double inv = 1.0 / sqrt(ss + eps);", "double inv = 1.0 / (ss + eps);"),
    "sigmoid_sign": ("return 1.0 / (1.0 + exp(-x));", "return 1.0 / (1.0 + exp(x));"),
    "rmsnorm_sum_not_mean": ("ms /= d;", "(void)0;"),
    "rmsnorm_eps_outside_root": ("double inv_rms = 1.0 / sqrt(ms + eps);", "double inv_rms = 1.0 / (sqrt(ms) + eps);"),
    "rmsnorm_no_weight": ("xr[c] * inv_rms * w[c] * sigmoid(", "xr[c] * inv_rms * sigmoid("),
    "rmsnorm_gate_sign": ("sigmoid(bf16_to_double(z[(size_t)r * d + c]))", "sigmoid(-bf16_to_double(z[(size_t)r * d + c]))"),
    "rmsnorm_ungated": ("* w[c] * sigmoid(bf16_to_double(z[(size_t)r * d + c]));", "* w[c];"),
    "rmsnorm_rstd_not_inverse": ("rstd[r] = inv_rms;", "rstd[r] = 1.0 / inv_rms;"),
    "conv_taps_reversed": ("acc += w[(size_t)c * W + j] * win[(size_t)j * d + c];",
                           "acc += w[(size_t)c * W + (W - 2 - j)] * win[(size_t)j * d + c];"),
    "conv_window_not_shifted": ("win[(size_t)j * d + c] = win[(size_t)(j + 1) * d + c];", "(void)0;"),
    "conv_no_silu": ("y[c] = silu ? acc * sigmoid(acc) : acc;", "y[c] = acc;"),
    "conv_silu_as_sigmoid": ("y[c] = silu ? acc * sigmoid(acc) : acc;", "y[c] = silu ? sigmoid(acc) : acc;"),
    "conv_q_k_swapped": ("double *dst[3] = {x, kh, vv};", "double *dst[3] = {kh, x, vv};"),
    "conv_window_not_seeded": ("if (W && J->conv_win0)", "if (W && J->conv_win0 && 0)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mpath = os.path.join(tmp_path, f"{name}.c")
    with open(mpath, "w") as f:
        f.write(src.replace(old, new))
    mut = oracle.Oracle(oracle.build(force=True, src=mpath, out=os.path.join(tmp_path, f"lib{name}.so")))
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mut)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
