"""Planted mistakes in the C oracle must be caught by the pins.

Each case copies ``oracle/kda_oracle.c``, plants one plausible mistake (a
dropped term, a wrong sign, a wrong index, a swapped operand), builds the
copy with gcc, swaps it in for the oracle and runs the pin checks of
``test_oracle_pins.py``: at least one of them must fail.  CPU only.
"""
from __future__ import annotations

import os
import subprocess

import pytest

import oracle
import tests.test_oracle_pins as pins

MUTATIONS = {
    "dropped_decay": ("for (int c = 0; c < KD; ++c) s[c] *= decay[c];",
                      "for (int c = 0; c < KD; ++c) s[c] *= 1.0;"),
    "dt_bias_sign": ("(double)gt[c] + (double)dt_bias[h * KD + c]",
                     "(double)gt[c] - (double)dt_bias[h * KD + c]"),
    "A_log_not_exponentiated": ("exp((double)A_log[h])", "((double)A_log[h])"),
    "sigmoid_sign": ("return 1.0 / (1.0 + exp(-x));", "return 1.0 / (1.0 + exp(x));"),
    "dropped_beta": ("const double u = beta * ((double)vt[v0 + j] - sk_dot);",
                     "const double u = ((double)vt[v0 + j] - sk_dot);"),
    "output_reads_key": ("o += s[c] * qh[c];", "o += s[c] * kh[c];"),
    "dropped_scale": ("qh[c] = scale * (double)qt[c] * rq;", "qh[c] = (double)qt[c] * rq;"),
    "gva_wrong_head": ("const int hq = h / ratio;", "const int hq = h % Hqk;"),
    "dropped_epsilon": ("1.0 / sqrt(sk + 1e-6)", "1.0 / sqrt(sk)"),
    "update_with_query": ("for (int c = 0; c < KD; ++c) s[c] += kh[c] * u;",
                          "for (int c = 0; c < KD; ++c) s[c] += qh[c] * u;"),
    "transposed_initial_state": ("S[j][c] = h0 ? h0[(((long)n * Hv + h) * KD + v0 + j) * KD + c] : 0.0;",
                                 "S[j][c] = h0 ? h0[(((long)n * Hv + h) * KD + c) * KD + v0 + j] : 0.0;"),
    "no_l2norm_on_query": ("const double rq = use_qk_l2norm ? 1.0 / sqrt(sq + 1e-6) : 1.0;",
                           "const double rq = 1.0;"),
}

PIN_CHECKS = [
    pins.test_gate_golden_values,
    pins.test_beta_zero_gate_zero_leaves_state_and_reads_it,
    pins.test_single_token_from_zero_state,
    pins.test_delta_rule_overwrite,
    lambda: pins.test_bruteforce_tiny(5, -5.0),
    lambda: pins.test_chunk_form_matches_recurrence(65, -0.05, 0.0),
    pins.test_chunk_form_varlen_gva,
    pins.test_corr_matches_windowed_solve,
]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path, monkeypatch):
    old, new = MUTATIONS[name]
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found once"
    path = tmp_path / "mut.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99",
                           str(path), "-o", str(so), "-lm"])
    monkeypatch.setattr(oracle, "_lib", oracle.open_library(str(so)))
    caught = 0
    for check in PIN_CHECKS:
        try:
            check()
        except AssertionError:
            caught += 1
    assert caught > 0, f"no pin caught the planted mistake {name}"


def test_unmutated_oracle_passes_every_check():
    for check in PIN_CHECKS:
        check()
