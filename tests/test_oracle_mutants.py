"""The oracle pins must catch plausible mistakes.

Each case compiles a copy of the oracle's C source with one planted mistake
(a dropped term, a wrong sign or index, a transposed operand, a shifted mask)
and runs the pins of ``test_oracle_pins`` against it; at least one pin must
fail. Mistakes are planted only in a temporary copy of the oracle, on the CPU.
"""
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "sink_oracle.c")

MUTANTS = {
    "sink_dropped_from_denominator": ("z[n] = sinks[h];", "z[n] = -1e300;"),
    "sink_multiplied_by_scale": ("z[n] = sinks[h];", "z[n] = P->scale * sinks[h];"),
    "sink_column_gets_upstream_gradient": ("u[n] = 0.0;", "u[n] = 1.0;"),
    "softmax_jacobian_sign": ("dz[t] = p[t] * (u[t] - c);", "dz[t] = p[t] * (c - u[t]);"),
    "dv_uses_score_gradient": ("dvj[e] += pij * doi[e];", "dvj[e] += dzij * doi[e];"),
    "dk_misses_scale": ("dkj[e] += scale * dzij * qi[e];", "dkj[e] += dzij * qi[e];"),
    "dq_uses_values_not_keys": ("const double* kj = k + ((size_t)(base + j0 + m) * h_kv + hk) * d;",
                                "const double* kj = v + ((size_t)(base + j0 + m) * h_kv + hk) * d;"),
    "key_pass_drops_row_term_c": ("(dot(doi, vj, d) - row_c[ri])", "(dot(doi, vj, d))"),
    "key_pass_skips_diagonal": ("*i0 = P->causal ? j : 0;", "*i0 = P->causal ? j + 1 : 0;"),
    "window_off_by_one": ("i - P->window + 1 > 0) *j0 = i - P->window + 1;",
                          "i - P->window > 0) *j0 = i - P->window;"),
    "causal_excludes_diagonal": ("*j1 = i + 1;", "*j1 = i + (i > 0 ? 0 : 1);"),
    "gqa_wrong_kv_head": ("const int g = P->h_q / P->h_kv, hk = h / g, d = P->d;\n    const int n = j1 - j0;\n    const double* qi",
                          "const int g = P->h_q / P->h_kv, hk = h % P->h_kv, d = P->d;\n    const int n = j1 - j0;\n    const double* qi"),
    "key_pass_window_too_short": ("if (P->causal && P->window > 0 && j + P->window < L) *i1 = j + P->window;",
                                  "if (P->causal && P->window > 0 && j + P->window - 1 < L) *i1 = j + P->window - 1;"),
    "lse_without_max": ("return m + log(sum);", "return log(sum);"),
    "dsink_sign": ("row_sink[(size_t)h * T + t] = dz[n];", "row_sink[(size_t)h * T + t] = -dz[n];"),
    "output_includes_sink_value": ("for (int u = 0; u < j1 - j0; ++u) {",
                                   "for (int u = 0; u <= j1 - j0 && u < L - j0; ++u) {"),
}


def _pin_calls():
    calls = []
    for case in pins.CASES:
        calls.append((pins.test_matches_sdpa_with_sink_as_zero_value_key, case))
    calls.append((pins.test_sink_to_minus_infinity_is_standard_attention, (True, 0)))
    calls.append((pins.test_row_probabilities_sum_to_one_and_row_identity, ()))
    calls.append((pins.test_sink_gradient_is_sum_of_row_terms, ()))
    calls.append((pins.test_central_finite_differences_every_input, ([5, 11], 2, 2, 3)))
    calls.append((pins.test_closed_form_single_key, ()))
    calls.append((pins.test_closed_form_equal_logits, ()))
    calls.append((pins.test_sink_to_plus_infinity, ()))
    calls.append((pins.test_window_one_is_diagonal_sigmoid_and_wide_window_is_causal, ()))
    calls.append((pins.test_gqa_equals_mha_with_repeated_kv, ()))
    calls.append((pins.test_hand_worked_example_fixture, ()))
    calls.append((pins.test_adding_a_constant_to_every_logit_of_a_row_changes_only_the_lse, (7.5,)))
    calls.append((pins.test_decode_window_one_is_a_sigmoid_of_the_newest_key, ()))
    return calls


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_some_pin_catches_planted_mistake(name, tmp_path, monkeypatch):
    old, new = MUTANTS[name]
    with open(SRC, encoding="utf-8") as f:
        src = f.read()
    assert src.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(old, new)
    csrc = tmp_path / "sink_oracle.c"
    csrc.write_text(mutated, encoding="utf-8")
    hdr = os.path.join(os.path.dirname(SRC), "sink_oracle.h")
    (tmp_path / "sink_oracle.h").write_text(open(hdr, encoding="utf-8").read(), encoding="utf-8")
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-o", str(so),
                    str(csrc), "-lm"], check=True)
    monkeypatch.setattr(oracle, "_lib", None)
    monkeypatch.setattr(oracle, "build", lambda force=False: str(so))
    caught = []
    for fn, args in _pin_calls():
        try:
            fn(*args)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(fn.__name__)
    monkeypatch.setattr(oracle, "_lib", None)
    assert caught, f"no pin caught the planted mistake {name}"
