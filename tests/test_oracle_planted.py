"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (a dropped
term, a wrong sign, an off-by-one tie rule, a swapped operand, a wrong
normalisation...), builds that copy into a library of its own under a
temporary directory, points the oracle at it, and runs the pins chosen to
catch that kind of mistake: at least one of them must fail.  The unchanged
source, built the same way, passes all of them.  Nothing here touches the
oracle on disk, and the GPU is not involved."""
import ctypes  # noqa: F401  (the oracle loads the library through ctypes)
import os
import subprocess

import pytest

import oracle
import seeded_inputs as si
import test_oracle_backward as tb
import test_oracle_fp8 as tf
import test_oracle_pins as tp

SRC = os.path.join(os.path.dirname(oracle.__file__), "moe_oracle.c")


def _build(tmp_path, name, old, new, count=1):
    src = open(SRC, encoding="utf-8").read()
    if old is not None:
        assert src.count(old) >= 1, f"planted mistake {name}: text not found"
        src = src.replace(old, new, count)
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"lib_{name}.so"
    c.write_text(src, encoding="utf-8")
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", str(so), str(c), "-lm"])
    return str(so)


def _use(monkeypatch, so):
    monkeypatch.setattr(oracle, "_SO", so)
    monkeypatch.setattr(oracle, "build", lambda force=False: so)
    monkeypatch.setattr(oracle, "_lib", None)


def _failures(checks):
    failed = []
    for name, fn in checks:
        try:
            fn()
        except AssertionError:
            failed.append(name)
    return failed


def _c(label, fn, *args):
    return (label, lambda: fn(*args))


# (name, text in the oracle source, the planted text, pins that must catch it)
PLANTED = [
    ("router_bias_dropped",
     "for (int e = 0; e < E; ++e) l[e] = bg ? ld(bg, dtype, e) : 0.0;",
     "for (int e = 0; e < E; ++e) l[e] = 0.0;",
     [_c("logits vs matmul", tp.test_router_logits_match_library_matmul, si.F32, True)]),
    ("softmax_wrong_sign",
     "p[e] = exp(l[e] - m);", "p[e] = exp(m - l[e]);",
     [_c("softmax vs library", tp.test_softmax_probs_sum_to_one_and_match_library)]),
    ("sigmoid_wrong_sign",
     "p[e] = 1.0 / (1.0 + exp(-l[e])); z += p[e];", "p[e] = 1.0 / (1.0 + exp(l[e])); z += p[e];",
     [_c("normalised sigmoid", tp.test_normalised_sigmoid_gating)]),
    ("topk_ties_to_higher_index",
     "while (j >= 0 && v[order[j]] < v[key])", "while (j >= 0 && v[order[j]] <= v[key])",
     [_c("ties", tp.test_topk_ties_go_to_lower_index), _c("brute force", tp.test_topk_brute_force, 8)]),
    ("renormalised_over_all_experts",
     "for (int j = 0; j < k; ++j) z += p[idx[t * k + j]];", "for (int e2 = 0; e2 < E; ++e2) z += p[e2];",
     [_c("worked example", tp.test_worked_example_topk), _c("k=1", tp.test_k1_weight_is_exactly_one)]),
    ("capacity_floor",
     "return (int64_t)ceil((double)T * cf / (double)E);", "return (int64_t)floor((double)T * cf / (double)E);",
     [_c("formula", tp.test_capacity_formula), _c("hand cases", tp.test_capacity_hand_cases)]),
    ("capacity_one_too_many",
     "if (C < 0 || counts[e] < C) {", "if (C < 0 || counts[e] <= C) {",
     [_c("hand cases", tp.test_capacity_hand_cases), _c("invariants", tp.test_dispatch_invariants, 1.0)]),
    ("gelu_tanh_form",
     "if (act == OACT_GELU) return 0.5 * z * (1.0 + erf(z / sqrt(2.0)));",
     "if (act == OACT_GELU) return 0.5 * z * (1.0 + tanh(sqrt(2.0 / acos(-1.0)) * (z + 0.044715 * z * z * z)));",
     [_c("activation values", tp.test_activation_values)]),
    ("swiglu_operands_swapped",
     "h[j] = (act == OACT_SWIGLU) ? oracle_act(OACT_SWIGLU, h[j]) * u[j] : oracle_act(act, h[j]);",
     "h[j] = (act == OACT_SWIGLU) ? oracle_act(OACT_SWIGLU, u[j]) * h[j] : oracle_act(act, h[j]);",
     [_c("k=E dense", tp.test_identical_experts_with_k_equal_E_is_the_dense_ffn, si.SWIGLU, si.F32)]),
    ("shared_experts_dropped",
     "    for (int s = 0; s < S; ++s) {\n      oracle_expert_ffn(d, f, act, dtype, E + s, xr, W1, b1, W2, b2, W3, o);",
     "    for (int s = 0; s < 0; ++s) {\n      oracle_expert_ffn(d, f, act, dtype, E + s, xr, W1, b1, W2, b2, W3, o);",
     [_c("dense masked", tp.test_sparse_equals_dense_masked, si.SWIGLU, si.SIGMOID_NORM, 0.0, 2)]),
    ("dropped_assignment_kept",
     "      if (dropped[t * k + j]) continue;\n      oracle_expert_ffn(d, f, act, dtype, idx[t * k + j],",
     "      oracle_expert_ffn(d, f, act, dtype, idx[t * k + j],",
     [_c("dense masked", tp.test_sparse_equals_dense_masked, si.GELU, si.SOFTMAX, 1.0, 0)]),
    ("f_divided_by_T",
     "f[e] = T > 0 ? (double)n_pre[e] / ((double)T * (double)k) : 0.0;",
     "f[e] = T > 0 ? (double)n_pre[e] / (double)T : 0.0;",
     [_c("uniform router", tp.test_laux_is_alpha_under_uniform_router, 2, si.SOFTMAX),
      _c("f before the cut", tp.test_f_counts_selections_before_the_capacity_cut)]),
    ("laux_without_E",
     "*L_aux = alpha * (double)E * L;", "*L_aux = alpha * L;",
     [_c("uniform router", tp.test_laux_is_alpha_under_uniform_router, 1, si.SOFTMAX),
      _c("uniform f", tp.test_laux_is_alpha_when_f_is_uniform)]),
    ("noise_subtracted",
     "logits[i] += (double)noise[i];", "logits[i] -= (double)noise[i];",
     [_c("noise shifts logits", tp.test_zero_noise_changes_nothing_and_noise_shifts_logits_exactly)]),
    ("entropy_in_bits",
     "if (f > 0.0) H -= f * log(f);", "if (f > 0.0) H -= f * log2(f);",
     [_c("health closed forms", tp.test_route_health_closed_forms)]),
    ("ec_ties_to_higher_token",
     "while (j >= 0 && scores[(int64_t)order[j] * E + e] < scores[(int64_t)key * E + e]) {",
     "while (j >= 0 && scores[(int64_t)order[j] * E + e] <= scores[(int64_t)key * E + e]) {",
     [_c("brute force", tp.test_ec_select_brute_force), _c("flat router", tp.test_ec_flat_router_takes_the_first_tokens)]),
    ("ec_capacity_without_k",
     "ceil((double)T * (double)k / (double)E)", "ceil((double)T / (double)E)",
     [_c("capacity", tp.test_ec_capacity)]),
]

PLANTED += [
    ("backward_renormalised_weight_sign",
     "dl[e] += w[t * k + j] * (dw[j] - wdw);", "dl[e] += w[t * k + j] * (wdw - dw[j]);",
     [_c("finite differences", tb.test_backward_gelu_softmax_capacity_bias_noise)]),
    ("backward_gelu_density_term_dropped",
     "return 0.5 * (1.0 + erf(z / sqrt(2.0))) + z * exp(-0.5 * z * z) / sqrt(2.0 * acos(-1.0));",
     "return 0.5 * (1.0 + erf(z / sqrt(2.0)));",
     [_c("finite differences", tb.test_backward_gelu_softmax_capacity_bias_noise)]),
    ("backward_swiglu_up_gradient",
     "du[r] = dh[r] * a[r] * sa;", "du[r] = dh[r] * sa;",
     [_c("finite differences", tb.test_backward_swiglu_sigmoid_shared)]),
    ("ec_backward_gating_mean_dropped",
     "        dl = p[e] * (dp[e] - pdp);", "        dl = p[e] * dp[e];",
     [_c("finite differences", tb.test_ec_backward_gelu_softmax_bias_noise_unchosen_tokens)]),
    ("ec_backward_output_weight_one",
     "dp[e] += expert_row_bwd(d, f, act, dtype, e, p[e], xr, dyt,",
     "dp[e] += expert_row_bwd(d, f, act, dtype, e, 1.0, xr, dyt,",
     [_c("finite differences", tb.test_ec_backward_swiglu_sigmoid_shared)]),
    ("rounding_ties_away_from_zero",
     "return ldexp(rint(ldexp(v, -qe)), qe);", "return ldexp(round(ldexp(v, -qe)), qe);",
     [_c("midpoints", tf.test_midpoints_round_to_even_and_overflow_saturates),
      _c("bf16 vs library", tf.test_bf16_round_matches_library)]),
    ("e4m3_saturates_to_nan",
     "if (a >= 448.0) return sign | 0x7E;                 /* saturate */",
     "if (a >= 448.0) return sign | 0x7F;                 /* saturate */",
     [_c("saturation", tf.test_midpoints_round_to_even_and_overflow_saturates)]),
    ("e4m3_subnormal_quantum",
     "a = round_bits(a, 4, -9);", "a = round_bits(a, 4, -10);",
     [_c("encode vs library", tf.test_encode_matches_library_in_range),
      _c("encode of every value", tf.test_encode_of_every_value_is_its_code)]),
    ("row_scale_inverted",
     "const float ss = a / 448.0f;", "const float ss = 448.0f / a;",
     [_c("hand row", tf.test_quantize_rows_hand_case), _c("row properties", tf.test_quantize_rows_properties)]),
    ("fp8_hidden_without_row_scale",
     "double a = (double)xs * (double)s1[(int64_t)g * f + j] * acc;",
     "double a = (double)s1[(int64_t)g * f + j] * acc;",
     [_c("halves vs numpy", tf.test_fp8_expert_halves_against_numpy, si.GELU)]),
    ("fp8_out_without_row_scale",
     "out[c] = (double)hs * (double)s2[(int64_t)g * d + c] * acc;",
     "out[c] = (double)s2[(int64_t)g * d + c] * acc;",
     [_c("halves vs numpy", tf.test_fp8_expert_halves_against_numpy, si.SWIGLU)]),
]


PLANTED += [
    ("ec_output_weight_dropped",
     "const double w = scores[t * E + e];", "const double w = 1.0;",
     [_c("soft mixture", tp.test_ec_every_token_to_every_expert_is_the_dense_soft_mixture, si.GELU)]),
    ("P_divided_by_Tk",
     "P[e] = T > 0 ? s / (double)T : 0.0;", "P[e] = T > 0 ? s / ((double)T * (double)k) : 0.0;",
     [_c("uniform router", tp.test_laux_is_alpha_under_uniform_router, 2, si.SOFTMAX)]),
    ("health_variance_unbiased",
     "  var /= (double)E;", "  var /= (double)(E - 1);",
     [_c("health closed forms", tp.test_route_health_closed_forms)]),
    ("dx_rows_router_term_sign",
     "        dl = w[t * k + j] * (dw[j] - wdw);", "        dl = w[t * k + j] * (wdw - dw[j]);",
     [_c("dx rows vs backward", tb.test_dx_rows_equal_the_backward_pass_without_the_aux_term,
         dict(capacity_factor=0.9))]),
]


@pytest.fixture(scope="module")
def tmp_lib(tmp_path_factory):
    return tmp_path_factory.mktemp("planted")


def test_the_unchanged_source_passes_every_catching_pin(tmp_lib, monkeypatch):
    _use(monkeypatch, _build(tmp_lib, "unchanged", None, None))
    checks = [chk for _, _, _, cs in PLANTED for chk in cs]
    assert _failures(checks) == []


@pytest.mark.parametrize("name,old,new,checks", PLANTED, ids=[p[0] for p in PLANTED])
def test_a_planted_mistake_fails_a_pin(tmp_lib, monkeypatch, name, old, new, checks):
    _use(monkeypatch, _build(tmp_lib, name, old, new))
    assert _failures(checks), f"no pin caught the planted mistake {name}"
