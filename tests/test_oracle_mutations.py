"""The pins catch plausible mistakes: each case plants one slip in a copy of
the oracle's C source (on the CPU), builds it, and checks that at least one
pin of tests/test_oracle_pins.py fails against the planted copy."""
import ctypes as C
import os
import subprocess

import pytest

import oracle as O
import test_oracle_pins as P

SRC = os.path.join(os.path.dirname(O.__file__), "mhc_oracle.c")

MUTATIONS = {
    "comb_transposed": ("(double)comb[i * 4 + j]", "(double)comb[j * 4 + i]"),
    "post_term_dropped": ("if (Y) v += (double)post_prev", "if (0) v += (double)post_prev"),
    "rstd_mean_over_H": ("sqrt(sR / (double)K + eps)", "sqrt(sR / (double)H + eps)"),
    "post_gate_not_doubled": ("2.0 * mhc_oracle_sigmoid(l[4 + i])", "mhc_oracle_sigmoid(l[4 + i])"),
    "alpha_groups_shifted": ("int g = k < 4 ? 0 : (k < 8 ? 1 : 2);", "int g = k < 8 ? 0 : 1;"),
    "unrounded_rprime": ("rp[i * H + h] = rprime_unrounded ? v : mhc_oracle_bf16_to_double(b);",
                         "rp[i * H + h] = v;"),
    "gamma_dropped": ("x[h] * rstdx * mhc_oracle_bf16_to_double(gamma[h])", "x[h] * rstdx"),
    "fn_index_transposed": ("(double)fn[(size_t)r * N_LOG + k]", "(double)fn[(size_t)k * K + r]"),
    "sinkhorn_columns_first": ("for (int it = 0; it < iters; ++it) {\n        for (int i = 0; i < n; ++i) {",
                               "for (int it = 0; it < iters; ++it) {\n        for (int i = 0; i < 0; ++i) {"),
    "bf16_truncates": ("double r = rint(a / spacing) * spacing;\n    if (r >= ldexp(1.0, 128))",
                       "double r = floor(a / spacing) * spacing;\n    if (r >= ldexp(1.0, 128))"),
    "e4m3_one_bit_short": ("spacing = ldexp(1.0, (e - 1) - 3);", "spacing = ldexp(1.0, (e - 1) - 2);"),
    "e8m0_bias_off_by_one": ("scales[r * G + g] = (uint8_t)(e + 127);", "scales[r * G + g] = (uint8_t)(e + 128);"),
    "x_uses_equal_weights": ("v += (double)pre[i] * rp[i * H + h];", "v += 0.25 * rp[i * H + h];"),
    "grid_scale_off_by_one": ("mhc_oracle_bf16_rne(ldexp(mhc_oracle_e4m3_decode(code), e))",
                              "mhc_oracle_bf16_rne(ldexp(mhc_oracle_e4m3_decode(code), e + 1))"),
    "e4m3_decode_bias_8": ("ldexp(1.0 + f / 8.0, E - 7)", "ldexp(1.0 + f / 8.0, E - 8)"),
    "identity_form_stream_shifted": ("const uint16_t b = Rt[i * H + h];", "const uint16_t b = Rt[((i + 1) % N_HC) * H + h];"),
    "unshifted_pre_index_shifted": ("v += pre_out[t * 4 + i] * mhc_oracle_bf16_to_double(residual_out[t * K + i * H + h]);",
                                    "v += pre_out[t * 4 + (i + 1) % N_HC] * mhc_oracle_bf16_to_double(residual_out[t * K + i * H + h]);"),
    "sigmoid_sign_flipped": ("return 1.0 / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(z));"),
    "eps_outside_rstd_sqrt": ("double rstdR = 1.0 / sqrt(sR / (double)K + eps);",
                              "double rstdR = 1.0 / (sqrt(sR / (double)K) + eps);"),
    "norm_uses_gate_rstd": ("mhc_oracle_bf16_rne(x[h] * rstdx * mhc_oracle_bf16_to_double(gamma[h]))",
                            "mhc_oracle_bf16_rne(x[h] * rstdR * mhc_oracle_bf16_to_double(gamma[h]))"),
    "post_gate_of_stream0_everywhere": ("if (Y) v += (double)post_prev[t * 4 + i] *", "if (Y) v += (double)post_prev[t * 4] *"),
    "bias_dropped_from_logits": ("l[k] = (double)alpha[g] * rstdR * d[k] + (double)bias[k];",
                                 "l[k] = (double)alpha[g] * rstdR * d[k];"),
    "comb_logits_shifted": ("for (int q = 0; q < 16; ++q) M[q] = exp(l[8 + q]);",
                            "for (int q = 0; q < 16; ++q) M[q] = exp(l[8 + (q + 1) % 16]);"),
    "sum_of_squares_halved": ("sR += rp[r] * rp[r];", "sR += 0.5 * rp[r] * rp[r];"),
    "e4m3_ties_away_from_zero": ("double r = rint(a / spacing) * spacing;   /* r <= 448: 448 is on the grid */",
                                 "double r = round(a / spacing) * spacing;   /* r <= 448: 448 is on the grid */"),
    "e4m3_subnormal_spacing": ("        spacing = ldexp(1.0, -9);\n    } else {", "        spacing = ldexp(1.0, -8);\n    } else {"),
    "amax_signed_not_abs": ("                double a = fabs(mhc_oracle_bf16_to_double(src[j]));\n                if (a > amax) amax = a;\n            }\n            int e = mhc_oracle_ue8m0_exponent(amax, amax_floor);\n            scales",
                            "                double a = mhc_oracle_bf16_to_double(src[j]);\n                if (a > amax) amax = a;\n            }\n            int e = mhc_oracle_ue8m0_exponent(amax, amax_floor);\n            scales"),
    "codes_scaled_up_not_down": ("codes[r * H + g * 32 + j] =\n                    mhc_oracle_e4m3_rne_satfinite(ldexp(mhc_oracle_bf16_to_double(src[j]), -e));",
                                 "codes[r * H + g * 32 + j] =\n                    mhc_oracle_e4m3_rne_satfinite(ldexp(mhc_oracle_bf16_to_double(src[j]), e));"),
    "x_pre_index_shifted": ("v += (double)pre[i] * rp[i * H + h];", "v += (double)pre[(i + 1) % N_HC] * rp[i * H + h];"),
    "unshifted_x_scaled": ("x_out[t * H + h] = mhc_oracle_bf16_rne(v);", "x_out[t * H + h] = mhc_oracle_bf16_rne(v * 1.0009765625);"),
}

PINS = [
    lambda o: P.test_stream_permutation_equivariance(o, (1, 2, 3, 0)),
    P.test_unshifted_zero_fn_gives_half_sum_of_streams,
    lambda o: P.test_brute_force_T1_H8_unshifted(o, 37, True, False),
    P.test_identity_form_keeps_signed_zeros_and_subnormals,
    P.test_e4m3_decode_matches_format_definition,
    P.test_grid_exact_on_the_e4m3_lattice,
    P.test_grid_is_the_dequantised_mxfp8_output,
    P.test_bf16_rne_matches_torch_cast_on_float32_inputs,
    P.test_e4m3_golden_codes_from_ocp_spec,
    P.test_ue8m0_exponent_exhaustive_over_bf16_amax,
    P.test_crafted_groups_448_times_power_of_two,
    P.test_sinkhorn_one_round_is_row_then_column,
    P.test_permutation_comb_permutes_streams,
    P.test_post_term_adds_post_times_Y,
    P.test_collapse_uses_carried_pre,
    P.test_zero_fn_gives_bias_gates,
    P.test_one_hot_fn_picks_stream_signs,
    P.test_constant_row_norm_closed_form,
]


def _build_mutant(tmp_path, name):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"lib_{name}.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", str(so), str(path), "-lm"])
    return O.bind(C.CDLL(str(so)))


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_slip_fails_a_pin(tmp_path, monkeypatch, name):
    mutant = _build_mutant(tmp_path, name)
    monkeypatch.setattr(O, "_lib", mutant)
    failed = []
    for pin in PINS:
        try:
            pin(O)
        except AssertionError:
            failed.append(pin.__name__)
    extra = []
    # the slowest pins (the brute force, the exhaustive e4m3 sweep with its
    # exact ties) run only if the quick ones missed the slip
    for slow in (lambda: P.test_brute_force_T1_H8_asymmetric_comb(O, 31),
                 lambda: P.test_e4m3_exhaustive_over_significands_and_exponents(O)):
        if failed or extra:
            break
        try:
            slow()
        except AssertionError:
            extra.append("slow pin")
    assert failed or extra, f"no pin caught {name}"
