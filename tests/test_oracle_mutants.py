"""The oracle's pins must catch plausible mistakes in the oracle itself.

Each mutant is a copy of the oracle's C source with one planted mistake (a
dropped term, a wrong sign or index, a transposed operand), compiled on the
CPU.  The test swaps it in for the real oracle and runs the pins of
test_oracle_pins.py; at least one pin must fail for every mutant.
"""
import pytest

import oracle
import test_oracle_pins as pins

MUTANTS = {
    "dropped scale": ("s[j] = J->scale * acc;", "s[j] = acc;"),
    "causal off by one": ("if (J->causal && i + 1 < nkept) nkept = i + 1;",
                          "if (J->causal && i + 2 < nkept) nkept = i + 2;"),
    "gqa head modulo": ("const int hk = hq / (J->Hq / J->Hkv);", "const int hk = hq % J->Hkv;"),
    "K transposed": ("acc += qrow[d] * kh[j * D + d];", "acc += qrow[d] * kh[(int64_t)d * J->Nkv + j];"),
    "lse drops max": ("*out_lse = M + log(L);", "*out_lse = log(L);"),
    "lse base 2": ("*out_lse = M + log(L);", "*out_lse = M + log2(L);"),
    "no normalisation": ("const double p = exp(s[j] - M) / L;", "const double p = exp(s[j] - M);"),
    "unshifted normaliser": ("L += exp(s[j] - M);", "L += exp(s[j]);"),
    "no max shift": ("M = s[j] > M ? s[j] : M;", "M = 0.0;"),
    "value row shifted": ("out[d] += p * vh[j * D + d];", "out[d] += p * vh[((j + 1) % J->Nkv) * D + d];"),
    "query ignores head": ("const uint16_t* qbits = J->q + r * D;", "const uint16_t* qbits = J->q + i * D;"),
    "fp16 exponent bias": ("mag = ldexp((double)(1024 + f), e - 25);", "mag = ldexp((double)(1024 + f), e - 24);"),
    "bf16 fraction width": ("mag = ldexp((double)(128 + f), e - 134);", "mag = ldexp((double)(128 + f), e - 133);"),
    "sign of score": ("s[j] = J->scale * acc;", "s[j] = -J->scale * acc;"),
    "merge drops max": ("lse[r] = M + log(L);", "lse[r] = log(L);"),
    "merge unnormalised": ("const double w = exp(lse_parts[(int64_t)s * rows + r] - M) / L;",
                           "const double w = exp(lse_parts[(int64_t)s * rows + r] - M);"),
    "merge weight sign": ("const double w = exp(lse_parts[(int64_t)s * rows + r] - M) / L;",
                          "const double w = exp(M - lse_parts[(int64_t)s * rows + r]) / L;"),
    "merge part index": ("const double* os = o_parts + ((int64_t)s * rows + r) * D;",
                         "const double* os = o_parts + ((int64_t)0 * rows + r) * D;"),
    "merge unshifted normaliser": ("L += exp(lse_parts[(int64_t)s * rows + r] - M);",
                                   "L += exp(lse_parts[(int64_t)s * rows + r]);"),
    "alibi sign": ("s[j - lo] = J->scale * dot - slope * dist;", "s[j - lo] = J->scale * dot + slope * dist;"),
    "variant K transposed": ("dot += qrow[d] * kh[j * D + d];", "dot += qrow[d] * kh[(int64_t)d * n_keys + j];"),
    "variant lse drops max": ("*out_lse = log(L) + M;", "*out_lse = log(L);"),
    "variant query row": ("const uint16_t* qsrc = J->q + r * D;", "const uint16_t* qsrc = J->q + (r % J->Nq) * D;"),
    "alibi distance sign": ("const double dist = (double)(i > j ? i - j : j - i);",
                            "const double dist = (double)(j - i);"),
    "window left off by one": ("if (J->window_left >= 0 && i - J->window_left > lo) lo = i - J->window_left;",
                               "if (J->window_left >= 0 && i - J->window_left + 1 > lo) lo = i - J->window_left + 1;"),
    "window right off by one": ("if (J->window_right >= 0 && i + J->window_right + 1 < hi) hi = i + J->window_right + 1;",
                                "if (J->window_right >= 0 && i + J->window_right < hi) hi = i + J->window_right;"),
    "varlen key offset": ("kh = J->k + ((int64_t)kv_head * J->Nkv + J->cu_k[z]) * D;",
                          "kh = J->k + ((int64_t)kv_head * J->Nkv + J->cu_q[z]) * D;"),
    "variant gqa head modulo": ("const int group = J->Hq / J->Hkv;", "const int group = 1;"),
    "varlen key count": ("n_keys = J->cu_k[z + 1] - J->cu_k[z];", "n_keys = J->cu_q[z + 1] - J->cu_q[z];"),
    "bwd dq scale dropped": ("dqi[d] += J->scale * dsj * kh[j * D + d];", "dqi[d] += dsj * kh[j * D + d];"),
    "bwd softmax jacobian": ("const double dsj = pj * (dp[j] - rowdot);", "const double dsj = pj * dp[j];"),
    "bwd dv uses dp": ("dvh[j * D + d] += pj * gi[d];", "dvh[j * D + d] += dp[j] * gi[d];"),
    "bwd dk uses k": ("dkh[j * D + d] += J->scale * dsj * qi[d];", "dkh[j * D + d] += J->scale * dsj * kh[j * D + d];"),
    "bwd causal dropped": ("if (J->causal && i + 1 < n) n = i + 1;", "if (0 && i + 1 < n) n = i + 1;"),
    "bwd rowdot unweighted": ("rowdot += pj * acc;", "rowdot += acc;"),
    "bwd unshifted normaliser": ("Ls += exp(sc[j] - Mx);", "Ls += exp(sc[j]);"),
    "bwd score scale dropped": ("sc[j] = J->scale * qk;", "sc[j] = qk;"),
    "bwd dp uses q": ("for (int d = 0; d < D; ++d) acc += gi[d] * vh[j * D + d];",
                      "for (int d = 0; d < D; ++d) acc += qi[d] * vh[j * D + d];"),
    "bwd ex alibi sign": ("se[j] = J->scale * dotk - slope * gap;", "se[j] = J->scale * dotk + slope * gap;"),
    "bwd ex window left off by one": ("if (J->window_left >= 0 && i - J->window_left > klo) klo = i - J->window_left;",
                                      "if (J->window_left >= 0 && i - J->window_left + 1 > klo) klo = i - J->window_left + 1;"),
    "bwd ex window right dropped": ("if (J->window_right >= 0 && i + J->window_right + 1 < khi) khi = i + J->window_right + 1;",
                                    "if (0 && i + J->window_right + 1 < khi) khi = i + J->window_right + 1;"),
    "bwd ex causal dropped": ("if (J->causal && i + 1 < khi) khi = i + 1;", "if (0 && i + 1 < khi) khi = i + 1;"),
    "bwd ex softmax jacobian": ("const double dse = pe * (dpe[j] - rsum);", "const double dse = pe * dpe[j];"),
    "bwd ex dk uses k": ("dkb[j * D + d] += J->scale * dse * qr[d];", "dkb[j * D + d] += J->scale * dse * kb[j * D + d];"),
    "bwd ex slope head": ("const double slope = J->alibi ? J->alibi[hq] : 0.0;\n            for (int64_t i = 0; i < J->Nq; ++i) {\n                const double* qr",
                          "const double slope = J->alibi ? J->alibi[hk] : 0.0;\n            for (int64_t i = 0; i < J->Nq; ++i) {\n                const double* qr"),
    "variant causal dropped": ("if (J->causal && i + 1 < hi) hi = i + 1;", "if (0 && i + 1 < hi) hi = i + 1;"),
}

PIN_CALLS = [
    ("decode fp16", lambda: pins.test_decode_every_bit_pattern("fp16")),
    ("decode bf16", lambda: pins.test_decode_every_bit_pattern("bf16")),
    ("single key", lambda: pins.test_single_key_gives_v0("fp16", False)),
    ("identical keys", lambda: pins.test_identical_keys_give_mean_v("bf16")),
    ("causal row 0", lambda: pins.test_causal_row0_is_v0("fp16")),
    ("probabilities", lambda: pins.test_identity_values_expose_probabilities(True)),
    ("mpmath", lambda: pins.test_mpmath_bruteforce("fp16", 0.25, False)),
    ("mpmath large", lambda: pins.test_mpmath_bruteforce("fp16", 200.0, False)),
    ("mpmath causal", lambda: pins.test_mpmath_bruteforce("bf16", 0.25, True)),
    ("scipy", lambda: pins.test_matches_scipy("fp16", True, (2, 4, 2, 37, 53, 32))),
    ("gqa", pins.test_gqa_equals_mha_on_repeated_kv),
    ("prefix", pins.test_causal_row_is_prefix_attention),
    ("merge shards", lambda: pins.test_merge_of_key_shards_is_attention_over_their_union((0, 40, 97))),
    ("merge closed form", pins.test_merge_two_parts_closed_form),
    ("merge equal lse", pins.test_merge_equal_lse_gives_mean_and_log_count),
    ("ex base", lambda: pins.test_ex_with_no_variant_is_the_base_forward(True)),
    ("window", lambda: pins.test_window_is_attention_over_the_window((5, 3), False)),
    ("window causal", lambda: pins.test_window_is_attention_over_the_window((7, 2), True)),
    ("alibi extra dim", lambda: pins.test_alibi_is_an_extra_dimension_where_the_distance_has_one_sign(False)),
    ("alibi weights", pins.test_alibi_weights_decay_geometrically_and_symmetrically),
    ("varlen", lambda: pins.test_varlen_is_attention_per_sequence(True)),
    ("bwd fd", lambda: pins.test_bwd_matches_finite_differences("bf16", True, (2, 4, 2, 9, 6, 4))),
    ("bwd single key", pins.test_bwd_single_key_closed_form),
    ("bwd scale zero", pins.test_bwd_scale_zero_closed_form),
    ("bwd ex fd", lambda: pins.test_bwd_ex_matches_finite_differences("bf16", True, (3, -1), [0.5, 0.125],
                                                                      (1, 2, 2, 8, 10, 4))),
    ("bwd ex fd window", lambda: pins.test_bwd_ex_matches_finite_differences("fp16", False, (-1, 2),
                                                                             [0.25, 1.0, 0.0, 0.75], (2, 4, 2, 7, 6, 8))),
    ("bwd ex diagonal", pins.test_bwd_ex_diagonal_window_closed_form),
]


def test_every_mutation_is_applicable():
    src = open(oracle.SOURCE).read()
    for name, (old, _new) in MUTANTS.items():
        assert src.count(old) == 1, name


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, monkeypatch):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read().replace(old, new)
    lib = oracle.load(src, tag="-mutant")
    monkeypatch.setattr(oracle, "load", lambda *a, **k: lib)
    caught = []
    for pin_name, call in PIN_CALLS:
        try:
            call()
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(pin_name)
    assert caught, f"no pin caught the mutant {name!r}"
