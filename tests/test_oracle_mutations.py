"""The oracle's pins have teeth: each plausible mistake planted in a copy of
csa_oracle.c (a wrong window token, column or APE row, a wrong segment base, a
dropped term, a flipped gradient sign, gradient from padding rows, a wrong exp
constant, a wrong rounding rule) makes at least one pin fail.

Every mutation keeps all memory accesses in bounds, so a mutant can only give
wrong numbers, never crash the test process.
"""
import os

import pytest

import oracle
import test_oracle_bruteforce as B
import test_oracle_exp as E
import test_oracle_grouped as G
import test_oracle_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "csa_oracle.c")

MUTATIONS = {
    "second_half_reads_first_half_column": ("        sl.col = head_dim + j;", "        sl.col = j;"),
    "previous_block_reads_own_block": ("        sl.token = ri->base - ratio + k;", "        sl.token = ri->base + k;"),
    "second_half_ape_rows_reversed": ("        sl.ape_row = k - ratio;", "        sl.ape_row = 2 * ratio - 1 - k;"),
    "segment_base_ignores_tails": ("            ri.base = (int64_t)cu_seqlens[s] + b * ratio;",
                                   "            ri.base = (int64_t)cu_comp[s] * ratio + b * ratio;"),
    "denominator_drops_terms": ("        den = den + ek;", "        den = ek;"),
    "grad_score_sign_flipped": ("                float ds = p * (g * v - go);",
                                "                float ds = p * (go - g * v);"),
    "grouped_grad_ape_sign_flipped": ("                float ds_k = p * (g * v - go);",
                                      "                float ds_k = p * (go - g * v);"),
    "grouped_grad_ape_skips_first_blocks": ("        const int32_t leaf = leaf_of_row[r];",
                                            "        const int32_t leaf = leaf_of_row[r];\n        if (ri.first)\n            continue;"),
    "fp64_grad_score_sign_flipped": ("                double ds = p[k] * g * (v - o);",
                                     "                double ds = p[k] * g * (o - v);"),
    "padding_rows_carry_gradient": ("            continue; /* padding rows: incoming gradient ignored */",
                                    "            ; /* mutated */"),
    "exp_drops_ln2_low_part": ("    r = fmaf(nf, -CSA_LN2_LO, r);", "    r = fmaf(nf, 0.0f, r);"),
    "exp_wrong_polynomial_coefficient": ("(float)(1.0 / 720.0)", "(float)(1.0 / 700.0)"),
    "exp_economization_dropped": ("(float)(1.0 / 120.0 + (1.0 / 5040.0) * (112.0 / 64.0) * CSA_H2)",
                                  "(float)(1.0 / 120.0)"),
    "bf16_rounds_ties_away": ("    u += 0x7fffu + ((u >> 16) & 1u);", "    u += 0x8000u;"),
}


def pins():
    out = []
    for ex in P.golden_examples():
        out.append(("golden_fwd_" + ex["name"], lambda ex=ex: P.test_hand_worked_forward(ex)))
        if "grad_kv" in ex or "grad_kv_at" in ex:
            out.append(("golden_bwd_" + ex["name"], lambda ex=ex: P.test_hand_worked_backward(ex)))
    out += [
        ("rounding", P.test_output_rounding_is_nearest_even),
        ("constant1", lambda: P.test_constant_kv_windows_return_the_constant(1)),
        ("constant2", lambda: P.test_constant_kv_windows_return_the_constant(2)),
        ("ones", P.test_softmax_weights_sum_to_one),
        ("uniform1", lambda: P.test_uniform_logits_give_block_means(1)),
        ("uniform2", lambda: P.test_uniform_logits_give_block_means(2)),
        ("identity", P.test_ratio_one_own_block_is_identity),
        ("first_block", P.test_first_block_equals_own_block_form_on_second_half),
        ("padding", P.test_padding_rows_are_first_blocks_from_token_zero_and_carry_no_gradient),
        ("exp_sweep", E.test_exp_accuracy_dense_sweep),
        ("exp_ln2", E.test_exp_accuracy_near_zero_and_at_integers_of_ln2),
        ("fd1", lambda: P.test_backward_matches_central_finite_differences(1)),
        ("fd2", lambda: P.test_backward_matches_central_finite_differences(2)),
        ("bruteforce_r3c2", lambda: B.test_window_map_bruteforce(3, 2)),
        ("grouped_rows", lambda: G.test_one_row_leaves_are_the_rows_ds(*G.CASES[0])),
        ("grouped_single", G.test_single_leaf_is_the_plain_sum),
    ]
    return out


def failing_pins():
    failed = []
    for name, fn in pins():
        try:
            fn()
        except AssertionError:
            failed.append(name)
    return failed


def test_pins_pass_on_the_real_oracle():
    assert failing_pins() == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation anchor not unique: " + name
    mutant_src = tmp_path / "mutant.c"
    mutant_src.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(mutant_src), str(tmp_path / "libmutant.so"))
    with oracle.using_library(lib):
        for pname, fn in pins():
            try:
                fn()
            except AssertionError:
                return  # caught
    pytest.fail("no pin caught the planted mistake " + name)
