"""The pins have teeth: each plants one plausible mistake in a copy of the
oracle source (on the CPU), rebuilds it, and checks that some pin fails.

The planted mistakes include the failure mode the Wan2.2 VSA capture page
describes for its outlier capture: a one-pass softmax without the row-max
shift, which overflows on logits of ~1e3.
"""
import os

import pytest

import oracle
import test_oracle_coarse as tc
import test_oracle_fine as tf
import test_oracle_tile as tt

SRC = os.path.join(os.path.dirname(oracle.__file__), "vsa_oracle.c")

TILE_LOOPS = """                    for (int64_t t = ct * CUBE_T; t < ct * CUBE_T + CUBE_T && t < T; ++t)
                        for (int64_t h = ch * CUBE_H; h < ch * CUBE_H + CUBE_H && h < Hh; ++h)
                            for (int64_t w = cw * CUBE_W; w < cw * CUBE_W + CUBE_W && w < W; ++w) {"""
TILE_LOOPS_SWAPPED = """                    for (int64_t t = ct * CUBE_T; t < ct * CUBE_T + CUBE_T && t < T; ++t)
                        for (int64_t w = cw * CUBE_W; w < cw * CUBE_W + CUBE_W && w < W; ++w)
                            for (int64_t h = ch * CUBE_H; h < ch * CUBE_H + CUBE_H && h < Hh; ++h) {"""

MUTANTS = {
    # name: (list of (old, new, count-of-old-to-replace-or-None-for-all), pins expected to fail)
    "one_pass_softmax": (
        [("const double p = exp(logits[x] - m);", "const double p = exp(logits[x]);", None),
         ("*lse = m + log(l);", "*lse = log(l);", None)],
        [lambda: tf.test_outlier_logits_stay_finite()]),
    "pool_divides_by_64": (
        [("o[d] = cnt > 0 ? s / (double)cnt : 0.0;", "o[d] = cnt > 0 ? s / 64.0 : 0.0;", None)],
        [tc.test_pool_uses_only_real_tokens, tc.test_constant_cubes_closed_form]),
    "pool_sums_padding": (
        [("for (int64_t r = 0; r < cnt; ++r)", "for (int64_t r = 0; r < CUBE_TOKENS; ++r)", None)],
        [tc.test_pool_uses_only_real_tokens]),
    "fine_ignores_vbs": (
        [("s < J->vbs[j]", "s < CUBE_TOKENS", None)],
        [lambda: tf.test_brute_force_masked_matrix(None), tf.test_padded_slots_are_ignored]),
    "logits_use_values": (
        [("const uint16_t* k = J->kt +", "const uint16_t* k = J->vt +", None)],
        [lambda: tf.test_dense_equivalence_divisible(64)]),
    "coarse_sorts_ascending": (
        [("if (x->score > y->score) return -1;\n    if (x->score < y->score) return 1;",
          "if (x->score > y->score) return 1;\n    if (x->score < y->score) return -1;", None)],
        [tc.test_einsum_argsort_restatement, tc.test_constant_cubes_closed_form]),
    "tile_w_before_h": (
        [(TILE_LOOPS, TILE_LOOPS_SWAPPED, 1)],
        [lambda: tt.test_brute_force_enumeration((5, 6, 10)),
         lambda: tt.test_reshape_restatement_on_divisible_grids((4, 8, 12))]),
    "lse_drops_max": (
        [("*lse = m + log(l);", "*lse = log(l);", None)],
        [lambda: tf.test_brute_force_masked_matrix(None)]),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    patches, pins = MUTANTS[name]
    src = open(SRC).read()
    for old, new, count in patches:
        assert old in src, f"patch anchor missing for {name}"
        src = src.replace(old, new) if count is None else src.replace(old, new, count)
    path = tmp_path / "mutant.c"
    path.write_text(src)
    lib_path = oracle.build(force=True, src=str(path), out=str(tmp_path / "libmutant.so"))
    with oracle.using_library(lib_path):
        for pin in pins:
            with pytest.raises(AssertionError):
                pin()
