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


# ---- the Python-level oracle functions (numpy): a planted mistake in a copy
# of the module source, the mutated function patched in, its pins must fail.
import test_oracle_block_select as tb  # noqa: E402
import test_oracle_coarse_attn as tca  # noqa: E402
import test_oracle_quality as tq  # noqa: E402

PY_SRC = os.path.join(os.path.dirname(oracle.__file__), "__init__.py")

PY_MUTANTS = {
    # name: (function, (old, new), pins expected to fail)
    "coarse_attn_values_from_keys": (
        "coarse_attn", ("qm, km, vm = pool(qt, vbs), pool(kt, vbs), pool(vt, vbs)",
                        "qm, km, vm = pool(qt, vbs), pool(kt, vbs), pool(kt, vbs)"),
        [lambda: tca.test_equals_dense_sdpa_on_pooled_cubes("tiny"), tca.test_equal_keys_give_the_plain_mean_of_values]),
    "coarse_attn_unscaled": (
        "coarse_attn", ("s = sm_scale * np.matmul(", "s = 1.0 * np.matmul("),
        [lambda: tca.test_equals_dense_sdpa_on_pooled_cubes("mid")]),
    "coarse_attn_keeps_empty_keys": (
        "coarse_attn", ("live = vbs > 0", "live = vbs >= 0"),
        [tca.test_empty_cubes_are_no_keys_and_give_zero_rows]),
    "gated_swaps_gates": (
        "gated_combine", ("return _bf16_to_f64(gate_c) * per_slot + _bf16_to_f64(gate_f) * fine_out",
                          "return _bf16_to_f64(gate_f) * per_slot + _bf16_to_f64(gate_c) * fine_out"),
        [tca.test_gates_select_one_stage, tca.test_gated_sum_by_hand]),
    "gated_broadcast_by_token_not_cube": (
        "gated_combine", ("np.repeat(np.asarray(coarse_out, np.float64).transpose(0, 2, 1, 3), 64, axis=1)",
                          "np.tile(np.asarray(coarse_out, np.float64).transpose(0, 2, 1, 3), (1, 64, 1, 1))"),
        [tca.test_gates_select_one_stage, tca.test_gated_sum_by_hand]),
    "block_select_one_past_threshold": (
        "block_select_cdf", ("while kept < nb and (kept == 0 or mass < tau):",
                             "while kept < nb and (kept == 0 or mass - w[order[kept - 1]] < tau):"),
        [lambda: tb.test_brute_force_smallest_subset(7, 0.9, 8.0), tb.test_threshold_limits]),
    "block_select_ascending": (
        "block_select_cdf", ("order = sorted(range(nb), key=lambda j: (-s[j], j))",
                             "order = sorted(range(nb), key=lambda j: (s[j], j))"),
        [tb.test_threshold_limits, lambda: tb.test_brute_force_smallest_subset(5, 0.8, 0.5)]),
    "block_select_unscaled_weights": (
        "block_select_cdf", ("w = np.exp(sm_scale * (s - s.max()))", "w = np.exp(s - s.max())"),
        [lambda: tb.test_brute_force_smallest_subset(7, 0.9, 8.0)]),
    "cube_lut_neighbouring_blocks": (
        "blocks_to_cube_lut", ("sub = np.where(idx >= 0, idx * c + r, -1)", "sub = np.where(idx >= 0, idx + r, -1)"),
        [tb.test_block_table_to_cube_table_by_hand, tb.test_block_sparse_attention_is_dense_attention_over_kept_blocks]),
    "max_prob_is_the_normaliser": (
        "row_peak", ("max_prob[n] = 1.0 / l", "max_prob[n] = l"),
        [tq.test_equal_logits_spread_evenly]),
    "max_prob_without_the_row_max": (
        "row_peak", ("l = np.exp(logits - m[:, None]).sum(axis=1)", "l = np.exp(logits).sum(axis=1)"),
        [tq.test_row_peak_lse_agrees_with_the_fine_stage]),
    "captured_mass_inverted": (
        "captured_mass", ("np.exp(a - b)", "np.exp(b - a)"),
        [tq.test_captured_mass_is_the_dense_weight_of_the_selection]),
    "fine_counts_ignores_counts": (
        "fine_counts", ("idx2[:, :, :N] = np.where(np.arange(k)[None, None, None, :] < c[..., None], topk_idx, N)",
                        "idx2[:, :, :N] = topk_idx"),
        [lambda: tf.test_counts_brute_force(0), tf.test_count_zero_rows_are_empty]),
}


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_planted_python_mistake_is_caught(name, monkeypatch):
    func, (old, new), pins = PY_MUTANTS[name]
    src = open(PY_SRC).read()
    assert src.count(old) == 1, f"patch anchor missing for {name}"
    ns = {"__name__": "oracle_mutant", "__file__": PY_SRC}
    exec(compile(src.replace(old, new), PY_SRC, "exec"), ns)
    monkeypatch.setattr(oracle, func, ns[func])
    for pin in pins:
        with pytest.raises(AssertionError):
            pin()
