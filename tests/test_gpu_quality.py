"""GPU quality signals against the oracle ("Optimizing block-sparse INT8
attention and multi-expert step caching for Wan 2.2": Dynamic Sparsity
Budgeting via Softmax Normalizer Registers -- max_prob; Selection Heuristic
Ablation and Recall Analysis -- the share of dense attention mass a selection
captures; the glossary's relative-L1 of sparse against dense output).

max_prob comes from vsa_sparse_attn_fwd_peak (the exact row max beside the
fine kernel's lazy softmax offset).  The dense reference is the same fine
stage with every cube selected (topk = N), compared itself with the oracle.
Tolerances: max_prob and the captured mass inherit the LSE bound
|d lse| <= 1e-3 max(1, |lse|) (a relative error of that size in
exp(m - lse)); rel-L1 within 2% of the oracle's value, the bf16 rounding of
both outputs being far below the sparse-dense difference it measures.
"""
import numpy as np
import pytest
import torch

import block_sparse_video_vsa_gb300 as vsa
import oracle
from block_sparse_video_vsa_gb300 import synth
from gpu_util import (LSE_REL, assert_lse_close, assert_scoring_rule, i32_dev, score_outputs, tiled_inputs,
                      to_bits, to_dev)

pytestmark = pytest.mark.gpu


def peak_run(qt, kt, vt, idx, vbs, sm, paired=False):
    idx_d = i32_dev(idx)
    pairs = vsa.pair_cubes(idx_d) if paired else None
    o, lse, mp = vsa.sparse_attn_fwd_peak(to_dev(qt), to_dev(kt), to_dev(vt), idx_d, i32_dev(vbs), sm, pairs=pairs)
    torch.cuda.synchronize()
    assert vsa.device_error(reset=True) == 0
    return to_bits(o), lse.cpu().numpy(), mp.cpu().numpy()


def unit_rows(units, N, heads):
    b, h, i = units // (heads * N), (units // N) % heads, units % N
    return b, h, 64 * i[:, None] + np.arange(64)[None, :]


def assert_peak_close(got, ref, ref_lse):
    bound = LSE_REL * np.maximum(1.0, np.abs(np.where(np.isfinite(ref_lse), ref_lse, 0.0)))
    assert (np.abs(got - ref) <= 1.01 * bound * ref + 1e-7).all(), np.abs(got - ref).max()


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_max_prob_matches_the_oracle(name):
    wl = synth.WORKLOADS[name]
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
    got, lse, mp = peak_run(qt, kt, vt, idx, vbs, wl.sm_scale)
    units = np.arange(wl.B * wl.heads * wl.ncubes)
    ref_mp, ref_lse = oracle.row_peak(qt, kt, idx, vbs, wl.sm_scale, units)
    b, h, rows = unit_rows(units, wl.ncubes, wl.heads)
    assert_peak_close(mp[b[:, None], h[:, None], rows], ref_mp, ref_lse)
    # the peak entry point leaves the output and lse those of the plain call
    o2, l2 = vsa.sparse_attn_fwd(to_dev(qt), to_dev(kt), to_dev(vt), i32_dev(idx), i32_dev(vbs), wl.sm_scale)
    assert np.array_equal(to_bits(o2), got) and np.array_equal(l2.cpu().numpy(), lse)


def test_max_prob_outlier_and_empty_rows():
    """Logits ~1e3 (the exact max then sits far above the lazy offset's
    updates) stay finite and close; rows with no key get 0."""
    wl = synth.Workload("outlier_small", 1, 9, 16, 16, heads=3, D=128, topk=12, seed=77, outlier=True)
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
    _, _, mp = peak_run(qt, kt, vt, idx, vbs, wl.sm_scale, paired=True)
    units = np.arange(wl.heads * wl.ncubes)
    ref_mp, ref_lse = oracle.row_peak(qt, kt, idx, vbs, wl.sm_scale, units)
    b, h, rows = unit_rows(units, wl.ncubes, wl.heads)
    assert np.isfinite(mp).all() and (mp <= 1.0).all()
    assert_peak_close(mp[b[:, None], h[:, None], rows], ref_mp, ref_lse)
    vb0 = np.zeros_like(vbs)
    _, _, mp0 = peak_run(qt, kt, vt, idx, vb0, wl.sm_scale)
    assert (mp0 == 0).all()


def test_dense_reference_mass_and_rel_l1_mid():
    """mid (48 cubes): the dense run against the oracle's dense attention, then
    the captured mass of every row and rel-L1 of sparse against dense."""
    wl = synth.WORKLOADS["mid"]
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
    dense = np.broadcast_to(np.arange(wl.ncubes, dtype=np.int32), (1, wl.heads, wl.ncubes, wl.ncubes)).copy()
    so, slse, _ = peak_run(qt, kt, vt, idx, vbs, wl.sm_scale)
    do, dlse, _ = peak_run(qt, kt, vt, dense, vbs, wl.sm_scale)
    ref_s, ref_slse = oracle.fine_full(qt, kt, vt, idx, vbs, wl.sm_scale)
    ref_d, ref_dlse = oracle.fine_full(qt, kt, vt, dense, vbs, wl.sm_scale)
    assert_scoring_rule(score_outputs(do, ref_d))
    assert_lse_close(dlse, ref_dlse)
    got_cm = np.exp(slse.astype(np.float64) - dlse)
    ref_cm = oracle.captured_mass(ref_slse, ref_dlse)
    bound = 2 * LSE_REL * np.maximum(1.0, np.abs(ref_dlse))
    assert (np.abs(got_cm - ref_cm) <= bound * ref_cm + 1e-7).all()
    assert ((ref_cm > 0) & (ref_cm <= 1 + 1e-12)).all()
    got_rel = oracle.rel_l1(synth.bf16_to_f32(so), synth.bf16_to_f32(do))
    ref_rel = oracle.rel_l1(ref_s, ref_d)
    assert abs(got_rel - ref_rel) <= 0.02 * ref_rel


def test_dense_reference_wan_sampled():
    """The Wan2.2 shape with every one of the 624 cubes selected (the dense
    attention, 624 cubes per row): lse, captured mass and max_prob of sampled
    query cubes against the oracle."""
    wl = synth.WORKLOADS["wan"]
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
    N = wl.ncubes
    dense = np.broadcast_to(np.arange(N, dtype=np.int32), (1, wl.heads, N, N)).copy()
    _, slse, smp = peak_run(qt, kt, vt, idx, vbs, wl.sm_scale, paired=True)
    do, dlse, _ = peak_run(qt, kt, vt, dense, vbs, wl.sm_scale)
    assert np.isfinite(synth.bf16_to_f32(do)).all()
    rng = np.random.default_rng(9)
    units = np.unique(np.concatenate([rng.integers(0, wl.heads * N, 40), [0, N - 1]]))
    ref_smp, ref_slse = oracle.row_peak(qt, kt, idx, vbs, wl.sm_scale, units)
    _, ref_dlse = oracle.row_peak(qt, kt, dense, vbs, wl.sm_scale, units)
    b, h, rows = unit_rows(units, N, wl.heads)
    assert_lse_close(dlse[b[:, None], h[:, None], rows], ref_dlse)
    assert_peak_close(smp[b[:, None], h[:, None], rows], ref_smp, ref_slse)
    got_cm = np.exp(slse[b[:, None], h[:, None], rows].astype(np.float64) - dlse[b[:, None], h[:, None], rows])
    ref_cm = oracle.captured_mass(ref_slse, ref_dlse)
    bound = 2 * LSE_REL * np.maximum(1.0, np.abs(ref_dlse))
    assert (np.abs(got_cm - ref_cm) <= bound * ref_cm + 1e-7).all()
