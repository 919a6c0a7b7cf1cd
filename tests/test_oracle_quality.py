"""Pins of the oracle's quality signals ("Optimizing block-sparse INT8
attention and multi-expert step caching for Wan 2.2": Dynamic Sparsity
Budgeting via Softmax Normalizer Registers -- max_prob = 1 / l; Selection
Heuristic Ablation and Recall Analysis -- a selection against dense
attention; glossary -- relative-L1).

Single-key and equal-logit rows fix max_prob in closed form; the captured
mass is checked against dense softmax weights summed explicitly over the
selected keys; rel-L1 against hand values.
"""
import numpy as np

import oracle
from block_sparse_video_vsa_gb300 import synth


def tiny():
    wl = synth.WORKLOADS["tiny"]
    d = synth.make_inputs(wl)
    qt, vbs = oracle.tile(d["q"], wl.grid)
    kt, _ = oracle.tile(d["k"], wl.grid)
    vt, _ = oracle.tile(d["v"], wl.grid)
    return wl, qt, kt, vt, vbs


def test_single_key_is_fully_peaked():
    wl, qt, kt, vt, vbs = tiny()
    N = len(vbs)
    one = int(np.argmin(vbs))  # a partial cube; keep one of its slots only
    vbs1 = vbs.copy()
    vbs1[one] = 1
    idx = np.full((1, wl.heads, N, 1), one, np.int32)
    mp, lse = oracle.row_peak(qt, kt, idx, vbs1, wl.sm_scale, np.arange(wl.heads * N))
    assert np.array_equal(mp, np.ones_like(mp))


def test_equal_logits_spread_evenly():
    rng = np.random.default_rng(0)
    N, heads, D = 4, 1, 8
    vbs = np.array([64, 10, 64, 3], np.int32)
    q = synth.bf16_bits(rng.standard_normal((1, 64 * N, heads, D)).astype(np.float32))
    k = synth.bf16_bits(np.zeros((1, 64 * N, heads, D), np.float32))  # every logit 0
    idx = np.array([[[[1, 3], [0, 2], [1, 2], [3, 0]]]], np.int32)
    mp, lse = oracle.row_peak(q, k, idx, vbs, 0.5, np.arange(N))
    for i in range(N):
        count = sum(vbs[j] for j in idx[0, 0, i])
        assert np.allclose(mp[i], 1.0 / count, rtol=0, atol=1e-15)
        assert np.allclose(lse[i], np.log(count), rtol=0, atol=1e-12)


def test_row_peak_lse_agrees_with_the_fine_stage():
    wl, qt, kt, vt, vbs = tiny()
    idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
    units = np.arange(wl.heads * len(vbs))
    _, lse = oracle.row_peak(qt, kt, idx, vbs, wl.sm_scale, units)
    _, fine_lse, _ = oracle.fine(qt, kt, vt, idx, vbs, wl.sm_scale, units)
    assert np.abs(lse - fine_lse).max() < 1e-12


def test_captured_mass_is_the_dense_weight_of_the_selection():
    wl, qt, kt, vt, vbs = tiny()
    N = len(vbs)
    idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
    dense = np.tile(np.arange(N, dtype=np.int32), (1, wl.heads, N, 1))
    units = np.arange(wl.heads * N)
    _, lse_s, _ = oracle.fine(qt, kt, vt, idx, vbs, wl.sm_scale, units)
    _, lse_d, _ = oracle.fine(qt, kt, vt, dense, vbs, wl.sm_scale, units)
    got = oracle.captured_mass(lse_s, lse_d)
    q, k = synth.bf16_to_f32(qt).astype(np.float64), synth.bf16_to_f32(kt).astype(np.float64)
    real = np.concatenate([np.arange(64 * j, 64 * j + vbs[j]) for j in range(N)])
    for u in (0, 5, N + 3):
        h, i = u // N, u % N
        logits = wl.sm_scale * q[0, 64 * i: 64 * i + 64, h] @ k[0, real, h].T
        w = np.exp(logits - logits.max(axis=1, keepdims=True))
        w /= w.sum(axis=1, keepdims=True)
        sel = np.isin(real // 64, idx[0, h, i])
        assert np.abs(got[u] - w[:, sel].sum(axis=1)).max() < 1e-12
    assert np.abs(oracle.captured_mass(lse_d, lse_d) - 1.0).max() < 1e-15
    assert oracle.captured_mass(np.array([-np.inf]), np.array([2.0]))[0] == 0.0


def test_rel_l1_by_hand():
    ref = np.array([1.0, -2.0, 3.0, -4.0])
    assert oracle.rel_l1(ref, ref) == 0.0
    assert abs(oracle.rel_l1(ref + np.array([0.5, 0.5, -0.5, 0.5]), ref) - 0.5 / 2.5) < 1e-15
