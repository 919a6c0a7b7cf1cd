"""Pins of the oracle's fine stage (block-sparse attention over selected cubes).

Follows "Wan2.2 Production Values -- VSA Block-Sparse Attention Inputs +
Reference" (Operator contract) and the SDPA formula of "VSA: Accelerating
Video Diffusion Inference with Sparse Attention on AMD GPUs" (The Attention
Bottleneck).  Pins:
- topk = all cubes on a divisible grid is dense SDPA (torch's fp64 CPU routine);
- topk = all cubes with padding is dense SDPA over the unpadded tokens;
- an explicit S_pad x S_pad masked-softmax brute force (outputs and LSE);
- closed forms: constant v gives v; zero query rows give the mean of the
  attended values and lse = log(count); a single attended key gives its value;
- invariance to the order of each index row and to padded-slot contents;
- outlier logits (~1e3) stay finite.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_video_vsa_gb300 import synth


def f64(bits):
    return synth.bf16_to_f32(bits).astype(np.float64)


def rand_bits(rng, shape, scale=1.0):
    return synth.bf16_bits(scale * rng.standard_normal(shape, dtype=np.float32))


def sdpa_ref(q, k, v, scale):
    """q, k, v: [B, S, H, D] float64 -> (o [B, S, H, D], lse [B, H, S]) via torch."""
    Q, K, V = (torch.from_numpy(np.ascontiguousarray(a.transpose(0, 2, 1, 3))) for a in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=scale)
    lse = torch.logsumexp(scale * Q @ K.transpose(-1, -2), dim=-1)
    return o.numpy().transpose(0, 2, 1, 3), lse.numpy()


@pytest.mark.parametrize("D", [64, 128])
def test_dense_equivalence_divisible(D):
    rng = np.random.default_rng(0)
    grid = (1, 4, 8, 8)  # 8 cubes, all full
    S = 4 * 8 * 8
    q, k, v = (rand_bits(rng, (1, S, 2, D), 1.5) for _ in range(3))
    qt, vbs = oracle.tile(q, grid)
    kt, _ = oracle.tile(k, grid)
    vt, _ = oracle.tile(v, grid)
    N = len(vbs)
    idx = np.tile(np.arange(N, dtype=np.int32), (1, 2, N, 1))
    o, lse = oracle.fine_full(qt, kt, vt, idx, vbs, D ** -0.5)
    ref_o, ref_lse = sdpa_ref(f64(qt), f64(kt), f64(vt), D ** -0.5)
    assert np.abs(o - ref_o).max() < 1e-12
    assert np.abs(lse - ref_lse).max() < 1e-10


def test_dense_equivalence_with_padding():
    wl = synth.WORKLOADS["tiny"]
    d = synth.make_inputs(wl)
    qt, vbs = oracle.tile(d["q"], wl.grid)
    kt, _ = oracle.tile(d["k"], wl.grid)
    vt, _ = oracle.tile(d["v"], wl.grid)
    N = wl.ncubes
    idx = np.tile(np.arange(N, dtype=np.int32), (1, wl.heads, N, 1))
    o, lse = oracle.fine_full(qt, kt, vt, idx, vbs, wl.sm_scale)
    ref_o, ref_lse = sdpa_ref(f64(d["q"]), f64(d["k"]), f64(d["v"]), wl.sm_scale)
    # Map tiled rows back to raster tokens: untile the slot index.
    slot_ids = np.arange(64 * N, dtype=np.uint16).reshape(1, 64 * N, 1, 1)
    raster_slot = oracle.untile(slot_ids, wl.grid)[0, :, 0, 0].astype(np.int64)
    assert np.abs(o[0, raster_slot] - ref_o[0]).max() < 1e-12
    assert np.abs(lse[0][:, raster_slot] - ref_lse[0]).max() < 1e-10


def brute_force(qt, kt, vt, idx, vbs, scale, counts=None):
    """Explicit masked [S_pad x S_pad] softmax per (b, head); with counts, row
    cube i attends idx[b, h, i, :counts[b, h, i]] (every count >= 1)."""
    B, S, H, D = qt.shape
    N = S // 64
    q, k, v = f64(qt), f64(kt), f64(vt)
    o = np.zeros((B, S, H, D))
    lse = np.zeros((B, H, S))
    key_cube = np.arange(S) // 64
    key_ok = (np.arange(S) % 64) < vbs[key_cube]
    for b in range(B):
        for h in range(H):
            logits = scale * q[b, :, h] @ k[b, :, h].T
            allowed = np.zeros((S, S), bool)
            for i in range(N):
                row = idx[b, h, i] if counts is None else idx[b, h, i, :counts[b, h, i]]
                sel = np.isin(key_cube, row) & key_ok
                allowed[64 * i: 64 * (i + 1)] = sel[None]
            masked = np.where(allowed, logits, -np.inf)
            m = masked.max(axis=1, keepdims=True)
            w = np.exp(masked - m)
            o[b, :, h] = (w @ v[b, :, h]) / w.sum(axis=1, keepdims=True)
            lse[b, h] = (m[:, 0] + np.log(w.sum(axis=1)))
    return o, lse


def tiny_case(topk=None, seed_idx=None):
    wl = synth.WORKLOADS["tiny"]
    d = synth.make_inputs(wl)
    qt, vbs = oracle.tile(d["q"], wl.grid)
    kt, _ = oracle.tile(d["k"], wl.grid)
    vt, _ = oracle.tile(d["v"], wl.grid)
    if seed_idx is None:
        idx = oracle.coarse(qt, kt, vbs, topk or wl.topk, wl.sm_scale)
    else:
        idx = synth.random_topk(seed_idx, 1, wl.heads, wl.ncubes, topk or wl.topk)
    return wl, qt, kt, vt, idx, vbs


@pytest.mark.parametrize("seed_idx", [None, 7])
def test_brute_force_masked_matrix(seed_idx):
    wl, qt, kt, vt, idx, vbs = tiny_case(seed_idx=seed_idx)
    o, lse = oracle.fine_full(qt, kt, vt, idx, vbs, wl.sm_scale)
    ref_o, ref_lse = brute_force(qt, kt, vt, idx, vbs, wl.sm_scale)
    assert np.abs(o - ref_o).max() < 1e-12
    assert np.abs(lse - ref_lse).max() < 1e-10


def test_index_order_invariance():
    wl, qt, kt, vt, idx, vbs = tiny_case(topk=5)
    rng = np.random.default_rng(3)
    perm = idx.copy()
    for r in np.ndindex(idx.shape[:3]):
        perm[r] = rng.permutation(idx[r])
    a, la = oracle.fine_full(qt, kt, vt, idx, vbs, wl.sm_scale)
    b, lb = oracle.fine_full(qt, kt, vt, perm, vbs, wl.sm_scale)
    assert np.abs(a - b).max() < 1e-12 and np.abs(la - lb).max() < 1e-12


def test_padded_slots_are_ignored():
    wl, qt, kt, vt, idx, vbs = tiny_case(topk=6)
    rng = np.random.default_rng(4)
    k2, v2 = kt.copy(), vt.copy()
    for c in range(wl.ncubes):
        k2[:, 64 * c + vbs[c]: 64 * (c + 1)] = rand_bits(rng, k2[:, 64 * c + vbs[c]: 64 * (c + 1)].shape, 50.0)
        v2[:, 64 * c + vbs[c]: 64 * (c + 1)] = rand_bits(rng, v2[:, 64 * c + vbs[c]: 64 * (c + 1)].shape, 50.0)
    a, la = oracle.fine_full(qt, kt, vt, idx, vbs, wl.sm_scale)
    b, lb = oracle.fine_full(qt, k2, v2, idx, vbs, wl.sm_scale)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


def test_constant_values_give_the_constant():
    wl, qt, kt, vt, idx, vbs = tiny_case()
    c = synth.bf16_bits(np.linspace(-1, 1, wl.D, dtype=np.float32))
    vconst = np.broadcast_to(c, vt.shape).copy()
    o, _ = oracle.fine_full(qt, kt, vconst, idx, vbs, wl.sm_scale)
    assert np.abs(o - f64(c)).max() < 1e-14


def test_zero_query_rows_closed_form():
    wl, qt, kt, vt, idx, vbs = tiny_case()
    o, lse = oracle.fine_full(qt, kt, vt, idx, vbs, wl.sm_scale)
    v = f64(vt)
    for h in range(wl.heads):
        for i in range(wl.ncubes):
            keys = np.concatenate([64 * j + np.arange(vbs[j]) for j in idx[0, h, i]])
            for r in range(vbs[i], 64):  # padding query rows hold q = 0
                assert np.abs(o[0, 64 * i + r, h] - v[0, keys, h].mean(axis=0)).max() < 1e-14
                assert abs(lse[0, h, 64 * i + r] - np.log(len(keys))) < 1e-12


def test_single_key():
    rng = np.random.default_rng(5)
    N, H, D = 3, 1, 64
    qt, kt, vt = (rand_bits(rng, (1, 64 * N, H, D)) for _ in range(3))
    vbs = np.array([1, 64, 64], np.int32)
    idx = np.zeros((1, H, N, 1), np.int32)  # every query cube attends cube 0 = one key
    o, lse = oracle.fine_full(qt, kt, vt, idx, vbs, 0.3)
    assert np.array_equal(o[0, :, 0], np.broadcast_to(f64(vt)[0, 0, 0], (64 * N, D)))
    logit = 0.3 * f64(qt)[0, :, 0] @ f64(kt)[0, 0, 0]
    assert np.abs(lse[0, 0] - logit).max() < 1e-12


def test_empty_key_set_gives_zero_and_neg_inf():
    rng = np.random.default_rng(6)
    N, H, D = 2, 1, 64
    qt, kt, vt = (rand_bits(rng, (1, 64 * N, H, D)) for _ in range(3))
    vbs = np.array([0, 64], np.int32)
    idx = np.zeros((1, H, N, 1), np.int32)
    o, lse = oracle.fine_full(qt, kt, vt, idx, vbs, 0.1)
    assert (o == 0).all() and np.isneginf(lse).all()


def outlier_case():
    """A reduced-size stand-in for the outlier workload: head 0 logits ~1e3."""
    wl = synth.Workload("outlier_small", 1, 9, 16, 16, heads=3, D=128, topk=12, seed=77, outlier=True)
    d = synth.make_inputs(wl)
    qt, vbs = oracle.tile(d["q"], wl.grid)
    kt, _ = oracle.tile(d["k"], wl.grid)
    vt, _ = oracle.tile(d["v"], wl.grid)
    idx, scores = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale, want_scores=True)
    return wl, qt, kt, vt, idx, vbs


def test_outlier_logits_stay_finite():
    wl, qt, kt, vt, idx, vbs = outlier_case()
    o, lse = oracle.fine_full(qt, kt, vt, idx, vbs, wl.sm_scale)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    # The head-0 logits really are large enough to overflow exp without a max shift.
    q, k = f64(qt)[0, :, 0], f64(kt)[0, :, 0]
    assert (wl.sm_scale * q @ k.T).max() > 710.0


# ---- per-row counts (variable-length selection lists)
def test_counts_equal_to_topk_is_the_fixed_length_stage():
    wl, qt, kt, vt, idx, vbs = tiny_case(topk=5)
    full = np.full(idx.shape[:3], idx.shape[-1], np.int32)
    a, la = oracle.fine_full(qt, kt, vt, idx, vbs, wl.sm_scale)
    b, lb = oracle.fine_full_counts(qt, kt, vt, idx, full, vbs, wl.sm_scale)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


@pytest.mark.parametrize("seed", [0, 1])
def test_counts_brute_force(seed):
    wl, qt, kt, vt, idx, vbs = tiny_case(topk=6)
    rng = np.random.default_rng(40 + seed)
    counts = rng.integers(1, idx.shape[-1] + 1, size=idx.shape[:3]).astype(np.int32)
    garbage = idx.copy()
    for r in np.ndindex(idx.shape[:3]):  # entries past the count are never read
        garbage[r][counts[r]:] = rng.integers(0, wl.ncubes, size=idx.shape[-1] - counts[r])
    o, lse = oracle.fine_full_counts(qt, kt, vt, garbage, counts, vbs, wl.sm_scale)
    ref_o, ref_lse = brute_force(qt, kt, vt, idx, vbs, wl.sm_scale, counts)
    assert np.abs(o - ref_o).max() < 1e-12
    assert np.abs(lse - ref_lse).max() < 1e-10


def test_count_zero_rows_are_empty():
    wl, qt, kt, vt, idx, vbs = tiny_case(topk=4)
    counts = np.full(idx.shape[:3], 4, np.int32)
    counts[0, 1, 2] = 0
    o, lse = oracle.fine_full_counts(qt, kt, vt, idx, counts, vbs, wl.sm_scale)
    assert (o[0, 128:192, 1] == 0).all() and np.isneginf(lse[0, 1, 128:192]).all()
    ref_o, ref_lse = oracle.fine_full(qt, kt, vt, idx, vbs, wl.sm_scale)
    keep = np.ones(o.shape[1], bool)
    keep[128:192] = False
    assert np.array_equal(o[0, keep, 1], ref_o[0, keep, 1])
    assert np.array_equal(o[:, :, 0], ref_o[:, :, 0]) and np.array_equal(lse[0, 0], ref_lse[0, 0])
