"""Pins of the oracle's coarse stage (cube mean-pool, cube scores, top-k).

Follows "VSA: Accelerating Video Diffusion Inference with Sparse Attention on
AMD GPUs" (Stage 1: Coarse Selection; Generating Sparsity Patterns: pool,
einsum score, top-k).  The pins do not retype the oracle: they use closed
forms on integer-valued cubes (exact in binary floating point), a numpy
einsum + argsort restatement, invariances, and hand-built cases.
"""
import numpy as np
import pytest

import oracle
from block_sparse_video_vsa_gb300 import synth


def tiled_from_cube_vectors(vecs, vbs, pad_value=None, rng=None):
    """[heads, N, D] per-cube constant vectors -> tiled [1, 64N, heads, D] bits.
    Padding slots (s >= vbs) get pad_value (or zero)."""
    heads, N, D = vecs.shape
    xt = np.zeros((1, 64 * N, heads, D), np.float32)
    for c in range(N):
        xt[0, 64 * c: 64 * c + vbs[c]] = vecs[:, c][None]
        if pad_value is not None:
            xt[0, 64 * c + vbs[c]: 64 * (c + 1)] = pad_value
    return synth.bf16_bits(xt)


def test_pool_uses_only_real_tokens():
    rng = np.random.default_rng(0)
    N, heads, D = 5, 2, 8
    vbs = np.array([64, 5, 1, 33, 17], np.int32)
    vals = rng.integers(-8, 8, size=(1, 64 * N, heads, D)).astype(np.float32)
    for c in range(N):
        vals[0, 64 * c + vbs[c]: 64 * (c + 1)] = 4096.0  # must be ignored
    xt = synth.bf16_bits(vals)
    got = oracle.pool(xt, vbs)
    for c in range(N):
        ref = vals[0, 64 * c: 64 * c + vbs[c]].astype(np.float64).mean(axis=0)  # [heads, D]
        assert np.array_equal(got[0, :, c], ref)


def test_constant_cubes_closed_form():
    rng = np.random.default_rng(1)
    N, heads, D, k = 9, 3, 16, 4
    vbs = np.array([64, 12, 64, 3, 64, 48, 1, 64, 20], np.int32)
    qv = rng.integers(-3, 4, size=(heads, N, D)).astype(np.float32)
    kv = rng.integers(-3, 4, size=(heads, N, D)).astype(np.float32)
    qt = tiled_from_cube_vectors(qv, vbs, pad_value=100.0)
    kt = tiled_from_cube_vectors(kv, vbs, pad_value=-100.0)
    idx, scores = oracle.coarse(qt, kt, vbs, k, 0.25, want_scores=True)
    for h in range(heads):
        exact = 0.25 * (qv[h].astype(np.int64) @ kv[h].astype(np.int64).T)  # exact integers / 4
        assert np.array_equal(scores[0, h], exact)
        for i in range(N):
            order = sorted(range(N), key=lambda j: (-exact[i, j], j))
            assert list(idx[0, h, i]) == order[:k]


def test_topk_all_cubes():
    wl = synth.WORKLOADS["tiny"]
    d = synth.make_inputs(wl)
    qt, vbs = oracle.tile(d["q"], wl.grid)
    kt, _ = oracle.tile(d["k"], wl.grid)
    idx = oracle.coarse(qt, kt, vbs, wl.ncubes, wl.sm_scale)
    assert (np.sort(idx, -1) == np.arange(wl.ncubes)).all()


def test_scale_invariance():
    wl = synth.WORKLOADS["mid"]
    d = synth.make_inputs(wl)
    qt, vbs = oracle.tile(d["q"], wl.grid)
    kt, _ = oracle.tile(d["k"], wl.grid)
    a = oracle.coarse(qt, kt, vbs, wl.topk, 0.05)
    b = oracle.coarse(qt, kt, vbs, wl.topk, 7.0)
    assert np.array_equal(a, b)


def test_einsum_argsort_restatement():
    wl = synth.WORKLOADS["mid"]
    d = synth.make_inputs(wl)
    qt, vbs = oracle.tile(d["q"], wl.grid)
    kt, _ = oracle.tile(d["k"], wl.grid)
    idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
    N, heads = wl.ncubes, wl.heads

    def pool_np(xt):
        x = synth.bf16_to_f32(xt).astype(np.float64)[0].reshape(N, 64, heads, wl.D)
        mask = (np.arange(64)[None, :] < vbs[:, None]).astype(np.float64)
        return np.einsum("cshd,cs->hcd", x, mask) / vbs[None, :, None]

    qm, km = pool_np(qt), pool_np(kt)
    sc = wl.sm_scale * np.einsum("hqd,hkd->hqk", qm, km)
    checked = 0
    for h in range(heads):
        for i in range(N):
            row = sc[h, i]
            order = np.argsort(-row, kind="stable")
            srt = row[order]
            gap = np.abs(srt[wl.topk - 1] - srt[wl.topk])
            if gap <= 1e-9 * np.abs(row).max():
                continue  # near-tie at the boundary: the restatement is not decisive
            assert set(idx[0, h, i].tolist()) == set(order[: wl.topk].tolist())
            checked += 1
    assert checked > 0.95 * heads * N


def test_two_cube_hand_cases():
    D = 4
    e0 = np.eye(D, dtype=np.float32)[0]
    qv = np.stack([e0, -e0])[None]     # query cube 0 points along +e0, cube 1 along -e0
    kv = np.stack([-e0, e0])[None]     # key cube 0 along -e0, key cube 1 along +e0
    vbs = np.array([64, 7], np.int32)
    idx = oracle.coarse(tiled_from_cube_vectors(qv, vbs), tiled_from_cube_vectors(kv, vbs), vbs, 1, 1.0)
    assert idx[0, 0, 0, 0] == 1 and idx[0, 0, 1, 0] == 0


def test_ties_go_to_the_lower_index():
    N, D = 6, 8
    vbs = np.full(N, 64, np.int32)
    qt = tiled_from_cube_vectors(np.zeros((1, N, D), np.float32), vbs)
    kt = tiled_from_cube_vectors(np.ones((1, N, D), np.float32), vbs)
    idx = oracle.coarse(qt, kt, vbs, 3, 1.0)
    assert (idx[0, 0] == np.array([0, 1, 2])).all()
