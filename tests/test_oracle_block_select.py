"""Pins of the oracle's mean-pool block selector with a cumulative threshold
("Optimizing block-sparse INT8 attention and multi-expert step caching for
Wan 2.2", Decoupling Block Selection from Sparse CUDA Kernels: pool 128-token
query and key blocks, score block pairs by dot products, keep key blocks in
score order up to a cumulative-distribution threshold) and of its use with
the fine stage through the cube-level table.

Closed forms on constant blocks, limits of the threshold, a brute-force
search over key-block subsets and a dense masked softmax over the kept
blocks' tokens fix what the selector and the composition compute.
"""
import itertools

import numpy as np
import pytest

import oracle
from block_sparse_video_vsa_gb300 import synth


def blocks_from_vectors(vecs, block):
    """[heads, nb, D] per-block constant vectors -> raster bits [1, nb*block, heads, D]."""
    heads, nb, D = vecs.shape
    x = np.repeat(vecs.transpose(1, 0, 2)[:, None], block, axis=1).reshape(1, nb * block, heads, D)
    return synth.bf16_bits(x.astype(np.float32))


def random_qk(seed, nb, heads=2, D=32, block=128):
    rng = np.random.default_rng(seed)
    q = synth.bf16_bits(rng.standard_normal((1, nb * block, heads, D)).astype(np.float32))
    k = synth.bf16_bits(rng.standard_normal((1, nb * block, heads, D)).astype(np.float32))
    return q, k


def test_block_pool_closed_form():
    rng = np.random.default_rng(0)
    vecs = rng.integers(-6, 7, size=(3, 5, 8)).astype(np.float32)
    got = oracle.block_pool(blocks_from_vectors(vecs, 128), 128)
    assert np.array_equal(got[0], vecs.astype(np.float64))
    x = np.zeros((1, 256, 1, 4), np.float32)
    x[0, :128, 0, 0] = np.arange(128)  # mean 63.5
    assert oracle.block_pool(synth.bf16_bits(x), 128)[0, 0, 0, 0] == 63.5


def test_scores_are_block_mean_dot_products():
    rng = np.random.default_rng(1)
    qv = rng.integers(-3, 4, size=(2, 4, 8)).astype(np.float32)
    kv = rng.integers(-3, 4, size=(2, 4, 8)).astype(np.float32)
    _, _, s = oracle.block_select_cdf(blocks_from_vectors(qv, 128), blocks_from_vectors(kv, 128), 128, 0.5, 1.0)
    for h in range(2):
        assert np.array_equal(s[0, h], qv[h].astype(np.int64) @ kv[h].astype(np.int64).T)


def test_threshold_limits():
    q, k = random_qk(2, nb=6)
    idx, counts, s = oracle.block_select_cdf(q, k, 128, 1.0, 0.2)
    assert (counts == 6).all()
    assert all(sorted(r) == list(range(6)) for r in idx.reshape(-1, 6).tolist())
    idx, counts, s = oracle.block_select_cdf(q, k, 128, 1e-12, 0.2)
    assert (counts == 1).all()
    assert np.array_equal(idx[..., 0], np.argmax(s, axis=-1))
    assert (idx[..., 1:] == -1).all()


@pytest.mark.parametrize("m", [1, 3, 5])
def test_equal_scores_keep_a_fixed_share_in_index_order(m):
    nb = 6
    rng = np.random.default_rng(3)
    qv = rng.integers(-3, 4, size=(1, nb, 8)).astype(np.float32)
    kv = np.repeat(rng.integers(-3, 4, size=(1, 1, 8)).astype(np.float32), nb, axis=1)  # all keys alike
    tau = (m - 0.5) / nb  # uniform weights 1/nb: m blocks are the first to reach tau
    idx, counts, _ = oracle.block_select_cdf(blocks_from_vectors(qv, 128), blocks_from_vectors(kv, 128), 128,
                                             tau, 0.7)
    assert (counts == m).all()
    assert (idx[0, 0, :, :m] == np.arange(m)).all()


@pytest.mark.parametrize("seed, tau, scale", [(4, 0.5, 0.5), (5, 0.8, 0.5), (6, 0.95, 0.5), (7, 0.9, 8.0)])
def test_brute_force_smallest_subset(seed, tau, scale):
    q, k = random_qk(seed, nb=6, heads=1)
    idx, counts, s = oracle.block_select_cdf(q, k, 128, tau, scale)
    for i in range(6):
        w = np.exp(scale * (s[0, 0, i] - s[0, 0, i].max()))
        w /= w.sum()
        best = None
        for size in range(1, 7):  # the smallest key set whose share reaches tau
            for sub in itertools.combinations(range(6), size):
                if w[list(sub)].sum() >= tau:
                    best = size
                    break
            if best:
                break
        assert counts[0, 0, i] == best
        kept = set(idx[0, 0, i, :best].tolist())
        assert min(w[list(kept)]) >= max(np.delete(w, list(kept)), default=-1.0)


def test_block_table_to_cube_table_by_hand():
    idx = np.array([[[[2, 0, -1], [1, -1, -1], [0, 1, 2]]]], np.int32)
    counts = np.array([[[2, 1, 3]]], np.int32)
    cube_idx, cube_counts = oracle.blocks_to_cube_lut(idx, counts)
    assert cube_counts.tolist() == [[[4, 4, 2, 2, 6, 6]]]
    assert cube_idx[0, 0, 0].tolist() == [4, 5, 0, 1, -1, -1]
    assert cube_idx[0, 0, 1].tolist() == [4, 5, 0, 1, -1, -1]
    assert cube_idx[0, 0, 3].tolist() == [2, 3, -1, -1, -1, -1]
    assert cube_idx[0, 0, 5].tolist() == [0, 1, 2, 3, 4, 5]


def test_block_sparse_attention_is_dense_attention_over_kept_blocks():
    nb, heads, D, block = 4, 2, 64, 128
    rng = np.random.default_rng(7)
    q, k = random_qk(8, nb, heads, D)
    v = synth.bf16_bits(rng.standard_normal((1, nb * block, heads, D)).astype(np.float32))
    scale = 1 / np.sqrt(D)
    idx, counts, _ = oracle.block_select_cdf(q, k, block, 0.7, scale)
    assert 1 <= counts.min() and counts.max() < nb  # some blocks dropped
    cube_idx, cube_counts = oracle.blocks_to_cube_lut(idx, counts)
    vbs = np.full(2 * nb, 64, np.int32)  # no padding: the raster sequence is its own tiled layout
    out, lse = oracle.fine_full_counts(q, k, v, cube_idx, cube_counts, vbs, scale)
    qf, kf, vf = (synth.bf16_to_f32(x).astype(np.float64) for x in (q, k, v))
    for h in range(heads):
        for i in range(nb):
            keys = np.concatenate([np.arange(j * block, (j + 1) * block) for j in idx[0, h, i, :counts[0, h, i]]])
            rows = slice(i * block, (i + 1) * block)
            logits = scale * qf[0, rows, h] @ kf[0, keys, h].T
            mx = logits.max(axis=1, keepdims=True)
            w = np.exp(logits - mx)
            ref = (w / w.sum(1, keepdims=True)) @ vf[0, keys, h]
            assert np.abs(out[0, rows, h] - ref).max() < 1e-12
            assert np.abs(lse[0, h, rows] - (mx[:, 0] + np.log(w.sum(1)))).max() < 1e-12
