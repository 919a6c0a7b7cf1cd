"""Pins of the oracle's coarse-stage attention output and of the gated sum of
the two stages ("VSA: Accelerating Video Diffusion Inference with Sparse
Attention on AMD GPUs", Two-Stage Architecture: Stage 1 pools each cube into
cube-level Q, K, V and attends cube to cube; the final output gates the
coarse and fine outputs together).

The pins do not retype the oracle: dense attention over the pooled cubes is a
library routine (scaled_dot_product_attention in float64), and closed forms
on hand-built cubes fix the pooling, the masking of empty cubes and the
broadcast of a cube's output to its 64 token slots.
"""
import numpy as np
import pytest
import torch

import oracle
from block_sparse_video_vsa_gb300 import synth


def tiled_from_cube_vectors(vecs, vbs, pad_value=0.0):
    """[heads, N, D] per-cube constant vectors -> tiled [1, 64N, heads, D] bits;
    padding slots (s >= vbs) hold pad_value."""
    heads, N, D = vecs.shape
    xt = np.full((1, 64 * N, heads, D), pad_value, np.float32)
    for c in range(N):
        xt[0, 64 * c: 64 * c + vbs[c]] = vecs[:, c][None]
    return synth.bf16_bits(xt)


def tiled_case(name, seed=0):
    wl = synth.WORKLOADS[name]
    d = synth.make_inputs(wl)
    qt, vbs = oracle.tile(d["q"], wl.grid)
    kt, _ = oracle.tile(d["k"], wl.grid)
    vt, _ = oracle.tile(d["v"], wl.grid)
    return wl, qt, kt, vt, vbs


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_equals_dense_sdpa_on_pooled_cubes(name):
    wl, qt, kt, vt, vbs = tiled_case(name)
    got = oracle.coarse_attn(qt, kt, vt, vbs, wl.sm_scale)
    qm, km, vm = (torch.from_numpy(oracle.pool(x, vbs)) for x in (qt, kt, vt))
    ref = torch.nn.functional.scaled_dot_product_attention(qm, km, vm, scale=wl.sm_scale).numpy()
    assert np.abs(got - ref).max() < 1e-13


def test_equal_keys_give_the_plain_mean_of_values():
    rng = np.random.default_rng(3)
    heads, N, D = 2, 7, 16
    vbs = np.array([64, 9, 64, 1, 30, 64, 12], np.int32)
    qv = rng.integers(-4, 5, size=(heads, N, D)).astype(np.float32)
    kv = np.repeat(rng.integers(-4, 5, size=(heads, 1, D)).astype(np.float32), N, axis=1)  # one key for all
    vv = rng.integers(-8, 9, size=(heads, N, D)).astype(np.float32)
    qt = tiled_from_cube_vectors(qv, vbs, pad_value=50.0)
    kt = tiled_from_cube_vectors(kv, vbs, pad_value=-50.0)
    vt = tiled_from_cube_vectors(vv, vbs, pad_value=77.0)
    got = oracle.coarse_attn(qt, kt, vt, vbs, 0.3)
    mean_v = vv.astype(np.float64).mean(axis=1)  # [heads, D]: every key cube weighs the same
    for i in range(N):
        assert np.abs(got[0, :, i] - mean_v).max() < 1e-12


def test_dominant_key_cube_gives_its_value():
    heads, N, D = 1, 6, 8
    vbs = np.full(N, 64, np.int32)
    qv = np.zeros((heads, N, D), np.float32)
    qv[..., 0] = 1.0
    kv = np.zeros((heads, N, D), np.float32)
    kv[0, 4, 0] = 64.0  # score 64 * scale against every query; all others 0
    vv = np.arange(heads * N * D, dtype=np.float32).reshape(heads, N, D) / 8
    got = oracle.coarse_attn(*(tiled_from_cube_vectors(x, vbs) for x in (qv, kv, vv)), vbs, 1.0)
    w_other = np.exp(-64.0)
    expect = (vv[0, 4] + w_other * (vv[0].sum(0) - vv[0, 4])) / (1 + 5 * w_other)
    for i in range(N):
        assert np.abs(got[0, 0, i] - expect).max() < 1e-12


def test_empty_cubes_are_no_keys_and_give_zero_rows():
    wl, qt, kt, vt, vbs = tiled_case("tiny")
    full = oracle.coarse_attn(qt, kt, vt, vbs, wl.sm_scale)
    vbs2 = vbs.copy()
    vbs2[[1, 4]] = 0
    got = oracle.coarse_attn(qt, kt, vt, vbs2, wl.sm_scale)
    assert (got[:, :, [1, 4]] == 0).all()
    # the same as attending over the other cubes only
    live = np.ones(len(vbs), bool)
    live[[1, 4]] = False
    qm, km, vm = (torch.from_numpy(oracle.pool(x, vbs)) for x in (qt, kt, vt))
    ref = torch.nn.functional.scaled_dot_product_attention(qm, km[:, :, live], vm[:, :, live],
                                                           scale=wl.sm_scale).numpy()
    assert np.abs(got[:, :, live] - ref[:, :, live]).max() < 1e-13
    assert not np.allclose(got[:, :, live], full[:, :, live])


def test_gates_select_one_stage():
    wl, qt, kt, vt, vbs = tiled_case("tiny")
    idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
    fine, _ = oracle.fine_full(qt, kt, vt, idx, vbs, wl.sm_scale)
    coarse = oracle.coarse_attn(qt, kt, vt, vbs, wl.sm_scale)
    one = synth.bf16_bits(np.ones(fine.shape, np.float32))
    zero = synth.bf16_bits(np.zeros(fine.shape, np.float32))
    assert np.array_equal(oracle.gated_combine(fine, coarse, zero, one), fine)
    c_only = oracle.gated_combine(fine, coarse, one, zero)
    for i in range(len(vbs)):  # every token slot of cube i carries cube i's coarse output
        for s in (0, 17, 63):
            assert np.array_equal(c_only[0, 64 * i + s], coarse[0, :, i])


def test_gated_sum_by_hand():
    B, N, heads, D = 1, 2, 2, 4
    rng = np.random.default_rng(5)
    fine = rng.standard_normal((B, 64 * N, heads, D))
    coarse = rng.standard_normal((B, heads, N, D))
    gc = rng.integers(0, 5, size=fine.shape).astype(np.float32) / 4  # exact in bf16
    gf = rng.integers(0, 5, size=fine.shape).astype(np.float32) / 4
    got = oracle.gated_combine(fine, coarse, synth.bf16_bits(gc), synth.bf16_bits(gf))
    for t in (0, 5, 63, 64, 100, 127):
        i = t // 64
        for h in range(heads):
            want = gc[0, t, h] * coarse[0, h, i] + gf[0, t, h] * fine[0, t, h]
            assert np.abs(got[0, t, h] - want).max() < 1e-15
