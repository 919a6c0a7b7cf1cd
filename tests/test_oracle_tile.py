"""Pins of the oracle's cube tiling against facts the pages fix.

- The worked shape example of "Wan2.2 Production Values -- VSA Block-Sparse
  Attention Inputs + Reference" (Shapes): 21 x 30 x 52 -> 6 x 8 x 13 = 624
  cubes, 39,936 padded and 32,760 real tokens.
- Brute force: an independent enumeration of (cube, slot) for every token.
- On grids divisible by 4 the tiling is the reshape/permute partition of
  "FastVideo Guide: Sliding Tile Attention" (Implementation), restated here.
- untile(tile(x)) = x; padding slots are exactly zero.
"""
import json
import os

import numpy as np
import pytest

import oracle
from block_sparse_video_vsa_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "wan_shapes.json")


def rand_bits(rng, shape):
    return synth.bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def test_worked_shape_example():
    g = json.load(open(GOLDEN))
    T, H, W = g["grid"]
    assert oracle.num_cubes(T, H, W) == g["ncubes"] == int(np.prod(g["cube_grid"]))
    x = rand_bits(np.random.default_rng(0), (1, T * H * W, 1, 8))
    xt, vbs = oracle.tile(x, (1, T, H, W))
    assert xt.shape[1] == g["s_padded"]
    assert int(vbs.sum()) == g["real_tokens"] == T * H * W
    assert 1 - g["topk"] / g["ncubes"] == pytest.approx(g["sparsity"])
    assert sorted(set(vbs.tolist())) == [8, 16, 32, 64]


@pytest.mark.parametrize("grid,ncubes,s_pad,real,vset", [
    ((5, 6, 10), 12, 768, 300, {4, 8, 16, 32, 64}),
    ((9, 16, 16), 48, 3072, 2304, {16, 64}),
    ((30, 48, 80), 1920, 122880, 115200, {32, 64}),
])
def test_shape_arithmetic(grid, ncubes, s_pad, real, vset):
    T, H, W = grid
    assert oracle.num_cubes(T, H, W) == ncubes
    x = np.zeros((1, T * H * W, 1, 8), np.uint16)
    xt, vbs = oracle.tile(x, (1, T, H, W))
    assert xt.shape[1] == s_pad and int(vbs.sum()) == real and set(vbs.tolist()) == vset


@pytest.mark.parametrize("grid", [(5, 6, 10), (3, 5, 7), (1, 1, 1), (4, 9, 4)])
def test_brute_force_enumeration(grid):
    T, H, W = grid
    B, heads, D = 2, 2, 8
    x = rand_bits(np.random.default_rng(1), (B, T * H * W, heads, D))
    xt, vbs = oracle.tile(x, (B, T, H, W))
    nh, nw = -(-H // 4), -(-W // 4)
    N = oracle.num_cubes(T, H, W)
    members = {c: [] for c in range(N)}
    for t in range(T):
        for h in range(H):
            for w in range(W):
                members[((t // 4) * nh + h // 4) * nw + w // 4].append((t * H + h) * W + w)
    for c in range(N):
        toks = sorted(members[c])
        assert vbs[c] == len(toks)
        for s, n in enumerate(toks):
            assert np.array_equal(xt[:, 64 * c + s], x[:, n])
        assert not xt[:, 64 * c + len(toks): 64 * (c + 1)].any()


@pytest.mark.parametrize("grid", [(4, 8, 12), (8, 4, 4)])
def test_reshape_restatement_on_divisible_grids(grid):
    T, H, W = grid
    B, heads, D = 1, 3, 8
    x = rand_bits(np.random.default_rng(2), (B, T * H * W, heads, D))
    xt, vbs = oracle.tile(x, (B, T, H, W))
    nt, nh, nw = T // 4, H // 4, W // 4
    ref = (x.reshape(B, nt, 4, nh, 4, nw, 4, heads, D)
           .transpose(0, 1, 3, 5, 2, 4, 6, 7, 8)
           .reshape(B, nt * nh * nw * 64, heads, D))
    assert np.array_equal(xt, ref)
    assert (vbs == 64).all()


@pytest.mark.parametrize("grid", [(5, 6, 10), (9, 16, 16), (3, 5, 7)])
def test_untile_inverts_tile(grid):
    T, H, W = grid
    x = rand_bits(np.random.default_rng(3), (2, T * H * W, 2, 16))
    xt, _ = oracle.tile(x, (2, T, H, W))
    assert np.array_equal(oracle.untile(xt, (2, T, H, W)), x)
