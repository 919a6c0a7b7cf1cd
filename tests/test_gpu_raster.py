"""GPU parity of vsa_sparse_attn_fwd_raster (q read and the output written in
raster token order) and of vsa_tile_pool without a tiled copy of q.

The raster path runs the same arithmetic as the tiled one, so its output must
equal vsa_untile of the tiled output bit for bit, and lse must be identical;
the tiled path itself is checked against the oracle in test_gpu_fine, and
test_gpu_pipeline checks the raster pipeline against the oracle end to end."""
import numpy as np
import pytest
import torch

import block_sparse_video_vsa_gb300 as vsa
from block_sparse_video_vsa_gb300 import synth
from gpu_util import i32_dev, to_dev

pytestmark = pytest.mark.gpu


def raster_vs_tiled(q, k, v, grid, topk, sm, paired=True, counts=None):
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    qt, kt, vbs, ws = vsa.tile_pool(qd, kd, grid)
    vt, _ = vsa.tile(vd, grid, vbs=torch.empty_like(vbs))
    B, _, heads, D = q.shape
    idx = vsa.coarse_select_pooled(ws, vbs, B, heads, D, topk, sm)
    pairs = vsa.pair_cubes(idx) if paired else None
    ot, lse_t = vsa.sparse_attn_fwd(qt, kt, vt, idx, vbs, sm, pairs=pairs, counts=counts)
    ref = vsa.untile(ot, grid)
    out, lse = vsa.sparse_attn_fwd_raster(qd, kt, vt, idx, vbs, grid, sm, pairs=pairs, counts=counts)
    torch.cuda.synchronize()
    assert vsa.device_error(reset=True) == 0
    assert torch.equal(out, ref), "raster output differs from untile(tiled output)"
    assert torch.equal(lse, lse_t)
    return qd, kd, kt, vbs, ws


@pytest.mark.parametrize("name,B,paired", [("tiny", 1, True), ("tiny", 1, False), ("mid", 2, True),
                                           ("wan_outlier", 1, True)])
def test_raster_equals_untiled_tiled_output(name, B, paired):
    wl = synth.WORKLOADS[name]
    d = synth.make_inputs(wl, B)
    grid = (d["q"].shape[0],) + wl.grid[1:]
    raster_vs_tiled(d["q"], d["k"], d["v"], grid, wl.topk, wl.sm_scale, paired)


@pytest.mark.parametrize("B,grid,heads,D,topk", [
    (2, (3, 5, 7), 3, 64, 2),      # every cube partial, D = 64, batch 2
    (1, (8, 8, 8), 2, 128, 4),     # no padding slot at all
    (1, (1, 1, 1), 1, 64, 1),      # one token, one cube
])
def test_raster_shapes(B, grid, heads, D, topk):
    g = (B,) + grid
    S = int(np.prod(grid))
    rng = np.random.default_rng(S + heads)
    x = [synth.bf16_bits(rng.standard_normal((B, S, heads, D), dtype=np.float32)) for _ in range(3)]
    raster_vs_tiled(*x, g, topk, 0.0)


def test_raster_with_counts_and_empty_rows():
    """Per-row counts, some rows empty (their raster rows are written as zeros
    and lse as -inf, as in the tiled path)."""
    wl = synth.WORKLOADS["mid"]
    d = synth.make_inputs(wl)
    rng = np.random.default_rng(3)
    counts = rng.integers(0, wl.topk + 1, size=(1, wl.heads, wl.ncubes)).astype(np.int32)
    counts[0, 0, :5] = 0
    raster_vs_tiled(d["q"], d["k"], d["v"], wl.grid, wl.topk, wl.sm_scale, counts=i32_dev(counts))


def test_tile_pool_without_qt():
    """want_qt=False (and want_kt=False): kt, vbs and the pooled statistics as
    with the copies."""
    wl = synth.WORKLOADS["mid"]
    d = synth.make_inputs(wl)
    q, k = to_dev(d["q"]), to_dev(d["k"])
    qt, kt, vbs, ws = vsa.tile_pool(q, k, wl.grid)
    qt2, kt2, vbs2, ws2 = vsa.tile_pool(q, k, wl.grid, want_qt=False)
    torch.cuda.synchronize()
    assert qt2 is None
    head = 16 * wl.heads * wl.ncubes * wl.D + 8 * wl.heads * wl.ncubes
    assert torch.equal(kt, kt2) and torch.equal(vbs, vbs2) and torch.equal(ws[:head], ws2[:head])
    qt3, kt3, vbs3, ws3 = vsa.tile_pool(q, k, wl.grid, want_qt=False, want_kt=False)  # statistics alone
    torch.cuda.synchronize()
    assert qt3 is None and kt3 is None
    assert torch.equal(vbs, vbs3) and torch.equal(ws[:head], ws3[:head])


def test_wan_full_size():
    wl = synth.WORKLOADS["wan"]
    d = synth.make_inputs(wl)
    raster_vs_tiled(d["q"], d["k"], d["v"], wl.grid, wl.topk, wl.sm_scale)


def test_raster_refusals():
    wl = synth.WORKLOADS["tiny"]
    d = synth.make_inputs(wl)
    q, k, v = (to_dev(d[n]) for n in "qkv")
    _, kt, vbs, ws = vsa.tile_pool(q, k, wl.grid, want_qt=False)
    vt, _ = vsa.tile(v, wl.grid)
    idx = vsa.coarse_select_pooled(ws, vbs, 1, wl.heads, wl.D, wl.topk, wl.sm_scale)
    with pytest.raises(ValueError):
        vsa.sparse_attn_fwd_raster(q[:, :-1], kt, vt, idx, vbs, wl.grid)
    bad = (1, wl.T + 4, wl.H, wl.W)  # a grid with more cubes than the tiled tensors hold
    with pytest.raises(ValueError):
        vsa.sparse_attn_fwd_raster(q, kt, vt, idx, vbs, bad)
