"""GPU parity of vsa_tile_pool + vsa_coarse_select_pooled.

The fused pass must give the same bits as the separate calls it replaces:
tiled q and k and vbs equal to the oracle's tiling (bit-exact), the pooled
statistics equal byte for byte to those vsa_coarse_select computes from the
tiled tensors, and topk_idx equal to vsa_coarse_select's (and, like it, to
the oracle's exact top-k under the tie rule of test_gpu_coarse)."""
import numpy as np
import pytest
import torch

import block_sparse_video_vsa_gb300 as vsa
import oracle
from block_sparse_video_vsa_gb300 import synth
from gpu_util import check_topk_tie_rule, to_bits, to_dev

pytestmark = pytest.mark.gpu


def pooled_bytes(B, heads, N, D):
    """Size of the workspace head the pooling writes (means, residuals, norms)."""
    return 16 * B * heads * N * D + 8 * B * heads * N


def fused_vs_separate(q, k, grid, topk, sm):
    B, _, heads, D = q.shape
    qd, kd = to_dev(q), to_dev(k)
    qt, kt, vbs, ws = vsa.tile_pool(qd, kd, grid)
    idx = vsa.coarse_select_pooled(ws, vbs, B, heads, D, topk, sm)
    torch.cuda.synchronize()
    qt_s, vbs_s = vsa.tile(qd, grid)
    kt_s, _ = vsa.tile(kd, grid)
    ws_s = torch.empty_like(ws)
    idx_s = vsa.coarse_select(qt_s, kt_s, vbs_s, topk, sm, workspace=ws_s)
    torch.cuda.synchronize()
    N = vbs.numel()
    head = pooled_bytes(B, heads, N, D)
    assert torch.equal(qt, qt_s) and torch.equal(kt, kt_s) and torch.equal(vbs, vbs_s)
    assert torch.equal(ws[:head], ws_s[:head]), "pooled statistics differ from vsa_coarse_select's"
    assert torch.equal(idx, idx_s)
    return qt, kt, vbs, idx


@pytest.mark.parametrize("name,B", [("tiny", 1), ("mid", 1), ("mid", 2), ("wan_outlier", 1)])
def test_fused_equals_separate_and_oracle(name, B):
    wl = synth.WORKLOADS[name]
    d = synth.make_inputs(wl, B)
    grid = (d["q"].shape[0],) + wl.grid[1:]
    qt, kt, vbs, idx = fused_vs_separate(d["q"], d["k"], grid, wl.topk, wl.sm_scale)
    ref_qt, ref_vbs = oracle.tile(d["q"], grid)
    ref_kt, _ = oracle.tile(d["k"], grid)
    assert np.array_equal(to_bits(qt), ref_qt) and np.array_equal(to_bits(kt), ref_kt)
    assert np.array_equal(vbs.cpu().numpy(), ref_vbs)
    _, scores = oracle.coarse(ref_qt, ref_kt, ref_vbs, wl.topk, wl.sm_scale, want_scores=True)
    rows, differ = check_topk_tie_rule(idx.cpu().numpy(), scores, wl.topk)
    assert differ <= rows * 1e-3 if wl.ncubes >= 256 else differ == 0


@pytest.mark.parametrize("B,grid,heads,D,topk", [
    (1, (5, 6, 10), 1, 64, 3),      # 8 columns per row: a 64-thread block, mostly idle
    (2, (3, 5, 7), 3, 64, 2),       # batch 2, every cube partial
    (1, (8, 8, 8), 5, 128, 4),      # no padding; 80 columns
    (1, (9, 16, 16), 24, 128, 9),   # 384 columns: 192 threads, two columns each
    (1, (13, 36, 36), 3, 128, 30),  # 324 cubes: scores through memory
])
def test_fused_shapes(B, grid, heads, D, topk):
    g = (B,) + grid
    S = int(np.prod(grid))
    rng = np.random.default_rng(sum(grid) + heads)
    q = synth.bf16_bits(rng.standard_normal((B, S, heads, D), dtype=np.float32))
    k = synth.bf16_bits(rng.standard_normal((B, S, heads, D), dtype=np.float32))
    qt, kt, vbs, idx = fused_vs_separate(q, k, g, topk, 0.0)
    ref_qt, ref_vbs = oracle.tile(q, g)
    assert np.array_equal(to_bits(qt), ref_qt) and np.array_equal(vbs.cpu().numpy(), ref_vbs)


def test_wan_full_size():
    """The Wan2.2 shape (624 cubes, 40 heads): tiling bit-exact against the
    oracle, statistics and top-k equal to the separate calls."""
    wl = synth.WORKLOADS["wan"]
    d = synth.make_inputs(wl)
    qt, kt, vbs, idx = fused_vs_separate(d["q"], d["k"], wl.grid, wl.topk, wl.sm_scale)
    ref_qt, ref_vbs = oracle.tile(d["q"], wl.grid)
    assert np.array_equal(to_bits(qt), ref_qt) and np.array_equal(vbs.cpu().numpy(), ref_vbs)


def test_refusals():
    wl = synth.WORKLOADS["tiny"]
    d = synth.make_inputs(wl)
    q, k = to_dev(d["q"]), to_dev(d["k"])
    with pytest.raises(ValueError):
        vsa.tile_pool(q, k[:, :-1], wl.grid)
    small = torch.empty((16,), dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        vsa.tile_pool(q, k, wl.grid, workspace=small)
    x16 = to_dev(synth.bf16_bits(np.zeros((1, d["q"].shape[1], d["q"].shape[2], 16), np.float32)))
    with pytest.raises(vsa.VsaError):
        vsa.tile_pool(x16, x16, wl.grid)  # D = 16: no pooled statistics
    _, _, vbs, ws = vsa.tile_pool(q, k, wl.grid)
    with pytest.raises(vsa.VsaError):
        vsa.coarse_select_pooled(ws, vbs, 1, wl.heads, wl.D, wl.ncubes + 1, 0.0)
