"""End to end on the GPU: tile k, v (q, k pooled in the same pass) -> coarse
select -> pairing -> sparse attention on raster q, written in raster order,
against the oracle's own end-to-end result on the same raster inputs."""
import numpy as np
import pytest
import torch

import block_sparse_video_vsa_gb300 as vsa
import oracle
from block_sparse_video_vsa_gb300 import synth
from gpu_util import assert_lse_close, assert_scoring_rule, check_topk_tie_rule, score_outputs, to_bits, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_pipeline_matches_oracle(name):
    wl = synth.WORKLOADS[name]
    d = synth.make_inputs(wl)
    out, lse, idx = vsa.pipeline(to_dev(d["q"]), to_dev(d["k"]), to_dev(d["v"]), wl.grid, wl.topk, wl.sm_scale)
    torch.cuda.synchronize()
    qt, vbs = oracle.tile(d["q"], wl.grid)
    kt, _ = oracle.tile(d["k"], wl.grid)
    vt, _ = oracle.tile(d["v"], wl.grid)
    ref_idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
    assert np.array_equal(np.sort(ref_idx, -1), idx.cpu().numpy())
    ref_t, ref_lse = oracle.fine_full(qt, kt, vt, ref_idx, vbs, wl.sm_scale)
    # Real rows in raster order: untile the oracle's tiled output row map.
    N = wl.ncubes
    slot = oracle.untile(np.arange(64 * N, dtype=np.uint16).reshape(1, -1, 1, 1), wl.grid)[0, :, 0, 0]
    ref = ref_t[:, slot.astype(np.int64)]
    assert_scoring_rule(score_outputs(to_bits(out), ref))
    assert_lse_close(lse.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("grid, expect", [
    ((1, 9, 16, 16), 9),     # 48 cubes: tile of k + pool of q, k; tile of v; fused score/top-k; pairing x5;
                             # fine stage on raster q writing raster output
    ((1, 16, 32, 32), 10),   # 256 cubes: the score GEMM and the selection run as two kernels
])
def test_launch_counter_counts_every_kernel(grid, expect):
    wl = synth.Workload("count", *grid, heads=2, D=64, topk=3, seed=5)
    d = synth.make_inputs(wl)
    q, k, v = (to_dev(d[n]) for n in "qkv")
    n0 = vsa.kernel_launches()
    vsa.pipeline(q, k, v, wl.grid, wl.topk, wl.sm_scale)
    assert vsa.kernel_launches() - n0 == expect
    torch.cuda.synchronize()
    assert vsa.device_error(reset=True) == 0


def test_pipeline_hunyuan_full_size_sampled():
    """The HunyuanVideo shape (30 x 48 x 80 grid, 1920 cubes, all 24 heads,
    k = 192) end to end through pipeline(): the tiling of q, k and v bit-exact
    against the oracle at every head, the pipeline's top-k sets against the
    oracle's exact scores (tie rule of test_gpu_coarse), and the raster output
    and lse of sampled query cubes (grid corners included) against the oracle's
    fine stage on the same selection."""
    wl = synth.WORKLOADS["hunyuan"]
    d = synth.make_inputs(wl)
    q, k, v = (to_dev(d[n]) for n in "qkv")
    out, lse, idx = vsa.pipeline(q, k, v, wl.grid, wl.topk, wl.sm_scale)
    torch.cuda.synchronize()
    assert vsa.device_error(reset=True) == 0
    tiled = {}
    for n, x in (("q", q), ("k", k), ("v", v)):
        xt, vbs = vsa.tile(x, wl.grid)
        ref_t, ref_vbs = oracle.tile(d[n], wl.grid)
        assert np.array_equal(to_bits(xt), ref_t), f"tiled {n} differs from the oracle"
        assert np.array_equal(vbs.cpu().numpy(), ref_vbs)
        tiled[n] = ref_t
        del xt
    N = wl.ncubes
    g_idx = idx.cpu().numpy()
    _, scores = oracle.coarse(tiled["q"], tiled["k"], ref_vbs, wl.topk, wl.sm_scale, want_scores=True)
    rows, differ = check_topk_tie_rule(g_idx, scores, wl.topk)
    assert differ <= rows * 1e-3
    del scores
    rng = np.random.default_rng(24)
    _, nh, nw = wl.cube_grid
    corners = [0, nw - 1, nh * nw - 1, N - nw, N - 1, N // 2]
    units = np.unique(np.concatenate([rng.integers(0, wl.heads * N, 96),
                                      (rng.integers(0, wl.heads, len(corners)) * N + corners)])).astype(np.int64)
    ref_u, ref_lse_u, _ = oracle.fine(tiled["q"], tiled["k"], tiled["v"], g_idx, ref_vbs, wl.sm_scale, units)
    # Raster token of each (cube, slot): the oracle's tiling of the token
    # index (plus one, so padding slots read -1), carried as two 16-bit halves.
    ids = (np.arange(wl.tokens, dtype=np.int64) + 1)
    lo = (ids & 0xFFFF).astype(np.uint16).reshape(1, -1, 1, 1)
    hi = (ids >> 16).astype(np.uint16).reshape(1, -1, 1, 1)
    t_lo, _ = oracle.tile(lo, wl.grid)
    t_hi, _ = oracle.tile(hi, wl.grid)
    tok_of_slot = (t_lo[0, :, 0, 0].astype(np.int64) | (t_hi[0, :, 0, 0].astype(np.int64) << 16)) - 1
    h, i = units // N, units % N
    got_out = to_bits(out)[0]  # [tokens, heads, D] bf16 bits
    got_lse = lse.cpu().numpy()
    g_rows, r_rows = [], []
    for uu, (hh, ii) in enumerate(zip(h, i)):
        vb = int(ref_vbs[ii])
        toks = tok_of_slot[64 * ii: 64 * ii + vb]
        assert (toks >= 0).all() and (tok_of_slot[64 * ii + vb: 64 * ii + 64] == -1).all()
        g_rows.append(synth.bf16_to_f32(got_out[toks, hh, :]))
        r_rows.append(ref_u[uu, :vb])
    g = np.concatenate(g_rows)[None, :, None, :]
    r = np.concatenate(r_rows)[None, :, None, :]
    assert_scoring_rule(score_outputs(g.astype(np.float32), r))
    lse_rows = 64 * i[:, None] + np.arange(64)[None, :]
    assert_lse_close(got_lse[0][h[:, None], lse_rows], ref_lse_u)
