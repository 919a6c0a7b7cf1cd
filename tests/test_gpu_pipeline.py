"""End to end on the GPU: tile k, v (q, k pooled in the same pass) -> coarse
select -> pairing -> sparse attention on raster q, written in raster order,
against the oracle's own end-to-end result on the same raster inputs."""
import numpy as np
import pytest
import torch

import block_sparse_video_vsa_gb300 as vsa
import oracle
from block_sparse_video_vsa_gb300 import synth
from gpu_util import assert_lse_close, assert_scoring_rule, score_outputs, to_bits, to_dev

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
