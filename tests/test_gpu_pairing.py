"""GPU query-cube pairing (vsa_pair_cubes) and the fine stage run with it.

The pairing is a schedule, not part of the method: it decides which two query
cubes share a 128-row tensor-core tile.  It is integer work, so the GPU result
must equal, unit for unit, the plain restatement of the same procedure in
tests/pairing_ref.py.  Every cube must appear exactly once, and the fine stage
run with the pairing must match the fp64 oracle like the unpaired one.
"""
import numpy as np
import pytest
import torch

import block_sparse_video_vsa_gb300 as vsa
import oracle
import pairing_ref
from block_sparse_video_vsa_gb300 import synth
from gpu_util import (assert_lse_close, assert_scoring_rule, i32_dev, score_outputs, tiled_inputs,
                      to_bits, to_dev)

pytestmark = pytest.mark.gpu


def gpu_pairs(idx):
    p = vsa.pair_cubes(i32_dev(idx))
    torch.cuda.synchronize()
    return p.cpu().numpy().view(np.uint32)


def decode(units_u32):
    out = []
    for e in units_u32:
        i, j = int(e & 0xFFFF), int(e >> 16)
        out.append((i, -1 if j == 0xFFFF else j))
    return out


def check_partition(units, n):
    assert len(units) == (n + 1) // 2
    seen = np.zeros(n, np.int64)
    prev = -1
    singles = 0
    for i, j in units:
        assert i > prev, "units must be in increasing order of their first cube"
        prev = i
        seen[i] += 1
        if j < 0:
            singles += 1
        else:
            assert i < j < n
            seen[j] += 1
    assert (seen == 1).all(), "every cube exactly once"
    assert singles == n % 2


def compare_with_reference(idx):
    B, H, N, k = idx.shape
    got = gpu_pairs(idx)
    for b in range(B):
        for h in range(H):
            units = decode(got[b, h])
            check_partition(units, N)
            ref = pairing_ref.pair_cubes([idx[b, h, i] for i in range(N)], N)
            assert units == ref, f"(b={b}, h={h}) differs from the reference procedure"


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_pairing_matches_reference_on_coarse_selections(name):
    wl = synth.WORKLOADS[name]
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    compare_with_reference(oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale))


@pytest.mark.parametrize("N,k,heads,seed", [(1, 1, 1, 1), (2, 1, 2, 2), (3, 3, 1, 3), (75, 10, 3, 4),
                                             (624, 78, 2, 5), (1920, 192, 1, 6)])
def test_pairing_matches_reference_on_random_selections(N, k, heads, seed):
    # random lists leave many cubes unpaired after the first rounds: the
    # leftover window, its length cap (640 cubes) and the final
    # index-order pairing all run
    compare_with_reference(synth.random_topk(seed, 1, heads, N, k))


def test_pairing_batch_two_window_pattern():
    idx = synth.window_topk((3, 5, 6), (1, 1, 1), 2, 2)  # 90 cubes, 27 per list
    compare_with_reference(idx)


def test_pairing_ignores_out_of_range_entries():
    idx = synth.random_topk(7, 1, 2, 40, 6)
    idx[0, 0, 3, 2] = -5
    idx[0, 1, 7, 0] = 40
    got = gpu_pairs(idx)
    for h in range(2):
        check_partition(decode(got[0, h]), 40)


def test_pairing_deterministic():
    idx = synth.random_topk(8, 1, 3, 301, 24)
    assert np.array_equal(gpu_pairs(idx), gpu_pairs(idx))


def test_pairing_shrinks_the_unions_at_wan_size():
    wl = synth.WORKLOADS["wan"]
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
    got = gpu_pairs(idx[:, :8])
    N = wl.ncubes
    adjacent = [(2 * p, 2 * p + 1 if 2 * p + 1 < N else -1) for p in range((N + 1) // 2)]
    for h in range(8):
        rows = [idx[0, h, i] for i in range(N)]
        units = decode(got[0, h])
        check_partition(units, N)
        assert pairing_ref.union_steps(units, rows) < 0.95 * pairing_ref.union_steps(adjacent, rows)


def fine_paired_compare(wl, idx):
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    idx_d = i32_dev(idx)
    pairs = vsa.pair_cubes(idx_d)
    o, lse = vsa.sparse_attn_fwd(to_dev(qt), to_dev(kt), to_dev(vt), idx_d, i32_dev(vbs), wl.sm_scale,
                                 pairs=pairs)
    torch.cuda.synchronize()
    assert vsa.device_error(reset=True) == 0
    ref, ref_lse = oracle.fine_full(qt, kt, vt, idx, vbs, wl.sm_scale)
    assert_scoring_rule(score_outputs(to_bits(o), ref))
    assert_lse_close(lse.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_fine_with_pairing_matches_oracle(name):
    wl = synth.WORKLOADS[name]
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    fine_paired_compare(wl, oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale))


def test_fine_with_pairing_random_lists_and_odd_count():
    wl = synth.Workload("odd", 1, 9, 13, 17, heads=3, D=128, topk=9, seed=77)  # 3*4*5 = 60 cubes
    fine_paired_compare(wl, synth.random_topk(9, 1, wl.heads, wl.ncubes, wl.topk))
    wl = synth.Workload("odd2", 2, 5, 9, 13, heads=2, D=64, topk=5, seed=78)  # batch 2, 2*3*4 = 24 cubes
    fine_paired_compare(wl, synth.random_topk(10, 2, wl.heads, wl.ncubes, wl.topk))
