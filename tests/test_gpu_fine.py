"""GPU parity of vsa_sparse_attn_fwd against the fp64 oracle.

Both sides take the same topk_idx (the oracle's coarse selection, or a
structured pattern).  Small workloads are compared element by element over
every output (unpaired schedule: cubes 2u, 2u + 1 share a tile); the
full-size Wan2.2 and HunyuanVideo shapes run in the launch configuration the
benchmark times (vsa_pair_cubes, then the paired fine stage) and are compared
on sampled query cubes (all 64 rows, every channel) plus whole-output
finiteness.
"""
import numpy as np
import pytest
import torch

import block_sparse_video_vsa_gb300 as vsa
import oracle
from block_sparse_video_vsa_gb300 import synth
from gpu_util import (assert_lse_close, assert_scoring_rule, i32_dev, score_outputs, tiled_inputs,
                      to_bits, to_dev)

pytestmark = pytest.mark.gpu


def gpu_fine(qt, kt, vt, idx, vbs, sm, paired=False, counts=None):
    idx_d = i32_dev(idx)
    pairs = vsa.pair_cubes(idx_d) if paired else None
    cnt = None if counts is None else i32_dev(counts)
    o, lse = vsa.sparse_attn_fwd(to_dev(qt), to_dev(kt), to_dev(vt), idx_d, i32_dev(vbs), sm, pairs=pairs,
                                 counts=cnt)
    torch.cuda.synchronize()
    assert vsa.device_error(reset=True) == 0
    return to_bits(o), lse.cpu().numpy()


def full_compare(qt, kt, vt, idx, vbs, sm):
    got, got_lse = gpu_fine(qt, kt, vt, idx, vbs, sm)
    ref, ref_lse = oracle.fine_full(qt, kt, vt, idx, vbs, sm)
    stats = score_outputs(got, ref)
    assert_scoring_rule(stats)
    assert_lse_close(got_lse, ref_lse)
    return stats


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_workload_full_output(name):
    wl = synth.WORKLOADS[name]
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
    full_compare(qt, kt, vt, idx, vbs, wl.sm_scale)


@pytest.mark.parametrize("topk", [1, 2, 3, 11, 48])
def test_topk_range(topk):
    wl = synth.WORKLOADS["mid"]
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    idx = oracle.coarse(qt, kt, vbs, topk, wl.sm_scale)
    full_compare(qt, kt, vt, idx, vbs, wl.sm_scale)


def test_random_distinct_indices():
    wl = synth.WORKLOADS["mid"]
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    idx = synth.random_topk(21, 1, wl.heads, wl.ncubes, 13)
    full_compare(qt, kt, vt, idx, vbs, wl.sm_scale)


def test_sliding_window_pattern():
    wl = synth.WORKLOADS["mid"]  # 3 x 4 x 4 cubes
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    idx = synth.window_topk(wl.cube_grid, (1, 1, 1), 1, wl.heads)  # 27 cubes: odd count
    full_compare(qt, kt, vt, idx, vbs, wl.sm_scale)


def test_batch_two_and_head_dim_64():
    wl = synth.Workload("b2", 2, 7, 9, 11, heads=3, D=64, topk=5, seed=31, sigma=4.0)
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
    full_compare(qt, kt, vt, idx, vbs, wl.sm_scale)


def test_index_order_does_not_matter():
    wl = synth.WORKLOADS["mid"]
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
    rev = np.ascontiguousarray(idx[..., ::-1])
    a, la = gpu_fine(qt, kt, vt, idx, vbs, wl.sm_scale)
    b, lb = gpu_fine(qt, kt, vt, rev, vbs, wl.sm_scale)
    d = np.abs(synth.bf16_to_f32(a) - synth.bf16_to_f32(b))
    assert d.max() <= 2e-3 and np.abs(la - lb).max() <= 1e-4


def test_empty_cubes_give_zero_and_neg_inf():
    rng = np.random.default_rng(8)
    N, H, D = 6, 2, 128
    qt, kt, vt = (synth.bf16_bits(rng.standard_normal((1, 64 * N, H, D), dtype=np.float32)) for _ in range(3))
    vbs = np.array([0, 0, 64, 5, 0, 64], np.int32)
    idx = np.zeros((1, H, N, 2), np.int32)
    idx[..., 0], idx[..., 1] = 0, 1          # only empty cubes ...
    idx[0, 1, 3] = [4, 3]                    # ... except one row: an empty and a partial cube
    full_compare(qt, kt, vt, idx, vbs, 0.1)
    got, lse = gpu_fine(qt, kt, vt, idx, vbs, 0.1)
    assert np.isneginf(lse[0, 0]).all()


def test_outlier_small():
    wl = synth.Workload("outlier_small", 1, 9, 16, 16, heads=3, D=128, topk=12, seed=77, outlier=True)
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
    full_compare(qt, kt, vt, idx, vbs, wl.sm_scale)


def test_deterministic():
    wl = synth.WORKLOADS["mid"]
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
    a, la = gpu_fine(qt, kt, vt, idx, vbs, wl.sm_scale)
    b, lb = gpu_fine(qt, kt, vt, idx, vbs, wl.sm_scale)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


# ---------------------------------------------- per-row counts (variable length)
def ragged_counts(idx, seed, fill=-1):
    """Random counts in [0, topk] (0 and topk always present); entries past a
    row's count are overwritten by `fill` (-1, or "garbage": random cubes)."""
    rng = np.random.default_rng(seed)
    k = idx.shape[-1]
    counts = rng.integers(0, k + 1, size=idx.shape[:3]).astype(np.int32)
    counts.reshape(-1)[:4] = [0, k, 1, k]
    out = idx.copy()
    N = idx.shape[2]
    for r in np.ndindex(idx.shape[:3]):
        tail = k - counts[r]
        out[r][counts[r]:] = rng.integers(0, N, size=tail) if fill == "garbage" else fill
    return out, counts


@pytest.mark.parametrize("paired", [False, True])
@pytest.mark.parametrize("topk", [5, 48])
def test_counts_ragged_rows(paired, topk):
    wl = synth.WORKLOADS["mid"]
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    idx, counts = ragged_counts(oracle.coarse(qt, kt, vbs, topk, wl.sm_scale), 5 + topk)
    got, got_lse = gpu_fine(qt, kt, vt, idx, vbs, wl.sm_scale, paired=paired, counts=counts)
    ref, ref_lse = oracle.fine_full_counts(qt, kt, vt, idx, counts, vbs, wl.sm_scale)
    assert_scoring_rule(score_outputs(got, ref))
    assert_lse_close(got_lse, ref_lse)
    empty = np.repeat(counts == 0, 64, axis=2)                 # [B, H, S]
    assert np.isneginf(got_lse[empty]).all() and np.isfinite(got_lse[~empty]).all()
    assert (synth.bf16_to_f32(got).transpose(0, 2, 1, 3)[empty] == 0).all()


def test_counts_ignore_entries_past_the_count():
    wl = synth.WORKLOADS["mid"]
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    base = oracle.coarse(qt, kt, vbs, 11, wl.sm_scale)
    a_idx, counts = ragged_counts(base, 9)
    b_idx, _ = ragged_counts(base, 9, fill="garbage")
    a, la = gpu_fine(qt, kt, vt, a_idx, vbs, wl.sm_scale, counts=counts)
    b, lb = gpu_fine(qt, kt, vt, b_idx, vbs, wl.sm_scale, counts=counts)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


def test_counts_full_equal_the_fixed_length_call():
    wl = synth.WORKLOADS["mid"]
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    idx = oracle.coarse(qt, kt, vbs, 13, wl.sm_scale)
    full = np.full(idx.shape[:3], 13, np.int32)
    a, la = gpu_fine(qt, kt, vt, idx, vbs, wl.sm_scale)
    b, lb = gpu_fine(qt, kt, vt, idx, vbs, wl.sm_scale, counts=full)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


# ------------------------------------------------------------- full size
_CACHE = {}


def big_case(name):
    if name not in _CACHE:
        wl = synth.WORKLOADS[name]
        _, _, qt, kt, vt, vbs = tiled_inputs(wl)
        idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
        _CACHE.clear()
        _CACHE[name] = (wl, qt, kt, vt, vbs, idx)
    return _CACHE[name]


def sample_units(wl, n, seed, heads=None):
    rng = np.random.default_rng(seed)
    N = wl.ncubes
    hs = rng.integers(0, wl.heads, size=n) if heads is None else rng.choice(heads, size=n)
    cubes = rng.integers(0, N, size=n)
    cubes[:4] = [0, N - 1, N // 2, wl.cube_grid[2] - 1]  # grid corners hold partial cubes
    return np.unique(hs.astype(np.int64) * N + cubes)


def sampled_compare(wl, qt, kt, vt, vbs, idx, units, counts=None):
    # the launch configuration the benchmark times: pairing, then the paired fine stage
    got, got_lse = gpu_fine(qt, kt, vt, idx, vbs, wl.sm_scale, paired=True, counts=counts)
    assert np.isfinite(synth.bf16_to_f32(got)).all()
    if counts is None:
        ref_u, ref_lse_u, _ = oracle.fine(qt, kt, vt, idx, vbs, wl.sm_scale, units)
    else:
        ref_u, ref_lse_u, _ = oracle.fine_counts(qt, kt, vt, idx, counts, vbs, wl.sm_scale, units)
    N = wl.ncubes
    h = units // N
    i = units % N
    rows = (64 * i[:, None] + np.arange(64)[None, :])          # [u, 64]
    got_u = got[0][rows, h[:, None], :]                       # [u, 64, D]
    glse_u = got_lse[0][h[:, None], rows]                     # [u, 64]
    # Per-head cosine over the sampled rows of each head.
    by_head = {}
    for n_u, hh in enumerate(h):
        by_head.setdefault(int(hh), []).append(n_u)
    cos_min = 1.0
    for hh, us in by_head.items():
        a = synth.bf16_to_f32(got_u[us]).astype(np.float64).ravel()
        b = ref_u[us].astype(np.float32).astype(np.float64).ravel()
        na, nb = np.linalg.norm(a), np.linalg.norm(b)
        cos_min = min(cos_min, 1.0 if na == nb == 0 else float(a @ b / max(na * nb, 1e-300)))
    stats = score_outputs(got_u[None].transpose(0, 2, 1, 3), ref_u[None].transpose(0, 2, 1, 3), 2)
    stats["min_head_cos"] = cos_min
    assert_scoring_rule(stats)
    assert_lse_close(glse_u, ref_lse_u)
    return stats


def test_wan_full_size_sampled():
    wl, qt, kt, vt, vbs, idx = big_case("wan")
    sampled_compare(wl, qt, kt, vt, vbs, idx, sample_units(wl, 96, 1))


@pytest.mark.parametrize("topk", [187, 78, 31])
def test_wan_outlier_sweep_sampled(topk):
    wl0, qt, kt, vt, vbs, _ = big_case("wan_outlier")
    wl = wl0.with_topk(topk)
    idx = oracle.coarse(qt, kt, vbs, topk, wl.sm_scale)
    units = sample_units(wl, 48, 2 + topk, heads=[0, 0, 0, 1, 2, 5])
    sampled_compare(wl, qt, kt, vt, vbs, idx, units)


def test_wan_full_size_counts_sampled():
    wl, qt, kt, vt, vbs, idx = big_case("wan")
    ridx, counts = ragged_counts(idx, 17)
    units = sample_units(wl, 64, 4)
    counts.reshape(-1)[units[:2]] = 0                          # sampled empty rows as well
    sampled_compare(wl, qt, kt, vt, vbs, ridx, units, counts)


def test_hunyuan_full_size_sampled():
    wl, qt, kt, vt, vbs, idx = big_case("hunyuan")
    sampled_compare(wl, qt, kt, vt, vbs, idx, sample_units(wl, 32, 3))
