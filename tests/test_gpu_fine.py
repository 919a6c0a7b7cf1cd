"""GPU parity of vsa_sparse_attn_fwd against the fp64 oracle.

Both sides take the same topk_idx (the oracle's coarse selection, or a
structured pattern).  Small workloads are compared element by element over
every output (unpaired schedule: cubes 2u, 2u + 1 share a tile).  The
full-size shapes run in the launch configuration the benchmark times
(vsa_pair_cubes, then the paired fine stage) with whole-output finiteness:
the Wan2.2 call is compared on every query cube, the outlier sweep on the
whole outlier head plus every cube an extreme token touches, and the
HunyuanVideo call and the ragged-count case on sampled query cubes (all 64
rows, every channel).
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


def test_deterministic_with_counts():
    """Rows of variable length take the dynamic unit schedule (which CTA runs
    a unit varies from run to run): the bits must not."""
    wl = synth.WORKLOADS["mid"]
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
    ridx, counts = ragged_counts(idx, 21)
    runs = [gpu_fine(qt, kt, vt, ridx, vbs, wl.sm_scale, paired=paired, counts=counts)
            for paired in (False, True) for _ in range(3)]
    for a, la in runs[1:3]:
        assert np.array_equal(a, runs[0][0]) and np.array_equal(la, runs[0][1])
    for a, la in runs[4:]:
        assert np.array_equal(a, runs[3][0]) and np.array_equal(la, runs[3][1])


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
        d, _, qt, kt, vt, vbs = tiled_inputs(wl)
        idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
        _CACHE.clear()
        _CACHE[name] = (wl, qt, kt, vt, vbs, idx, d["extreme"])
    return _CACHE[name]


def sample_units(wl, n, seed, heads=None):
    rng = np.random.default_rng(seed)
    N = wl.ncubes
    hs = rng.integers(0, wl.heads, size=n) if heads is None else rng.choice(heads, size=n)
    cubes = rng.integers(0, N, size=n)
    cubes[:4] = [0, N - 1, N // 2, wl.cube_grid[2] - 1]  # grid corners hold partial cubes
    return np.unique(hs.astype(np.int64) * N + cubes)


def extreme_units(wl, idx, extreme):
    """Units (head * N + cube) of every query cube that holds an extreme token,
    and of every query cube of that head whose selection contains such a cube."""
    nt, nh, nw = wl.cube_grid
    N = wl.ncubes
    out = set()
    for head, tok in extreme:
        t, rem = divmod(tok, wl.H * wl.W)
        h, w = divmod(rem, wl.W)
        c = ((t // 4) * nh + h // 4) * nw + w // 4
        out.add(head * N + c)
        sel = np.nonzero((idx[0, head] == c).any(axis=-1))[0]
        out.update((head * N + sel).tolist())
    return np.array(sorted(out), np.int64)


def gpu_paired(wl, qt, kt, vt, vbs, idx, counts=None):
    """The launch configuration the benchmark times: pairing, then the paired fine stage."""
    got, got_lse = gpu_fine(qt, kt, vt, idx, vbs, wl.sm_scale, paired=True, counts=counts)
    assert np.isfinite(synth.bf16_to_f32(got)).all()
    return got, got_lse


def compare_units(wl, qt, kt, vt, vbs, idx, got, got_lse, units, counts=None, chunk=4992):
    """Every row and channel of the listed units (flat (b * heads + h) * N + i)
    against the oracle, chunk by chunk; the cosine of each head is taken over
    all of that head's compared elements."""
    N, H = wl.ncubes, wl.heads
    dot, na, nb = np.zeros(H), np.zeros(H), np.zeros(H)
    seen = np.zeros(H, bool)
    max_abs, sum_abs, n_el, finite = 0.0, 0.0, 0, True
    for c0 in range(0, len(units), chunk):
        us = np.asarray(units[c0:c0 + chunk], np.int64)
        if counts is None:
            ref_u, ref_lse_u, _ = oracle.fine(qt, kt, vt, idx, vbs, wl.sm_scale, us)
        else:
            ref_u, ref_lse_u, _ = oracle.fine_counts(qt, kt, vt, idx, counts, vbs, wl.sm_scale, us)
        b, h, i = us // (H * N), (us // N) % H, us % N
        rows = 64 * i[:, None] + np.arange(64)[None, :]                       # [u, 64]
        g = synth.bf16_to_f32(got[b[:, None], rows, h[:, None], :]).astype(np.float64)  # [u, 64, D]
        r = ref_u.astype(np.float32).astype(np.float64)  # reference held in fp32, as the page's scorer
        finite &= bool(np.isfinite(g).all())
        d = np.abs(g - r)
        max_abs = max(max_abs, float(d.max()))
        sum_abs += float(d.sum())
        n_el += d.size
        for hh in np.unique(h):
            m = h == hh
            dot[hh] += float((g[m] * r[m]).sum())
            na[hh] += float((g[m] * g[m]).sum())
            nb[hh] += float((r[m] * r[m]).sum())
            seen[hh] = True
        assert_lse_close(got_lse[b[:, None], h[:, None], rows], ref_lse_u)
    cos = np.where((na == 0) & (nb == 0), 1.0, dot / np.maximum(np.sqrt(na * nb), 1e-300))
    stats = {"finite": finite, "min_head_cos": float(cos[seen].min()), "max_abs": max_abs,
             "mean_abs": sum_abs / n_el, "units": int(len(units)), "heads": int(seen.sum())}
    assert_scoring_rule(stats)
    return stats


def test_wan_full_size_every_unit():
    """All 24,960 query cubes of the Wan2.2-shape call (40 heads x 624 cubes,
    k = 78): every output element against the oracle, per-head cosine over
    each whole head."""
    wl, qt, kt, vt, vbs, idx, _ = big_case("wan")
    got, got_lse = gpu_paired(wl, qt, kt, vt, vbs, idx)
    units = np.arange(wl.B * wl.heads * wl.ncubes, dtype=np.int64)
    stats = compare_units(wl, qt, kt, vt, vbs, idx, got, got_lse, units)
    assert stats["heads"] == wl.heads


@pytest.mark.parametrize("topk", [187, 78, 31])
def test_wan_outlier_sweep(topk):
    """The outlier head (logits ~1e3) compared whole, plus every query cube
    that holds an extreme (x30) token or selects a cube that does."""
    wl0, qt, kt, vt, vbs, _, extreme = big_case("wan_outlier")
    wl = wl0.with_topk(topk)
    idx = oracle.coarse(qt, kt, vbs, topk, wl.sm_scale)
    got, got_lse = gpu_paired(wl, qt, kt, vt, vbs, idx)
    ext = extreme_units(wl, idx, extreme)
    assert len(ext) > 3
    units = np.union1d(np.arange(wl.ncubes, dtype=np.int64), ext)
    stats = compare_units(wl, qt, kt, vt, vbs, idx, got, got_lse, units)
    assert stats["heads"] == 3  # head 0 and the two heads with extreme tokens


def test_wan_full_size_counts_sampled():
    wl, qt, kt, vt, vbs, idx, _ = big_case("wan")
    ridx, counts = ragged_counts(idx, 17)
    units = sample_units(wl, 256, 4)
    counts.reshape(-1)[units[:2]] = 0                          # sampled empty rows as well
    got, got_lse = gpu_paired(wl, qt, kt, vt, vbs, ridx, counts)
    compare_units(wl, qt, kt, vt, vbs, ridx, got, got_lse, units, counts)


def test_hunyuan_full_size_sampled():
    wl, qt, kt, vt, vbs, idx, _ = big_case("hunyuan")
    got, got_lse = gpu_paired(wl, qt, kt, vt, vbs, idx)
    compare_units(wl, qt, kt, vt, vbs, idx, got, got_lse, sample_units(wl, 128, 3))


def test_named_entry_points_match_the_binding_bit_for_bit():
    """vsa_sparse_attn_fwd and vsa_sparse_attn_fwd_paired called directly
    through the C ABI give the same bits as the binding's path (the gated
    entry point with the gate pointers NULL): pins their argument order."""
    wl = synth.WORKLOADS["mid"]
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
    q, k, v = to_dev(qt), to_dev(kt), to_dev(vt)
    idx_d, vbs_d = i32_dev(idx), i32_dev(vbs)
    B, S, H, D = q.shape
    N = S // 64
    lib = vsa.library()
    st = torch.cuda.current_stream().cuda_stream
    pairs = vsa.pair_cubes(idx_d)
    for paired in (False, True):
        ref_o, ref_lse = vsa.sparse_attn_fwd(q, k, v, idx_d, vbs_d, wl.sm_scale, pairs=pairs if paired else None)
        out = torch.full_like(q, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        if paired:
            status = lib.vsa_sparse_attn_fwd_paired(q.data_ptr(), k.data_ptr(), v.data_ptr(), idx_d.data_ptr(),
                                                    vbs_d.data_ptr(), pairs.data_ptr(), B, N, H, D, wl.topk,
                                                    wl.sm_scale, out.data_ptr(), lse.data_ptr(), st)
        else:
            status = lib.vsa_sparse_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), idx_d.data_ptr(),
                                             vbs_d.data_ptr(), B, N, H, D, wl.topk, wl.sm_scale, out.data_ptr(),
                                             lse.data_ptr(), st)
        torch.cuda.synchronize()
        assert status == 0
        assert torch.equal(out.view(torch.int16), ref_o.view(torch.int16)), paired
        assert torch.equal(lse, ref_lse), paired


def test_dynamic_schedule_concurrent_streams():
    """Dynamic-schedule launches (rows with counts) on two streams at once
    take different unit-counter slots: each gives the bits it gives alone."""
    wl = synth.WORKLOADS["mid"]
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
    ridx, counts = ragged_counts(idx, 31)
    ref_a, ref_la = gpu_fine(qt, kt, vt, ridx, vbs, wl.sm_scale, counts=counts)
    ridx2, counts2 = ragged_counts(idx, 32)
    ref_b, ref_lb = gpu_fine(qt, kt, vt, ridx2, vbs, wl.sm_scale, counts=counts2)
    q, k, v, vb = to_dev(qt), to_dev(kt), to_dev(vt), i32_dev(vbs)
    args = [(i32_dev(ridx), i32_dev(counts)), (i32_dev(ridx2), i32_dev(counts2))]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    outs = []
    for rep in range(8):
        for s, (ix, cn) in zip(streams, args):
            with torch.cuda.stream(s):
                outs.append(vsa.sparse_attn_fwd(q, k, v, ix, vb, wl.sm_scale, counts=cn, stream=s))
    torch.cuda.synchronize()
    assert vsa.device_error(reset=True) == 0
    for n, (o, l) in enumerate(outs):
        ref, ref_l = (ref_a, ref_la) if n % 2 == 0 else (ref_b, ref_lb)
        assert np.array_equal(to_bits(o), ref) and np.array_equal(l.cpu().numpy(), ref_l)
