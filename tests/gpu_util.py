"""Helpers shared by the GPU parity tests (imported, not collected)."""
import numpy as np
import torch

import oracle
from block_sparse_video_vsa_gb300 import synth

# Acceptance rule of "Wan2.2 Production Values -- VSA Block-Sparse Attention
# Inputs + Reference" (Scoring / loss): every element finite, per-head cosine
# >= 0.9999, max|d| <= 3e-2, mean|d| <= 1e-4.  LSE: |d| <= 1e-3 max(1, |lse|).
COS_MIN = 0.9999
MAX_ABS = 3e-2
MEAN_ABS = 1e-4
LSE_REL = 1e-3


def to_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def to_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def i32_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def tiled_inputs(wl, B=None):
    d = synth.make_inputs(wl, B)
    grid = (d["q"].shape[0],) + wl.grid[1:]
    qt, vbs = oracle.tile(d["q"], grid)
    kt, _ = oracle.tile(d["k"], grid)
    vt, _ = oracle.tile(d["v"], grid)
    return d, grid, qt, kt, vt, vbs


def score_outputs(got_bits_or_f32, ref_f64, per_head_axis=2):
    """Scoring rule on [B, S, H, D] arrays; returns a dict of statistics."""
    got = got_bits_or_f32 if got_bits_or_f32.dtype == np.float32 else synth.bf16_to_f32(got_bits_or_f32)
    got = got.astype(np.float64)
    ref = ref_f64.astype(np.float32).astype(np.float64)  # reference held in fp32, as the page's scorer
    diff = np.abs(got - ref)
    H = got.shape[per_head_axis]
    a = np.moveaxis(got, per_head_axis, 0).reshape(H, -1)
    b = np.moveaxis(ref, per_head_axis, 0).reshape(H, -1)
    na, nb = np.linalg.norm(a, axis=1), np.linalg.norm(b, axis=1)
    cos = (a * b).sum(1) / np.maximum(na * nb, 1e-300)
    cos = np.where((na == 0) & (nb == 0), 1.0, cos)  # both all-zero (no attended key)
    return {
        "finite": bool(np.isfinite(got).all()),
        "min_head_cos": float(cos.min()),
        "max_abs": float(diff.max()),
        "mean_abs": float(diff.mean()),
        "mean_abs_ref": float(np.abs(ref).mean()),
    }


def assert_scoring_rule(stats, cos_min=COS_MIN):
    assert stats["finite"], stats
    assert stats["min_head_cos"] >= cos_min, stats
    assert stats["max_abs"] <= MAX_ABS, stats
    assert stats["mean_abs"] <= MEAN_ABS, stats


def assert_lse_close(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    both_inf = np.isneginf(got) & np.isneginf(ref)
    with np.errstate(invalid="ignore"):  # -inf - -inf where both rows are empty
        d = np.where(both_inf, 0.0, np.abs(got - ref))
    bound = LSE_REL * np.maximum(1.0, np.abs(np.where(both_inf, 0.0, ref)))
    bad = ~(d <= bound)
    assert not bad.any(), f"lse mismatch at {np.argwhere(bad)[:5].tolist()}: max {np.nanmax(d):.3e}"


def check_topk_tie_rule(gpu_idx, scores, topk, rel=1e-6):
    """GPU top-k sets against oracle fp64 scores with the tie band of the
    spec: with tau the k-th largest exact score and delta = rel * max|s|, a
    GPU set passes iff it has k distinct entries, contains every j with
    s_j > tau + delta, and holds only j with s_j >= tau - delta.
    Returns (rows checked, rows whose set differs from the exact top-k)."""
    B, H, N, k = gpu_idx.shape
    assert k == topk
    differ = 0
    for r in np.ndindex(B, H, N):
        g = gpu_idx[r]
        assert len(set(g.tolist())) == k, f"duplicate entries in row {r}"
        assert ((g >= 0) & (g < N)).all()
        s = scores[r]
        order = np.argsort(-s, kind="stable")
        tau = s[order[k - 1]]
        delta = rel * np.abs(s).max()
        must = set(np.nonzero(s > tau + delta)[0].tolist())
        assert must <= set(g.tolist()), f"row {r}: missing a clearly selected cube"
        assert (s[g] >= tau - delta).all(), f"row {r}: selected a clearly unselected cube"
        if set(g.tolist()) != set(order[:k].tolist()):
            differ += 1
    return B * H * N, differ
