"""GPU parity of the coarse-stage attention output (vsa_coarse_attn) and of
the gated sum of the two stages (vsa_sparse_attn_fwd_gated) against the fp64
oracle ("VSA: Accelerating Video Diffusion Inference with Sparse Attention on
AMD GPUs", Two-Stage Architecture).

The coarse output is fp32 end to end on the GPU; its tolerance follows from
fp32 rounding (unit u = 2^-24): the pooled means carry <= 64u relative
error, a D-term dot product <= D u |q||k| sm_scale absolute in the logit,
which moves each softmax weight by the same relative amount, so outputs
agree to ~1e-5 relative to their scale; the test allows 1e-4 of max|ref|
and a cosine of 0.99999.  The gated output is bf16 and takes the scoring
rule of the fine stage.
"""
import numpy as np
import pytest
import torch

import block_sparse_video_vsa_gb300 as vsa
import oracle
from block_sparse_video_vsa_gb300 import synth
from gpu_util import (assert_lse_close, assert_scoring_rule, i32_dev, score_outputs, tiled_inputs, to_bits,
                      to_dev)

pytestmark = pytest.mark.gpu

REL = 1e-4
COS = 0.99999


def gpu_coarse_attn(qt, kt, vt, vbs, sm):
    out = vsa.coarse_attn(to_dev(qt), to_dev(kt), to_dev(vt), i32_dev(vbs), sm)
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


def assert_close_f32(got, ref):
    assert np.isfinite(got).all()
    scale = max(np.abs(ref).max(), 1e-30)
    assert np.abs(got - ref).max() <= REL * scale, (np.abs(got - ref).max(), scale)
    a, b = got.ravel(), ref.ravel()
    if np.linalg.norm(b) > 0:
        assert a @ b / (np.linalg.norm(a) * np.linalg.norm(b)) >= COS


def random_gates(shape, seed):
    rng = np.random.default_rng(seed)
    return synth.bf16_bits(rng.random(shape, dtype=np.float32)), synth.bf16_bits(rng.random(shape, dtype=np.float32))


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_coarse_attn_small(name):
    wl = synth.WORKLOADS[name]
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    assert_close_f32(gpu_coarse_attn(qt, kt, vt, vbs, wl.sm_scale), oracle.coarse_attn(qt, kt, vt, vbs, wl.sm_scale))


def test_coarse_attn_batch_two_head_dim_64_and_empty_cubes():
    wl = synth.Workload("b2", 2, 7, 9, 11, heads=3, D=64, topk=5, seed=31, sigma=4.0)
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    vbs = vbs.copy()
    vbs[[0, 5]] = 0  # no real token: no key, zero row
    got = gpu_coarse_attn(qt, kt, vt, vbs, wl.sm_scale)
    ref = oracle.coarse_attn(qt, kt, vt, vbs, wl.sm_scale)
    assert (got[:, :, [0, 5]] == 0).all()
    assert_close_f32(got, ref)


@pytest.mark.parametrize("name", ["wan", "hunyuan"])
def test_coarse_attn_full_size(name):
    wl = synth.WORKLOADS[name]
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    assert_close_f32(gpu_coarse_attn(qt, kt, vt, vbs, wl.sm_scale), oracle.coarse_attn(qt, kt, vt, vbs, wl.sm_scale))


def gated_gpu(qt, kt, vt, idx, vbs, sm, gc, gf, paired=False, counts=None):
    q, k, v = to_dev(qt), to_dev(kt), to_dev(vt)
    vb = i32_dev(vbs)
    idx_d = i32_dev(idx)
    oc = vsa.coarse_attn(q, k, v, vb, sm)
    pairs = vsa.pair_cubes(idx_d) if paired else None
    cnt = None if counts is None else i32_dev(counts)
    o, lse = vsa.sparse_attn_fwd(q, k, v, idx_d, vb, sm, pairs=pairs, counts=cnt, coarse_out=oc,
                                 gate_c=to_dev(gc), gate_f=to_dev(gf))
    torch.cuda.synchronize()
    assert vsa.device_error(reset=True) == 0
    return to_bits(o), lse.cpu().numpy()


@pytest.mark.parametrize("name, paired", [("tiny", False), ("mid", False), ("mid", True)])
def test_gated_output_small(name, paired):
    wl = synth.WORKLOADS[name]
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
    gc, gf = random_gates(qt.shape, 11)
    got, got_lse = gated_gpu(qt, kt, vt, idx, vbs, wl.sm_scale, gc, gf, paired=paired)
    fine, lse = oracle.fine_full(qt, kt, vt, idx, vbs, wl.sm_scale)
    ref = oracle.gated_combine(fine, oracle.coarse_attn(qt, kt, vt, vbs, wl.sm_scale), gc, gf)
    assert_scoring_rule(score_outputs(got, ref))
    assert_lse_close(got_lse, lse)


def test_gated_with_counts_and_empty_rows():
    wl = synth.WORKLOADS["mid"]
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    idx = oracle.coarse(qt, kt, vbs, 9, wl.sm_scale)
    rng = np.random.default_rng(2)
    counts = rng.integers(0, 10, size=idx.shape[:3]).astype(np.int32)
    counts.reshape(-1)[:3] = 0
    gc, gf = random_gates(qt.shape, 12)
    got, _ = gated_gpu(qt, kt, vt, idx, vbs, wl.sm_scale, gc, gf, paired=True, counts=counts)
    fine, _ = oracle.fine_full_counts(qt, kt, vt, idx, counts, vbs, wl.sm_scale)
    ref = oracle.gated_combine(fine, oracle.coarse_attn(qt, kt, vt, vbs, wl.sm_scale), gc, gf)
    assert_scoring_rule(score_outputs(got, ref))


def test_fine_only_gates_reproduce_the_ungated_bits():
    wl = synth.WORKLOADS["mid"]
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
    zero = synth.bf16_bits(np.zeros(qt.shape, np.float32))
    one = synth.bf16_bits(np.ones(qt.shape, np.float32))
    got, got_lse = gated_gpu(qt, kt, vt, idx, vbs, wl.sm_scale, zero, one)
    o, lse = vsa.sparse_attn_fwd(to_dev(qt), to_dev(kt), to_dev(vt), i32_dev(idx), i32_dev(vbs), wl.sm_scale)
    assert np.array_equal(got, to_bits(o)) and np.array_equal(got_lse, lse.cpu().numpy())


def test_gated_wan_full_size_sampled():
    wl = synth.WORKLOADS["wan"]
    _, _, qt, kt, vt, vbs = tiled_inputs(wl)
    idx = oracle.coarse(qt, kt, vbs, wl.topk, wl.sm_scale)
    gc, gf = random_gates(qt.shape, 13)
    got, got_lse = gated_gpu(qt, kt, vt, idx, vbs, wl.sm_scale, gc, gf, paired=True)
    assert np.isfinite(synth.bf16_to_f32(got)).all()
    N = wl.ncubes
    rng = np.random.default_rng(4)
    units = np.unique(rng.integers(0, wl.heads, 48) * N + rng.integers(0, N, 48))
    fine_u, lse_u, _ = oracle.fine(qt, kt, vt, idx, vbs, wl.sm_scale, units)   # [u, 64, D]
    oc = oracle.coarse_attn(qt, kt, vt, vbs, wl.sm_scale)
    h, i = units // N, units % N
    rows = 64 * i[:, None] + np.arange(64)[None, :]
    g = lambda bits: synth.bf16_to_f32(bits[0][rows, h[:, None], :]).astype(np.float64)  # noqa: E731
    ref_u = g(gc) * oc[0, h, i][:, None, :] + g(gf) * fine_u
    got_u = got[0][rows, h[:, None], :]
    stats = score_outputs(got_u[None].transpose(0, 2, 1, 3), ref_u[None].transpose(0, 2, 1, 3), 2)
    assert_scoring_rule(stats)
    assert_lse_close(got_lse[0][h[:, None], rows], lse_u)
