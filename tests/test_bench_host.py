"""Host-side accounting of bench.py, checked on the CPU: the tensor-core work
the paired fine kernel issues for a selection (the union walk), against a
count over explicit Python sets."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def union_walk_flops(idx, pairs, D):
    total = 0
    B, H, N, k = idx.shape
    for b in range(B):
        for h in range(H):
            for e in pairs[b, h].tolist():
                e &= 0xFFFFFFFF
                i, j = e & 0xFFFF, e >> 16
                u = set(idx[b, h, i].tolist()) if i < N else set()
                if j < N:
                    u |= set(idx[b, h, j].tolist())
                steps = (len(u) + 1) // 2
                total += steps * 2 * 128 * 128 * D + len(u) * 2 * 128 * 64 * D
    return total


@pytest.mark.parametrize("B,H,N,k,D", [(1, 2, 5, 2, 64), (2, 3, 9, 4, 128), (1, 1, 1, 1, 128)])
def test_executed_tensor_flops_matches_set_count(B, H, N, k, D):
    rng = np.random.default_rng(N * 7 + k)
    idx = np.stack([np.stack([np.stack([rng.choice(N, size=k, replace=False) for _ in range(N)])
                              for _ in range(H)]) for _ in range(B)]).astype(np.int32)
    npairs = (N + 1) // 2
    pairs = np.zeros((B, H, npairs), dtype=np.int64)
    for b in range(B):
        for h in range(H):
            perm = rng.permutation(N).tolist()
            units = [(perm[2 * u], perm[2 * u + 1] if 2 * u + 1 < N else 0xFFFF) for u in range(npairs)]
            pairs[b, h] = [i | (j << 16) for i, j in units]
    pairs32 = pairs.astype(np.uint32).view(np.int32)  # as the device holds them (int32, j = 0xFFFF negative)
    assert bench.executed_tensor_flops(idx, pairs32, D) == union_walk_flops(idx, pairs32, D)


def test_selected_share_is_one_for_identical_selections():
    """Both cubes of every pair select the same k cubes (k even): nothing is
    walked beyond the selection, so executed work equals 4 * 64 * k * 64 * D
    per query cube, the effective count."""
    N, k, D = 8, 4, 128
    idx = np.tile(np.arange(k, dtype=np.int32), (1, 1, N, 1))
    pairs = np.array([[[2 * u | ((2 * u + 1) << 16) for u in range(N // 2)]]], dtype=np.int32)
    assert bench.executed_tensor_flops(idx, pairs, D) == 4.0 * 64 * k * 64 * D * N


def test_result_line_keeps_the_contract(monkeypatch, capsys):
    """main() assembles the one JSON line with every key the contract names,
    from a stubbed device run (the GPU legs are measured on the GPU machine)."""
    import json

    def fake_run_ours(args, wl, inputs, rank, world, dist):
        stage = {n: [1.0, 1.2] for n in ["tile_k_pool_qk", "coarse_select", "pair_cubes", "sparse_attn_fwd",
                                         "tile_v"]}
        clocks = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}
        return 2.0, stage, clocks, (None, 0, 0, None), 10, {}, 3.0e11

    monkeypatch.setattr(bench, "run_ours", fake_run_ours)
    monkeypatch.setattr(sys, "argv", ["bench.py", "--heads", "2", "--steps", "2", "--no-cpu-baseline", "--no-e2e"])
    assert bench.main() == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in line, key
    assert line["n_gpus"] == 1 and line["steps"] == 2 and line["warmup"] >= 3 and line["ms_per_step"] == 2.0
    assert line["higher_is_better"] is True and line["scaling"] == "weak" and line["dtype"] == "bf16"
    assert "workload" in line["config"]
    roof = line["roofline"]
    assert set(("bound", "achieved", "peak", "unit", "frac", "traffic")) <= set(roof)
    assert roof["bound"] == "tensor" and roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"])
    assert roof["traffic"] is None  # taken from a 40-head capture: none for another head count
    fk = line["fine_kernel"]
    assert fk["executed_tensor_flops"] == 3.0e11
    assert fk["selected_share_of_executed"] == pytest.approx(bench_flops(line) / 3.0e11)


def bench_flops(line):
    """The line's effective fine-stage FLOPs, back from its rate and time."""
    fk = line["fine_kernel"]
    return fk["effective_tflops"] * 1e12 * fk["ms_per_call_mean"] * 1e-3
