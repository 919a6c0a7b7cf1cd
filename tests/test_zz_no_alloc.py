"""The allocation-free coarse selection (vsa_coarse_select_noalloc).

It serves callers that cannot allocate device memory: it keeps its scratch
in a fixed 64 MiB array inside the library instead of taking a workspace.
This checks, through the C ABI, that two calls in a row give exactly the
indices of vsa_coarse_select on the same inputs (integer output: bit-exact),
and that a problem too large for the array is refused.
"""
import ctypes

import numpy as np
import pytest
import torch

import block_sparse_video_vsa_gb300 as vsa
from block_sparse_video_vsa_gb300 import synth

pytestmark = pytest.mark.gpu

_P = ctypes.c_void_p
_I = ctypes.c_int32


def noalloc_fn():
    lib = vsa.library()
    f = lib.vsa_coarse_select_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, ctypes.c_float, _P, _P]
    return f


def tiled_case(wl):
    d = synth.make_inputs(wl)
    dev = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
    qt, vbs = vsa.tile(dev(d["q"]), wl.grid)
    kt, _ = vsa.tile(dev(d["k"]), wl.grid, vbs=torch.empty_like(vbs))
    return qt, kt, vbs


def test_noalloc_matches_workspace_version_twice():
    f = noalloc_fn()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    cases = [synth.WORKLOADS["mid"],
             synth.Workload("noalloc2", 1, 13, 20, 24, heads=6, D=64, topk=17, seed=404)]
    for wl in cases:  # two calls in a row, different shapes: stale scratch must not matter
        qt, kt, vbs = tiled_case(wl)
        B, S, H, D = qt.shape
        N = S // 64
        ref = vsa.coarse_select(qt, kt, vbs, wl.topk, wl.sm_scale)
        got = torch.full((B, H, N, wl.topk), -7, dtype=torch.int32, device="cuda")
        st = f(qt.data_ptr(), kt.data_ptr(), vbs.data_ptr(), B, N, H, D, wl.topk, wl.sm_scale,
               got.data_ptr(), stream)
        assert st == 0, vsa.library().vsa_status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(got, ref)


def test_noalloc_refuses_problems_beyond_the_scratch():
    f = noalloc_fn()
    A = 0x10000  # never dereferenced: the size check fails first
    # 16 * 1 * 40 * 4096 * 128 bytes = 320 MiB > 64 MiB
    assert f(A, A, A, 1, 4096, 40, 128, 8, 0.0, A, None) == 2  # VSA_ERR_UNSUPPORTED


def test_noalloc_falls_back_to_the_fused_kernel_when_the_scores_do_not_fit():
    # 300 cubes, 80 heads, D = 128: with the score matrix the scratch would need
    # 78 MB (> 64 MiB), without it 49 MB.  The allocation-free call then takes
    # the fused kernel; both paths select the exact top-k, so the indices match
    # those of the workspace version (which keeps the scores in memory).
    f = noalloc_fn()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    B, N, H, D, k = 1, 300, 80, 128, 37
    g = torch.Generator(device="cuda").manual_seed(5)
    qt = torch.randn((B, 64 * N, H, D), generator=g, device="cuda").to(torch.bfloat16)
    kt = torch.randn((B, 64 * N, H, D), generator=g, device="cuda").to(torch.bfloat16)
    vbs = torch.full((N,), 64, dtype=torch.int32, device="cuda")
    vbs[::7] = 16
    assert vsa.coarse_workspace_bytes(B, H, N, D) > (64 << 20)
    ref = vsa.coarse_select(qt, kt, vbs, k)
    got = torch.full((B, H, N, k), -7, dtype=torch.int32, device="cuda")
    st = f(qt.data_ptr(), kt.data_ptr(), vbs.data_ptr(), B, N, H, D, k, 0.0, got.data_ptr(), stream)
    assert st == 0, vsa.library().vsa_status_string(st)
    torch.cuda.synchronize()
    assert torch.equal(got, ref)
