"""GB300-native Video Sparse Attention (VSA) hot path.

Python binding of ``libvsa.so`` (C ABI declared in ``include/vsa.h``).  Every
function here only marshals arguments: it checks tensor placement, dtype and
shape, allocates outputs with PyTorch, and calls the C entry point of the same
name on the current CUDA stream.  All computation runs in the library's
sm_103a kernels; there is no CPU fallback, and a missing library raises.

    xt, vbs  = tile(x, grid)                       # raster -> cube-major
    topk_idx = coarse_select(qt, kt, vbs, topk)    # mean-pool + score + top-k
    o, lse   = sparse_attn_fwd(qt, kt, vt, topk_idx, vbs)
    y        = untile(o, grid)                     # cube-major -> raster
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional, Sequence, Tuple

from .build import LIB_PATH

__all__ = [
    "VsaError", "library", "num_cubes", "tile", "untile", "coarse_workspace_bytes", "coarse_select",
    "sparse_attn_fwd", "validate_indices", "device_error", "debug_wait_timeout", "pipeline",
    "coarse_attn", "coarse_attn_workspace_bytes", "pair_cubes", "pair_workspace_bytes", "kernel_launches",
    "table_from_csr", "block_select", "block_select_workspace_bytes", "sparse_attn_fwd_peak", "all_cubes",
    "PipelineGraph",
]

_STATUS = {0: "VSA_OK", 1: "VSA_ERR_INVALID_ARG", 2: "VSA_ERR_UNSUPPORTED", 3: "VSA_ERR_ALIGNMENT",
           4: "VSA_ERR_INDEX_RANGE", 5: "VSA_ERR_TIMEOUT", 6: "VSA_ERR_CUDA"}


class VsaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {_STATUS.get(status, status)}")
        self.status = status


class VsaGrid(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("H", ctypes.c_int32),
                ("W", ctypes.c_int32), ("heads", ctypes.c_int32), ("D", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None
_p = ctypes.c_void_p
_i32 = ctypes.c_int32


def _declare(lib):
    lib.vsa_status_string.restype = ctypes.c_char_p
    lib.vsa_status_string.argtypes = [ctypes.c_int]
    lib.vsa_num_cubes.restype = ctypes.c_int64
    lib.vsa_num_cubes.argtypes = [ctypes.POINTER(VsaGrid)]
    lib.vsa_tile.restype = ctypes.c_int
    lib.vsa_tile.argtypes = [ctypes.POINTER(VsaGrid), _p, _p, _p, _p]
    lib.vsa_untile.restype = ctypes.c_int
    lib.vsa_untile.argtypes = [ctypes.POINTER(VsaGrid), _p, _p, _p]
    lib.vsa_coarse_workspace_bytes.restype = ctypes.c_size_t
    lib.vsa_coarse_workspace_bytes.argtypes = [_i32] * 4
    lib.vsa_coarse_select.restype = ctypes.c_int
    lib.vsa_coarse_select.argtypes = [_p, _p, _p, _i32, _i32, _i32, _i32, _i32, ctypes.c_float, _p, _p, _p]
    lib.vsa_tile_pool.restype = ctypes.c_int
    lib.vsa_tile_pool.argtypes = [ctypes.POINTER(VsaGrid), _p, _p, _p, _p, _p, _p, _p]
    lib.vsa_coarse_select_pooled.restype = ctypes.c_int
    lib.vsa_coarse_select_pooled.argtypes = [_p, _i32, _i32, _i32, _i32, _i32, ctypes.c_float, _p, _p, _p]
    lib.vsa_sparse_attn_fwd_raster.restype = ctypes.c_int
    lib.vsa_sparse_attn_fwd_raster.argtypes = [ctypes.POINTER(VsaGrid), _p, _p, _p, _p, _p, _p, _p, _i32,
                                               ctypes.c_float, _p, _p, _p]
    lib.vsa_sparse_attn_fwd.restype = ctypes.c_int
    lib.vsa_sparse_attn_fwd.argtypes = [_p, _p, _p, _p, _p, _i32, _i32, _i32, _i32, _i32, ctypes.c_float,
                                        _p, _p, _p]
    lib.vsa_sparse_attn_fwd_ex.restype = ctypes.c_int
    lib.vsa_sparse_attn_fwd_ex.argtypes = [_p, _p, _p, _p, _p, _p, _p, _i32, _i32, _i32, _i32, _i32,
                                           ctypes.c_float, _p, _p, _p]
    lib.vsa_sparse_attn_fwd_paired.restype = ctypes.c_int
    lib.vsa_sparse_attn_fwd_paired.argtypes = [_p, _p, _p, _p, _p, _p, _i32, _i32, _i32, _i32, _i32,
                                               ctypes.c_float, _p, _p, _p]
    lib.vsa_pair_workspace_bytes.restype = ctypes.c_size_t
    lib.vsa_pair_workspace_bytes.argtypes = [_i32] * 4
    lib.vsa_pair_cubes.restype = ctypes.c_int
    lib.vsa_pair_cubes.argtypes = [_p, _i32, _i32, _i32, _i32, _p, _p, _p]
    lib.vsa_validate_indices.restype = ctypes.c_int
    lib.vsa_validate_indices.argtypes = [_p, _p, _i32, _i32, _i32, _i32, _p, _p]
    lib.vsa_validate_indices_ex.restype = ctypes.c_int
    lib.vsa_validate_indices_ex.argtypes = [_p, _p, _p, _i32, _i32, _i32, _i32, _p, _p]
    lib.vsa_device_error.restype = ctypes.c_int
    lib.vsa_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), _i32]
    lib.vsa_debug_wait_timeout.restype = ctypes.c_int
    lib.vsa_debug_wait_timeout.argtypes = [ctypes.c_int64, _p, _p]
    lib.vsa_sparse_attn_fwd_gated.restype = ctypes.c_int
    lib.vsa_sparse_attn_fwd_gated.argtypes = [_p, _p, _p, _p, _p, _p, _p, _i32, _i32, _i32, _i32, _i32,
                                              ctypes.c_float, _p, _p, _p, _p, _p, _p]
    lib.vsa_sparse_attn_fwd_peak.restype = ctypes.c_int
    lib.vsa_sparse_attn_fwd_peak.argtypes = [_p, _p, _p, _p, _p, _p, _p, _i32, _i32, _i32, _i32, _i32,
                                             ctypes.c_float, _p, _p, _p, _p]
    lib.vsa_coarse_attn_workspace_bytes.restype = ctypes.c_size_t
    lib.vsa_coarse_attn_workspace_bytes.argtypes = [_i32] * 4
    lib.vsa_coarse_attn.restype = ctypes.c_int
    lib.vsa_coarse_attn.argtypes = [_p, _p, _p, _p, _i32, _i32, _i32, _i32, ctypes.c_float, _p, _p, _p]
    lib.vsa_table_from_csr.restype = ctypes.c_int
    lib.vsa_table_from_csr.argtypes = [_p, _p, ctypes.c_int64, ctypes.c_int64, _i32, _i32, _p, _p]
    lib.vsa_block_select_workspace_bytes.restype = ctypes.c_size_t
    lib.vsa_block_select_workspace_bytes.argtypes = [_i32] * 4
    lib.vsa_block_select.restype = ctypes.c_int
    lib.vsa_block_select.argtypes = [_p, _p, _i32, _i32, _i32, _i32, ctypes.c_float, ctypes.c_float, _p, _p, _p, _p]
    lib.vsa_kernel_launches.restype = ctypes.c_uint64
    lib.vsa_kernel_launches.argtypes = []
    return lib


def library():
    """The loaded libvsa.so (ctypes).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libvsa.so not found at {LIB_PATH}; build it first "
                    "(python -m block_sparse_video_vsa_gb300.build)")
            _lib = _declare(ctypes.CDLL(LIB_PATH))
    return _lib


def _check(status: int, what: str):
    if status != 0:
        raise VsaError(status, what)


def _torch():
    import torch
    return torch


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, dtype, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _grid(grid, heads: int, D: int) -> VsaGrid:
    B, T, H, W = (int(v) for v in grid)
    return VsaGrid(B, T, H, W, int(heads), int(D))


def num_cubes(grid: Sequence[int]) -> int:
    """Cubes covering a (B, T, H, W) grid (vsa_num_cubes)."""
    B, T, H, W = (int(v) for v in grid)
    g = VsaGrid(B, T, H, W, 1, 8)  # heads and D do not enter the count
    n = int(library().vsa_num_cubes(ctypes.byref(g)))
    if n < 0:
        raise ValueError(f"grid sizes must be positive, got {tuple(grid)}")
    return n


def tile(x, grid, out=None, vbs=None, stream=None):
    """Raster [B, T*H*W, heads, D] bf16 -> (cube-major [B, 64*N, heads, D], vbs [N] int32)."""
    torch = _torch()
    _need(x, torch.bfloat16, "x")
    B, S, heads, D = x.shape
    g = _grid(grid, heads, D)
    if (g.B, g.T * g.H * g.W) != (B, S):
        raise ValueError("x shape does not match the grid")
    N = num_cubes(grid)
    if out is None:
        out = torch.empty((B, 64 * N, heads, D), dtype=torch.bfloat16, device=x.device)
    if vbs is None:
        vbs = torch.empty((N,), dtype=torch.int32, device=x.device)
    _need(out, torch.bfloat16, "out")
    _need(vbs, torch.int32, "vbs")
    _check(library().vsa_tile(ctypes.byref(g), x.data_ptr(), out.data_ptr(), vbs.data_ptr(), _stream(stream)),
           "vsa_tile")
    return out, vbs


def untile(yt, grid, out=None, stream=None):
    """Cube-major [B, 64*N, heads, D] bf16 -> raster [B, T*H*W, heads, D]."""
    torch = _torch()
    _need(yt, torch.bfloat16, "yt")
    B, S, heads, D = yt.shape
    g = _grid(grid, heads, D)
    if S != 64 * num_cubes(grid) or B != g.B:
        raise ValueError("yt shape does not match the grid")
    if out is None:
        out = torch.empty((B, g.T * g.H * g.W, heads, D), dtype=torch.bfloat16, device=yt.device)
    _need(out, torch.bfloat16, "out")
    _check(library().vsa_untile(ctypes.byref(g), yt.data_ptr(), out.data_ptr(), _stream(stream)), "vsa_untile")
    return out


def coarse_workspace_bytes(B: int, heads: int, ncubes: int, D: int) -> int:
    return int(library().vsa_coarse_workspace_bytes(B, heads, ncubes, D))


def coarse_select(qt, kt, vbs, topk: int, sm_scale: float = 0.0, workspace=None, out=None, stream=None):
    """Top-k key cubes per query cube -> int32 [B, heads, N, topk] (ascending cube ids)."""
    torch = _torch()
    _need(qt, torch.bfloat16, "qt")
    _need(kt, torch.bfloat16, "kt")
    _need(vbs, torch.int32, "vbs")
    B, S, heads, D = qt.shape
    if kt.shape != qt.shape or S % 64:
        raise ValueError("qt/kt must share a tiled [B, 64*N, heads, D] shape")
    N = S // 64
    nbytes = coarse_workspace_bytes(B, heads, N, D)
    if workspace is None:
        workspace = torch.empty((max(nbytes, 16),), dtype=torch.uint8, device=qt.device)
    _need(workspace, torch.uint8, "workspace")
    if workspace.numel() < nbytes:
        raise ValueError(f"workspace needs {nbytes} bytes")
    if out is None:
        out = torch.empty((B, heads, N, int(topk)), dtype=torch.int32, device=qt.device)
    _need(out, torch.int32, "out")
    _check(library().vsa_coarse_select(qt.data_ptr(), kt.data_ptr(), vbs.data_ptr(), B, N, heads, D, int(topk),
                                       float(sm_scale), workspace.data_ptr(), out.data_ptr(), _stream(stream)),
           "vsa_coarse_select")
    return out


def tile_pool(q, k, grid, qt=None, kt=None, vbs=None, workspace=None, want_qt=True, want_kt=True, stream=None):
    """Tile q and k and pool their cubes in one pass (vsa_tile_pool).

    Returns (qt, kt, vbs, workspace); pass vbs and workspace to
    coarse_select_pooled for the same top-k as coarse_select(qt, kt, vbs, ...).
    want_qt=False skips the tiled copy of q (qt is then None), for
    sparse_attn_fwd_raster, which reads the raster q; want_kt=False likewise
    skips the tiled copy of k (kt is then None: the statistics alone)."""
    torch = _torch()
    _need(q, torch.bfloat16, "q")
    _need(k, torch.bfloat16, "k")
    if k.shape != q.shape:
        raise ValueError("q and k must share a [B, T*H*W, heads, D] shape")
    B, S, heads, D = q.shape
    g = _grid(grid, heads, D)
    if (g.B, g.T * g.H * g.W) != (B, S):
        raise ValueError("q shape does not match the grid")
    N = num_cubes(grid)
    shape = (B, 64 * N, heads, D)
    if qt is None and want_qt:
        qt = torch.empty(shape, dtype=torch.bfloat16, device=q.device)
    if kt is None and want_kt:
        kt = torch.empty(shape, dtype=torch.bfloat16, device=q.device)
    if vbs is None:
        vbs = torch.empty((N,), dtype=torch.int32, device=q.device)
    nbytes = coarse_workspace_bytes(B, heads, N, D)
    if workspace is None:
        workspace = torch.empty((max(nbytes, 16),), dtype=torch.uint8, device=q.device)
    for t, n in ((qt, "qt"), (kt, "kt")):
        if t is None:
            continue
        _need(t, torch.bfloat16, n)
        if tuple(t.shape) != shape:
            raise ValueError(f"{n} must be {shape}")
    _need(vbs, torch.int32, "vbs")
    _need(workspace, torch.uint8, "workspace")
    if workspace.numel() < nbytes:
        raise ValueError(f"workspace needs {nbytes} bytes")
    _check(library().vsa_tile_pool(ctypes.byref(g), q.data_ptr(), k.data_ptr(), None if qt is None else qt.data_ptr(),
                                   None if kt is None else kt.data_ptr(), vbs.data_ptr(), workspace.data_ptr(),
                                   _stream(stream)), "vsa_tile_pool")
    return qt, kt, vbs, workspace


def coarse_select_pooled(workspace, vbs, B: int, heads: int, D: int, topk: int, sm_scale: float = 0.0, out=None,
                         stream=None):
    """Top-k key cubes per query cube from the statistics tile_pool wrote
    -> int32 [B, heads, N, topk] (N = vbs.numel())."""
    torch = _torch()
    _need(vbs, torch.int32, "vbs")
    _need(workspace, torch.uint8, "workspace")
    N = vbs.numel()
    nbytes = coarse_workspace_bytes(B, heads, N, D)
    if workspace.numel() < nbytes:
        raise ValueError(f"workspace needs {nbytes} bytes")
    if out is None:
        out = torch.empty((B, heads, N, int(topk)), dtype=torch.int32, device=vbs.device)
    _need(out, torch.int32, "out")
    if tuple(out.shape) != (B, heads, N, int(topk)):
        raise ValueError("out must be [B, heads, N, topk]")
    _check(library().vsa_coarse_select_pooled(vbs.data_ptr(), int(B), N, int(heads), int(D), int(topk),
                                              float(sm_scale), workspace.data_ptr(), out.data_ptr(),
                                              _stream(stream)), "vsa_coarse_select_pooled")
    return out


def pair_workspace_bytes(B: int, heads: int, ncubes: int, topk: int) -> int:
    return int(library().vsa_pair_workspace_bytes(B, heads, ncubes, topk))


def pair_cubes(topk_idx, workspace=None, out=None, stream=None):
    """Query-cube pairing for the fine stage -> int32 [B, heads, (N + 1) // 2].

    Each entry holds the uint32 bit pattern i | (j << 16) (j = 0xFFFF: single
    cube); see vsa_pair_cubes."""
    torch = _torch()
    _need(topk_idx, torch.int32, "topk_idx")
    if topk_idx.dim() != 4:
        raise ValueError("topk_idx must be [B, heads, N, topk]")
    B, heads, N, topk = topk_idx.shape
    nbytes = pair_workspace_bytes(B, heads, N, topk)
    if workspace is None:
        workspace = torch.empty((max(nbytes, 16),), dtype=torch.uint8, device=topk_idx.device)
    _need(workspace, torch.uint8, "workspace")
    if workspace.numel() < nbytes:
        raise ValueError(f"workspace needs {nbytes} bytes")
    if out is None:
        out = torch.empty((B, heads, (N + 1) // 2), dtype=torch.int32, device=topk_idx.device)
    _need(out, torch.int32, "out")
    if tuple(out.shape) != (B, heads, (N + 1) // 2):
        raise ValueError("out must be [B, heads, (N + 1) // 2]")
    _check(library().vsa_pair_cubes(topk_idx.data_ptr(), B, N, heads, topk, workspace.data_ptr(),
                                    out.data_ptr(), _stream(stream)), "vsa_pair_cubes")
    return out


def sparse_attn_fwd(qt, kt, vt, topk_idx, vbs, sm_scale: float = 0.0, out=None, lse=None,
                    want_lse: bool = True, pairs=None, counts=None, coarse_out=None, gate_c=None, gate_f=None,
                    stream=None):
    """Block-sparse attention -> (out bf16 [B, 64*N, heads, D], lse fp32 [B, heads, 64*N] or None).

    `pairs` (from pair_cubes) sets which query cubes share a tile; None pairs
    cubes (2u, 2u + 1).  The results do not depend on it beyond rounding.
    `counts` (int32 [B, heads, N]) limits row i to its first counts[i] entries.
    With `coarse_out` (fp32 [B, heads, N, D], from coarse_attn) and the bf16
    gates `gate_c`, `gate_f` (shaped like out), out is the gated sum
    gate_c * coarse + gate_f * fine."""
    torch = _torch()
    for t, n in ((qt, "qt"), (kt, "kt"), (vt, "vt")):
        _need(t, torch.bfloat16, n)
    _need(topk_idx, torch.int32, "topk_idx")
    _need(vbs, torch.int32, "vbs")
    B, S, heads, D = qt.shape
    if kt.shape != qt.shape or vt.shape != qt.shape or S % 64:
        raise ValueError("qt/kt/vt must share a tiled [B, 64*N, heads, D] shape")
    N = S // 64
    if topk_idx.dim() != 4 or tuple(topk_idx.shape[:3]) != (B, heads, N):
        raise ValueError("topk_idx must be [B, heads, N, topk]")
    topk = topk_idx.shape[3]
    if out is None:
        out = torch.empty_like(qt)
    _need(out, torch.bfloat16, "out")
    if want_lse and lse is None:
        lse = torch.empty((B, heads, S), dtype=torch.float32, device=qt.device)
    if lse is not None:
        _need(lse, torch.float32, "lse")
    if pairs is not None:
        _need(pairs, torch.int32, "pairs")
        if tuple(pairs.shape) != (B, heads, (N + 1) // 2):
            raise ValueError("pairs must be [B, heads, (N + 1) // 2]")
    if counts is not None:
        _need(counts, torch.int32, "counts")
        if tuple(counts.shape) != (B, heads, N):
            raise ValueError("counts must be [B, heads, N]")
    gated = [coarse_out, gate_c, gate_f]
    if any(t is not None for t in gated):
        if any(t is None for t in gated):
            raise ValueError("coarse_out, gate_c and gate_f go together")
        _need(coarse_out, torch.float32, "coarse_out")
        _need(gate_c, torch.bfloat16, "gate_c")
        _need(gate_f, torch.bfloat16, "gate_f")
        if tuple(coarse_out.shape) != (B, heads, N, D) or gate_c.shape != qt.shape or gate_f.shape != qt.shape:
            raise ValueError("coarse_out must be [B, heads, N, D] and the gates shaped like qt")
    ptr = lambda t: t.data_ptr() if t is not None else None  # noqa: E731
    _check(library().vsa_sparse_attn_fwd_gated(qt.data_ptr(), kt.data_ptr(), vt.data_ptr(), topk_idx.data_ptr(),
                                               ptr(counts), vbs.data_ptr(), ptr(pairs), B, N, heads, D, topk,
                                               float(sm_scale), ptr(coarse_out), ptr(gate_c), ptr(gate_f),
                                               out.data_ptr(), ptr(lse), _stream(stream)),
           "vsa_sparse_attn_fwd")
    return out, lse


def sparse_attn_fwd_raster(q, kt, vt, topk_idx, vbs, grid, sm_scale: float = 0.0, out=None, lse=None,
                           want_lse: bool = True, pairs=None, counts=None, stream=None):
    """Block-sparse attention on raster q -> (out raster bf16 [B, T*H*W, heads, D],
    lse fp32 [B, heads, 64*N] cube-major or None); kt, vt tiled
    (vsa_sparse_attn_fwd_raster).  out equals untile(sparse_attn_fwd(tile(q), ...))."""
    torch = _torch()
    _need(q, torch.bfloat16, "q")
    _need(kt, torch.bfloat16, "kt")
    _need(vt, torch.bfloat16, "vt")
    _need(topk_idx, torch.int32, "topk_idx")
    _need(vbs, torch.int32, "vbs")
    B, S, heads, D = q.shape
    g = _grid(grid, heads, D)
    N = num_cubes(grid)
    if (g.B, g.T * g.H * g.W) != (B, S):
        raise ValueError("q shape does not match the grid")
    if tuple(kt.shape) != (B, 64 * N, heads, D) or vt.shape != kt.shape:
        raise ValueError("kt/vt must be tiled [B, 64*N, heads, D] of the grid")
    if topk_idx.dim() != 4 or tuple(topk_idx.shape[:3]) != (B, heads, N):
        raise ValueError("topk_idx must be [B, heads, N, topk]")
    topk = topk_idx.shape[3]
    if out is None:
        out = torch.empty_like(q)
    _need(out, torch.bfloat16, "out")
    if out.shape != q.shape:
        raise ValueError("out must match q")
    if want_lse and lse is None:
        lse = torch.empty((B, heads, 64 * N), dtype=torch.float32, device=q.device)
    if lse is not None:
        _need(lse, torch.float32, "lse")
        if tuple(lse.shape) != (B, heads, 64 * N):
            raise ValueError("lse must be [B, heads, 64*N]")
    if pairs is not None:
        _need(pairs, torch.int32, "pairs")
        if tuple(pairs.shape) != (B, heads, (N + 1) // 2):
            raise ValueError("pairs must be [B, heads, (N + 1) // 2]")
    if counts is not None:
        _need(counts, torch.int32, "counts")
        if tuple(counts.shape) != (B, heads, N):
            raise ValueError("counts must be [B, heads, N]")
    _check(library().vsa_sparse_attn_fwd_raster(
        ctypes.byref(g), q.data_ptr(), kt.data_ptr(), vt.data_ptr(), topk_idx.data_ptr(),
        None if counts is None else counts.data_ptr(), vbs.data_ptr(),
        None if pairs is None else pairs.data_ptr(), int(topk), float(sm_scale), out.data_ptr(),
        None if lse is None else lse.data_ptr(), _stream(stream)), "vsa_sparse_attn_fwd_raster")
    return out, lse


def block_select_workspace_bytes(B: int, S: int, heads: int, D: int) -> int:
    return int(library().vsa_block_select_workspace_bytes(B, S, heads, D))


def block_select(q, k, tau: float, sm_scale: float = 0.0, workspace=None, out=None, counts=None, stream=None):
    """Mean-pool block selector with a cumulative threshold on a token sequence
    q, k bf16 [B, S, heads, D] (S a multiple of 128) -> (cube table int32
    [B, heads, S / 64, S / 64], counts int32 [B, heads, S / 64]) for
    sparse_attn_fwd(..., counts=counts) with the default pairing."""
    torch = _torch()
    _need(q, torch.bfloat16, "q")
    _need(k, torch.bfloat16, "k")
    B, S, heads, D = q.shape
    if k.shape != q.shape or S % 128:
        raise ValueError("q and k must share a [B, S, heads, D] shape with S a multiple of 128")
    nbytes = block_select_workspace_bytes(B, S, heads, D)
    if workspace is None:
        workspace = torch.empty((max(nbytes, 16),), dtype=torch.uint8, device=q.device)
    _need(workspace, torch.uint8, "workspace")
    if workspace.numel() < nbytes:
        raise ValueError(f"workspace needs {nbytes} bytes")
    nc = S // 64
    if out is None:
        out = torch.empty((B, heads, nc, nc), dtype=torch.int32, device=q.device)
    if counts is None:
        counts = torch.empty((B, heads, nc), dtype=torch.int32, device=q.device)
    _need(out, torch.int32, "out")
    _need(counts, torch.int32, "counts")
    if tuple(out.shape) != (B, heads, nc, nc) or tuple(counts.shape) != (B, heads, nc):
        raise ValueError("out must be [B, heads, S / 64, S / 64] and counts [B, heads, S / 64]")
    _check(library().vsa_block_select(q.data_ptr(), k.data_ptr(), B, S, heads, D, float(tau), float(sm_scale),
                                      workspace.data_ptr(), out.data_ptr(), counts.data_ptr(), _stream(stream)),
           "vsa_block_select")
    return out, counts


def sparse_attn_fwd_peak(qt, kt, vt, topk_idx, vbs, sm_scale: float = 0.0, out=None, lse=None, max_prob=None,
                         pairs=None, counts=None, stream=None):
    """sparse_attn_fwd that also returns each row's largest softmax weight
    (vsa_sparse_attn_fwd_peak) -> (out, lse, max_prob fp32 [B, heads, 64*N])."""
    torch = _torch()
    for t, n in ((qt, "qt"), (kt, "kt"), (vt, "vt")):
        _need(t, torch.bfloat16, n)
    _need(topk_idx, torch.int32, "topk_idx")
    _need(vbs, torch.int32, "vbs")
    B, S, heads, D = qt.shape
    if kt.shape != qt.shape or vt.shape != qt.shape or S % 64:
        raise ValueError("qt/kt/vt must share a tiled [B, 64*N, heads, D] shape")
    N = S // 64
    if topk_idx.dim() != 4 or tuple(topk_idx.shape[:3]) != (B, heads, N):
        raise ValueError("topk_idx must be [B, heads, N, topk]")
    out = torch.empty_like(qt) if out is None else out
    lse = torch.empty((B, heads, S), dtype=torch.float32, device=qt.device) if lse is None else lse
    max_prob = torch.empty((B, heads, S), dtype=torch.float32, device=qt.device) if max_prob is None else max_prob
    _need(out, torch.bfloat16, "out")
    _need(lse, torch.float32, "lse")
    _need(max_prob, torch.float32, "max_prob")
    if pairs is not None:
        _need(pairs, torch.int32, "pairs")
        if tuple(pairs.shape) != (B, heads, (N + 1) // 2):
            raise ValueError("pairs must be [B, heads, (N + 1) // 2]")
    if counts is not None:
        _need(counts, torch.int32, "counts")
        if tuple(counts.shape) != (B, heads, N):
            raise ValueError("counts must be [B, heads, N]")
    ptr = lambda t: t.data_ptr() if t is not None else None  # noqa: E731
    _check(library().vsa_sparse_attn_fwd_peak(qt.data_ptr(), kt.data_ptr(), vt.data_ptr(), topk_idx.data_ptr(),
                                              ptr(counts), vbs.data_ptr(), ptr(pairs), B, N, heads, D,
                                              topk_idx.shape[3], float(sm_scale), out.data_ptr(), lse.data_ptr(),
                                              max_prob.data_ptr(), _stream(stream)), "vsa_sparse_attn_fwd_peak")
    return out, lse, max_prob


def all_cubes(B: int, heads: int, ncubes: int, device=None):
    """The dense selection: every cube for every query cube, int32 [B, heads, N, N]."""
    torch = _torch()
    row = torch.arange(ncubes, dtype=torch.int32, device=device)
    return row.expand(B, heads, ncubes, ncubes).contiguous()


def coarse_attn_workspace_bytes(B: int, heads: int, ncubes: int, D: int) -> int:
    return int(library().vsa_coarse_attn_workspace_bytes(B, heads, ncubes, D))


def coarse_attn(qt, kt, vt, vbs, sm_scale: float = 0.0, workspace=None, out=None, stream=None):
    """Coarse-stage attention over the mean-pooled cubes -> fp32 [B, heads, N, D]."""
    torch = _torch()
    for t, n in ((qt, "qt"), (kt, "kt"), (vt, "vt")):
        _need(t, torch.bfloat16, n)
    _need(vbs, torch.int32, "vbs")
    B, S, heads, D = qt.shape
    if kt.shape != qt.shape or vt.shape != qt.shape or S % 64:
        raise ValueError("qt/kt/vt must share a tiled [B, 64*N, heads, D] shape")
    N = S // 64
    if workspace is None:
        workspace = torch.empty((coarse_attn_workspace_bytes(B, heads, N, D),), dtype=torch.uint8,
                                device=qt.device)
    if out is None:
        out = torch.empty((B, heads, N, D), dtype=torch.float32, device=qt.device)
    _need(out, torch.float32, "out")
    _check(library().vsa_coarse_attn(qt.data_ptr(), kt.data_ptr(), vt.data_ptr(), vbs.data_ptr(), B, N, heads, D,
                                     float(sm_scale), workspace.data_ptr(), out.data_ptr(), _stream(stream)),
           "vsa_coarse_attn")
    return out


def validate_indices(topk_idx, vbs, counts=None, stream=None) -> int:
    """Runs the index validator; returns its flag (0 = valid).  Synchronises.

    With `counts` (int32 [B, heads, N]) only each row's first counts entries
    are checked (vsa_validate_indices_ex)."""
    torch = _torch()
    _need(topk_idx, torch.int32, "topk_idx")
    _need(vbs, torch.int32, "vbs")
    B, heads, N, topk = topk_idx.shape
    if counts is not None:
        _need(counts, torch.int32, "counts")
        if tuple(counts.shape) != (B, heads, N):
            raise ValueError("counts must be [B, heads, N]")
    flag = torch.zeros((1,), dtype=torch.int32, device=topk_idx.device)
    _check(library().vsa_validate_indices_ex(topk_idx.data_ptr(), counts.data_ptr() if counts is not None else None,
                                             vbs.data_ptr(), B, heads, N, topk, flag.data_ptr(), _stream(stream)),
           "vsa_validate_indices_ex")
    return int(flag.item())


def table_from_csr(lut_ptr, kv_idx, width: int, ncubes: int, shape=None):
    """Host-side: a compressed-row block table (int64 offsets `lut_ptr`
    [rows + 1], int32 indices `kv_idx`, each in [0, ncubes)) -> (table int32
    [rows, width] with -1 after each row's entries, counts int32 [rows]), as
    numpy arrays; `shape` (B, heads, ncubes) reshapes them for
    sparse_attn_fwd(..., counts=...)."""
    import numpy as np
    lut_ptr = np.ascontiguousarray(lut_ptr, dtype=np.int64)
    kv_idx = np.ascontiguousarray(kv_idx, dtype=np.int32)
    if lut_ptr.ndim != 1 or lut_ptr.shape[0] < 2:
        raise ValueError("lut_ptr must be 1-D with rows + 1 >= 2 entries")
    if kv_idx.ndim != 1 or kv_idx.size < lut_ptr[-1]:
        raise ValueError(f"kv_idx holds {kv_idx.size} entries, lut_ptr[-1] needs {int(lut_ptr[-1])}")
    rows = lut_ptr.shape[0] - 1
    table = np.empty((rows, width), np.int32)
    counts = np.empty((rows,), np.int32)
    _check(library().vsa_table_from_csr(lut_ptr.ctypes.data, kv_idx.ctypes.data if kv_idx.size else None,
                                        kv_idx.size, rows, int(width), int(ncubes), table.ctypes.data,
                                        counts.ctypes.data), "vsa_table_from_csr")
    if shape is not None:
        table = table.reshape(tuple(shape) + (width,))
        counts = counts.reshape(tuple(shape))
    return table, counts


def kernel_launches() -> int:
    """Kernels the library has launched in this process so far (host counter)."""
    return int(library().vsa_kernel_launches())


def device_error(reset: bool = False) -> int:
    v = ctypes.c_uint32(0)
    _check(library().vsa_device_error(ctypes.byref(v), 1 if reset else 0), "vsa_device_error")
    return int(v.value)


def debug_wait_timeout(limit_ns: int, stream=None) -> int:
    """Runs the bounded-wait self test; returns 1 if the wait ran out."""
    torch = _torch()
    res = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    _check(library().vsa_debug_wait_timeout(int(limit_ns), res.data_ptr(), _stream(stream)),
           "vsa_debug_wait_timeout")
    return int(res.item())


def pipeline(q, k, v, grid, topk: int, sm_scale: float = 0.0, stream=None):
    """Whole hot path on raster inputs: tile k (q, k pooled in the same pass) and v -> coarse select ->
    pairing -> sparse attention on raster q, written in raster order (no separate untile).

    Returns (out raster bf16, lse fp32 [B, heads, 64*N] in cube-major order, topk_idx)."""
    _, kt, vbs, ws = tile_pool(q, k, grid, want_qt=False, stream=stream)
    vt, _ = tile(v, grid, vbs=_torch().empty_like(vbs), stream=stream)
    B, _, heads, D = q.shape
    idx = coarse_select_pooled(ws, vbs, B, heads, D, topk, sm_scale, stream=stream)
    pairs = pair_cubes(idx, stream=stream)
    return (*sparse_attn_fwd_raster(q, kt, vt, idx, vbs, grid, sm_scale, pairs=pairs, stream=stream), idx)


class PipelineGraph:
    """pipeline() captured once as a CUDA graph for fixed shapes, then
    replayed: for repeated calls on inputs of one shape (serving), with no
    per-call launch or argument marshalling.

    The graph owns its inputs (copies of q, k, v made at construction) and its
    outputs (out, lse, topk_idx: pipeline()'s return values, overwritten by
    every replay).  Calling it copies any given inputs into the graph's
    buffers on the current stream, replays the graph there and returns the
    output tensors.  The kernels and their arguments (tensor maps included)
    are fixed at capture, so the buffers must not be reallocated."""

    def __init__(self, q, k, v, grid, topk: int, sm_scale: float = 0.0):
        torch = _torch()
        self.q, self.k, self.v = (x.detach().clone() for x in (q, k, v))
        dev = self.q.device
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):  # a first run outside the capture sets kernel attributes, loads modules
            pipeline(self.q, self.k, self.v, grid, topk, sm_scale)
        torch.cuda.current_stream(dev).wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.out, self.lse, self.topk_idx = pipeline(self.q, self.k, self.v, grid, topk, sm_scale)

    def __call__(self, q=None, k=None, v=None):
        for dst, src in ((self.q, q), (self.k, k), (self.v, v)):
            if src is not None:
                if src.shape != dst.shape or src.dtype != dst.dtype:
                    raise ValueError("inputs must keep the shape and dtype the graph was captured with")
                dst.copy_(src)
        self.graph.replay()
        return self.out, self.lse, self.topk_idx
