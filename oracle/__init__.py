"""CPU oracle for the VSA hot path -- TEST INFRASTRUCTURE ONLY.

The arithmetic lives in ``vsa_oracle.c`` (plain C, IEEE double); this module
compiles it with gcc on first use and marshals numpy arrays into it.  Only the
test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA path
and imports nothing from it.

Every function takes bf16 data as ``numpy.uint16`` bit patterns, shaped as in
the CUDA path's C ABI: token rows ``[B, S, heads, D]``.

Parity status of each function (what pins it is in ``tests/test_oracle_*.py``):
    num_cubes / tile / untile  -- pinned (worked shape example, brute force,
                                  reshape restatement, inverse identity)
    pool / coarse              -- pinned (closed forms, einsum+argsort
                                  restatement, invariances, hand cases)
    fine                       -- pinned (dense SDPA special case, brute-force
                                  masked matrix, closed forms, invariances)
    fine_counts                -- pinned (reduction to the fixed-length stage,
                                  brute force on truncated rows, empty rows)
    coarse_attn                -- pinned (dense SDPA on the pooled cubes,
                                  closed forms, excluded empty cubes)
    gated_combine              -- pinned (gate values that select one term,
                                  hand-computed broadcast)
    block_pool / block_select_cdf / blocks_to_cube_lut
                               -- pinned (closed forms, brute force over key
                                  subsets, limits of the threshold, dense
                                  attention over the kept blocks' tokens)
    row_peak / captured_mass / rel_l1
                               -- pinned (single key, equal logits, explicit
                                  dense weights summed over the selection,
                                  hand values)
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "vsa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_f64 = ctypes.c_double
_ptr = ctypes.c_void_p


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle shared library with gcc (-O2, no fast-math)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c99", "-D_POSIX_C_SOURCE=200809L", "-fPIC", "-shared",
             "-pthread", src, "-o", tmp, "-lm"],
            check=True,
        )
        os.replace(tmp, out)
    return out


def load_library(path: str):
    lib = ctypes.CDLL(path)
    lib.oracle_num_cubes.restype = _i64
    lib.oracle_num_cubes.argtypes = [_i64, _i64, _i64]
    lib.oracle_tile.restype = None
    lib.oracle_tile.argtypes = [_i64] * 6 + [_ptr, _ptr, _ptr]
    lib.oracle_untile.restype = None
    lib.oracle_untile.argtypes = [_i64] * 6 + [_ptr, _ptr]
    lib.oracle_pool.restype = None
    lib.oracle_pool.argtypes = [_i64] * 4 + [_ptr, _ptr, _ptr]
    lib.oracle_coarse.restype = None
    lib.oracle_coarse.argtypes = [_i64] * 4 + [_ptr, _ptr, _ptr, _i64, _f64, _ptr, _ptr]
    lib.oracle_fine.restype = _i64
    lib.oracle_fine.argtypes = ([_i64] * 4 + [_ptr] * 5 + [_i64, _f64, _ptr, _i64, _ptr, _ptr, _i64])
    lib.oracle_default_threads.restype = _i64
    lib.oracle_default_threads.argtypes = []
    return lib


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


class using_library:
    """Context manager: route every oracle call through another build of the
    oracle source (the tests use it to run the pins against planted mistakes)."""

    def __init__(self, path: str):
        self._new = load_library(path)
        self._old = None

    def __enter__(self):
        global _lib
        lib()
        with _lock:
            self._old, _lib = _lib, self._new
        return self._new

    def __exit__(self, *exc):
        global _lib
        with _lock:
            _lib = self._old
        return False


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, "bf16 data is passed as uint16 bit patterns"
    return a


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def num_cubes(T: int, H: int, W: int) -> int:
    return int(lib().oracle_num_cubes(T, H, W))


def tile(x: np.ndarray, grid):
    """x: [B, T*H*W, heads, D] uint16 -> (xt [B, N*64, heads, D], vbs [N])."""
    B, T, H, W = grid
    x = _u16(x)
    assert x.shape[:2] == (B, T * H * W)
    heads, D = x.shape[2], x.shape[3]
    N = num_cubes(T, H, W)
    xt = np.empty((B, N * 64, heads, D), np.uint16)
    vbs = np.empty((N,), np.int32)
    lib().oracle_tile(B, T, H, W, heads, D, _p(x), _p(xt), _p(vbs))
    return xt, vbs


def untile(yt: np.ndarray, grid) -> np.ndarray:
    B, T, H, W = grid
    yt = _u16(yt)
    heads, D = yt.shape[2], yt.shape[3]
    N = num_cubes(T, H, W)
    assert yt.shape[:2] == (B, N * 64)
    y = np.empty((B, T * H * W, heads, D), np.uint16)
    lib().oracle_untile(B, T, H, W, heads, D, _p(yt), _p(y))
    return y


def pool(xt: np.ndarray, vbs: np.ndarray) -> np.ndarray:
    """Cube means: xt [B, N*64, heads, D] -> [B, heads, N, D] float64."""
    xt = _u16(xt)
    vbs = _i32(vbs)
    B, S, heads, D = xt.shape
    N = S // 64
    out = np.empty((B, heads, N, D), np.float64)
    lib().oracle_pool(B, N, heads, D, _p(xt), _p(vbs), _p(out))
    return out


def coarse(qt, kt, vbs, topk: int, sm_scale: float, want_scores: bool = False):
    """Top-k KV cubes per query cube -> topk_idx [B, heads, N, topk] int32
    (and the fp64 score matrix [B, heads, N, N] if ``want_scores``)."""
    qt, kt, vbs = _u16(qt), _u16(kt), _i32(vbs)
    B, S, heads, D = qt.shape
    N = S // 64
    assert 1 <= topk <= N
    idx = np.empty((B, heads, N, topk), np.int32)
    scores = np.empty((B, heads, N, N), np.float64) if want_scores else None
    lib().oracle_coarse(B, N, heads, D, _p(qt), _p(kt), _p(vbs), topk, float(sm_scale),
                        _p(scores) if scores is not None else None, _p(idx))
    return (idx, scores) if want_scores else idx


def fine(qt, kt, vt, topk_idx, vbs, sm_scale: float, units=None, nthreads: int = 0):
    """Block-sparse attention over the listed query cubes.

    units: flat indices (b*heads + h)*N + i (default: all).  Returns
    (out [nunits, 64, D] float64, lse [nunits, 64] float64, threads used).
    """
    qt, kt, vt = _u16(qt), _u16(kt), _u16(vt)
    topk_idx, vbs = _i32(topk_idx), _i32(vbs)
    B, S, heads, D = qt.shape
    N = S // 64
    topk = topk_idx.shape[-1]
    assert topk_idx.shape == (B, heads, N, topk)
    if units is None:
        units = np.arange(B * heads * N, dtype=np.int64)
    units = np.ascontiguousarray(units, dtype=np.int64)
    out = np.empty((units.size, 64, D), np.float64)
    lse = np.empty((units.size, 64), np.float64)
    used = lib().oracle_fine(B, N, heads, D, _p(qt), _p(kt), _p(vt), _p(topk_idx), _p(vbs),
                             topk, float(sm_scale), _p(units), units.size, _p(out), _p(lse),
                             int(nthreads))
    return out, lse, int(used)


def fine_full(qt, kt, vt, topk_idx, vbs, sm_scale: float, nthreads: int = 0):
    """Fine stage over every query cube, returned in the tiled token layout:
    (out [B, N*64, heads, D] float64, lse [B, heads, N*64] float64)."""
    B, S, heads, D = qt.shape
    N = S // 64
    out_u, lse_u, _ = fine(qt, kt, vt, topk_idx, vbs, sm_scale, None, nthreads)
    out = out_u.reshape(B, heads, N * 64, D).transpose(0, 2, 1, 3).copy()
    lse = lse_u.reshape(B, heads, N * 64).copy()
    return out, lse


def fine_counts(qt, kt, vt, topk_idx, counts, vbs, sm_scale: float, units=None, nthreads: int = 0):
    """Fine stage with a per-row count of valid entries ([VSA-AMD] Block-Sparse
    Encoding: a per-row number of valid blocks beside the block-index table):
    query cube i attends the cubes topk_idx[b, h, i, :counts[b, h, i]] only.

    Computed by the fixed-length routine on an equivalent problem: one extra
    cube with no real token (vbs = 0) is appended and every unused entry
    points to it, so it adds no key.  Same returns as fine(); units index the
    original N cubes.
    """
    qt, kt, vt = _u16(qt), _u16(kt), _u16(vt)
    topk_idx, vbs = _i32(topk_idx), _i32(vbs)
    B, S, heads, D = qt.shape
    N = S // 64
    k = topk_idx.shape[-1]
    c = np.clip(np.asarray(counts, np.int64), 0, k)
    assert c.shape == (B, heads, N)
    pad = np.zeros((B, 64, heads, D), np.uint16)
    qt2, kt2, vt2 = (np.ascontiguousarray(np.concatenate([x, pad], axis=1)) for x in (qt, kt, vt))
    vbs2 = np.concatenate([vbs, np.zeros(1, np.int32)])
    idx2 = np.full((B, heads, N + 1, k), N, np.int32)
    idx2[:, :, :N] = np.where(np.arange(k)[None, None, None, :] < c[..., None], topk_idx, N)
    if units is None:
        units = np.arange(B * heads * N, dtype=np.int64)
    units = np.asarray(units, dtype=np.int64)
    units2 = (units // N) * (N + 1) + units % N
    return fine(qt2, kt2, vt2, idx2, vbs2, sm_scale, units2, nthreads)


def fine_full_counts(qt, kt, vt, topk_idx, counts, vbs, sm_scale: float, nthreads: int = 0):
    """fine_counts over every query cube, in the tiled token layout (as fine_full)."""
    B, S, heads, D = _u16(qt).shape
    N = S // 64
    out_u, lse_u, _ = fine_counts(qt, kt, vt, topk_idx, counts, vbs, sm_scale, None, nthreads)
    out = out_u.reshape(B, heads, N * 64, D).transpose(0, 2, 1, 3).copy()
    lse = lse_u.reshape(B, heads, N * 64).copy()
    return out, lse


def coarse_attn(qt, kt, vt, vbs, sm_scale: float) -> np.ndarray:
    """Coarse-stage attention output ([VSA-AMD] Two-Stage Architecture, Stage 1:
    Coarse Selection -- each cube mean-pooled into cube-level Qc, Kc, Vc,
    cube-to-cube attention; the final output gates it with the fine output).

    Per (b, head): O_c = softmax(sm_scale * Qc Kc^T) Vc over the key cubes that
    hold a real token (vbs > 0), in float64.  A query cube without a real token
    gets zeros.  Returns [B, heads, N, D] float64.
    """
    vbs = _i32(vbs)
    qm, km, vm = pool(qt, vbs), pool(kt, vbs), pool(vt, vbs)  # [B, heads, N, D]
    live = vbs > 0
    out = np.zeros_like(qm)
    if not live.any():
        return out
    s = sm_scale * np.matmul(qm, km[:, :, live, :].transpose(0, 1, 3, 2))  # [B, heads, N, n_live]
    s -= s.max(axis=-1, keepdims=True)
    w = np.exp(s)
    w /= w.sum(axis=-1, keepdims=True)
    out[:] = np.matmul(w, vm[:, :, live, :])
    out[:, :, ~live, :] = 0.0
    return out


def _bf16_to_f64(bits) -> np.ndarray:
    return (_u16(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def gated_combine(fine_out, coarse_out, gate_c, gate_f) -> np.ndarray:
    """Gated sum of the two stages ([VSA-AMD] Two-Stage Architecture: the
    final output combines the coarse and fine outputs through gates), in the
    tiled token layout: for token slot s of cube i,
        out[b, 64 i + s, h, :] = gate_c[b, 64 i + s, h, :] * O_c[b, h, i, :]
                               + gate_f[b, 64 i + s, h, :] * fine[b, 64 i + s, h, :].
    fine_out: float [B, 64 N, heads, D]; coarse_out: [B, heads, N, D];
    gate_c, gate_f: bf16 bits [B, 64 N, heads, D].  Returns float64."""
    fine_out = np.asarray(fine_out, np.float64)
    B, S, heads, D = fine_out.shape
    N = S // 64
    assert coarse_out.shape == (B, heads, N, D)
    per_slot = np.repeat(np.asarray(coarse_out, np.float64).transpose(0, 2, 1, 3), 64, axis=1)
    return _bf16_to_f64(gate_c) * per_slot + _bf16_to_f64(gate_f) * fine_out


def block_pool(x, block: int) -> np.ndarray:
    """Means of contiguous token blocks ([INT8-WAN] Decoupling Block Selection
    from Sparse CUDA Kernels, step 1): x bf16 bits [B, S, heads, D] in raster
    token order, S a multiple of `block` -> [B, heads, S / block, D] float64."""
    x = _bf16_to_f64(x)
    B, S, heads, D = x.shape
    assert S % block == 0
    nb = S // block
    return x.reshape(B, nb, block, heads, D).mean(axis=2).transpose(0, 2, 1, 3).copy()


def block_select_cdf(q, k, block: int, tau: float, sm_scale: float):
    """Mean-pool block selector with a cumulative threshold ([INT8-WAN]
    Decoupling Block Selection from Sparse CUDA Kernels, steps 1-3): pool each
    `block`-token query and key block, score S_ij = qbar_i . kbar_j, order each
    query block's key blocks by score (descending; equal scores: lower index
    first) and keep them in that order until the kept share of
    softmax_j(sm_scale * S_ij) reaches tau (at least one block; all of them if
    the sum never reaches tau).

    Returns (idx int32 [B, heads, nb, nb]: the kept blocks first, in that
    order, then -1; counts int32 [B, heads, nb]) and the fp64 scores."""
    qm, km = block_pool(q, block), block_pool(k, block)
    B, heads, nb, _ = qm.shape
    scores = np.matmul(qm, km.transpose(0, 1, 3, 2))  # [B, heads, nb, nb]
    idx = np.full((B, heads, nb, nb), -1, np.int32)
    counts = np.zeros((B, heads, nb), np.int32)
    for b in range(B):
        for h in range(heads):
            for i in range(nb):
                s = scores[b, h, i]
                order = sorted(range(nb), key=lambda j: (-s[j], j))
                w = np.exp(sm_scale * (s - s.max()))
                w /= w.sum()
                kept, mass = 0, 0.0
                while kept < nb and (kept == 0 or mass < tau):
                    mass += w[order[kept]]
                    kept += 1
                idx[b, h, i, :kept] = order[:kept]
                counts[b, h, i] = kept
    return idx, counts, scores


def blocks_to_cube_lut(idx, counts, cubes_per_block: int = 2):
    """A block-level table over `cubes_per_block`-cube blocks (128 tokens = 2
    cubes of 64) -> the cube-level table of the fine stage: query cube
    c * cubes_per_block + r (any r) attends the cubes of its block's kept key
    blocks, block j -> cubes j * cubes_per_block + 0 .. cubes_per_block - 1, in
    the block order.  Returns (cube_idx [B, heads, nb * cpb, nb * cpb] with -1
    past the count, cube_counts [B, heads, nb * cpb])."""
    B, heads, nb, kmax = idx.shape
    c = cubes_per_block
    out = np.full((B, heads, nb * c, kmax * c), -1, np.int32)
    cnt = np.repeat(counts * c, c, axis=2).astype(np.int32)
    for r in range(c):
        sub = np.where(idx >= 0, idx * c + r, -1)
        out[:, :, :, r::c] = np.repeat(sub, c, axis=2)
    return out, cnt


def row_peak(qt, kt, topk_idx, vbs, sm_scale: float, units):
    """Row peakedness over the row's selected keys ([INT8-WAN] Dynamic
    Sparsity Budgeting via Softmax Normalizer Registers: with m the row's
    largest logit and l = sum_x exp(s_x - m), max_prob = 1 / l is the row's
    largest softmax weight).

    units: flat indices (b * heads + h) * N + i.  Returns (max_prob, lse),
    each [len(units), 64] float64; a row with no key has max_prob 0 and
    lse -inf."""
    q, k = _bf16_to_f64(qt), _bf16_to_f64(kt)
    vbs = _i32(vbs)
    B, S, heads, D = q.shape
    N = S // 64
    units = np.asarray(units, np.int64)
    max_prob = np.zeros((len(units), 64))
    lse = np.full((len(units), 64), -np.inf)
    for n, u in enumerate(units):
        b, h, i = u // (heads * N), (u // N) % heads, u % N
        keys = [64 * j + s for j in topk_idx[b, h, i] if 0 <= j < N for s in range(vbs[j])]
        if not keys:
            continue
        logits = sm_scale * q[b, 64 * i: 64 * i + 64, h] @ k[b, keys, h].T  # [64, n_keys]
        m = logits.max(axis=1)
        l = np.exp(logits - m[:, None]).sum(axis=1)
        max_prob[n] = 1.0 / l
        lse[n] = m + np.log(l)
    return max_prob, lse


def captured_mass(lse_selected, lse_all) -> np.ndarray:
    """The share of a row's full (dense) softmax mass that falls on its
    selected keys, sum_{x selected} exp(s_x) / sum_{all x} exp(s_x) =
    exp(lse_selected - lse_all): the recall of a selection against dense
    attention ([INT8-WAN] Selection Heuristic Ablation and Recall Analysis).
    A row with no selected key captures 0."""
    a = np.asarray(lse_selected, np.float64)
    b = np.asarray(lse_all, np.float64)
    with np.errstate(invalid="ignore"):
        return np.where(np.isneginf(a), 0.0, np.exp(a - b))


def rel_l1(approx, ref) -> float:
    """Mean absolute error over the mean absolute reference value ([INT8-WAN]
    glossary: relative-L1, the quality gate of the sparse lever)."""
    approx = np.asarray(approx, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.abs(approx - ref).mean() / np.abs(ref).mean())


def default_threads() -> int:
    return int(lib().oracle_default_threads())
