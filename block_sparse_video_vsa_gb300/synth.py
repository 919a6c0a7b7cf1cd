"""Seeded synthetic workloads for the VSA hot path.

This module produces inputs only: bf16 q, k, v token rows in raster
(t, h, w) order with the shapes of the video-diffusion attention calls the
VSA pages describe, plus a few structured index patterns.  It holds none of
the method's arithmetic (no tiling, pooling, scoring, top-k or softmax), so
both the CUDA path's tests and the CPU oracle can consume its output.

Recipe (per head h):
  g, A_q, A_k, g'  independent smooth fields over the (t, h, w) grid, each a
                   random mix of 32 plane waves cos(w.x + phi) whose wave
                   numbers are drawn in [-pi/4, pi/4] per axis (periods of at
                   least 8 tokens), normalised to unit variance per channel;
  q = alpha_h * (g + A_q + 0.3 n),   k = alpha_h * (g + A_k + 0.3 n),
  v = beta    * (g' + 0.3 n),        n ~ N(0, 1) fresh per tensor.
The shared field g gives locality and data-dependent, head-varying cube
selections; A_q, A_k keep it from being a sliding window.  alpha_h is chosen
so that the standard deviation of q.k/sqrt(D) over 10^4 random token pairs is
sigma_h.  beta keeps output magnitudes near 0.03, where bf16 output rounding
stays well inside a 1e-4 mean-absolute-difference budget.

All randomness comes from numpy's PCG64 seeded per config and per head.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np

CUBE = 4  # cube edge along t, h and w; 64 tokens per cube


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int  # latent height (grid rows)
    W: int
    heads: int
    D: int
    topk: int
    seed: int
    sigma: Optional[float] = None  # fixed logit std, else U[1, 6] per head
    outlier: bool = False

    @property
    def grid(self):
        return (self.B, self.T, self.H, self.W)

    @property
    def tokens(self) -> int:
        return self.T * self.H * self.W

    @property
    def cube_grid(self):
        return (-(-self.T // CUBE), -(-self.H // CUBE), -(-self.W // CUBE))

    @property
    def ncubes(self) -> int:
        nt, nh, nw = self.cube_grid
        return nt * nh * nw

    @property
    def s_pad(self) -> int:
        return 64 * self.ncubes

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def fine_flops(self, topk: Optional[int] = None) -> float:
        """Effective FLOPs of the fine stage: 4 * S_pad * k * 64 * D * heads * B."""
        k = self.topk if topk is None else topk
        return 4.0 * self.s_pad * k * 64 * self.D * self.heads * self.B

    def with_topk(self, topk: int) -> "Workload":
        return dataclasses.replace(self, topk=topk, name=f"{self.name}-k{topk}")


# The five workloads: tiny (seconds on the oracle), mid, Wan2.2-A14B shape,
# the Wan shape with an overflow-provoking head, and the HunyuanVideo shape.
WORKLOADS = {
    "tiny": Workload("tiny", 1, 5, 6, 10, heads=2, D=64, topk=3, seed=1000, sigma=3.0),
    "mid": Workload("mid", 1, 9, 16, 16, heads=8, D=128, topk=12, seed=1001),
    "wan": Workload("wan", 1, 21, 30, 52, heads=40, D=128, topk=78, seed=1002),
    "wan_outlier": Workload("wan_outlier", 1, 21, 30, 52, heads=40, D=128, topk=78, seed=1003,
                            outlier=True),
    "hunyuan": Workload("hunyuan", 1, 30, 48, 80, heads=24, D=128, topk=192, seed=1004),
}
OUTLIER_TOPKS = (187, 78, 31)

# Token sequences attended in contiguous 128-token blocks (no cube tiling):
# the Wan2.1-shape attention call of "VSA: Accelerating Video Diffusion
# Inference with Sparse Attention on AMD GPUs" (q, k, v [1, 12, 32768, 128]).
# Its fields are those of the 21 x 30 x 52 grid flattened in raster order
# (32,760 tokens), zero-padded to 32,768.
SEQUENCE_WORKLOADS = {
    "blocks128": (Workload("blocks128", 1, 21, 30, 52, heads=12, D=128, topk=1, seed=1005), 32768),
}

V_SCALE = 0.05  # beta
NOISE = 0.3
N_MODES = 32
OUTLIER_HEAD0_SIGMA = 160.0  # logit std of head 0 in the outlier workload (max ~ 1e3)
OUTLIER_TOKEN_SCALE = 30.0


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even) and return the bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _coords(T: int, H: int, W: int):
    t, h, w = np.meshgrid(np.arange(T, dtype=np.float32), np.arange(H, dtype=np.float32),
                          np.arange(W, dtype=np.float32), indexing="ij")
    return t.reshape(-1), h.reshape(-1), w.reshape(-1)


def smooth_field(rng: np.random.Generator, coords, D: int, modes: int = N_MODES) -> np.ndarray:
    """[tokens, D] float32 field: a random mix of plane waves, unit variance per channel."""
    t, h, w = coords
    om = rng.uniform(-math.pi / 4, math.pi / 4, size=(3, modes)).astype(np.float32)
    phi = rng.uniform(0.0, 2 * math.pi, size=(modes,)).astype(np.float32)
    arg = t[:, None] * om[0] + h[:, None] * om[1] + w[:, None] * om[2] + phi
    F = np.cos(arg, dtype=np.float32)
    A = rng.standard_normal((modes, D), dtype=np.float32)
    G = F @ A
    G -= G.mean(axis=0, keepdims=True)
    G /= np.maximum(G.std(axis=0, keepdims=True), 1e-6)
    return G


def _logit_std(rng, qr: np.ndarray, kr: np.ndarray, pairs: int = 10_000) -> float:
    a = rng.integers(0, qr.shape[0], size=pairs)
    b = rng.integers(0, kr.shape[0], size=pairs)
    u = np.einsum("nd,nd->n", qr[a].astype(np.float64), kr[b].astype(np.float64))
    return float(u.std() / math.sqrt(qr.shape[1]))


def make_inputs(wl: Workload, B: Optional[int] = None):
    """Return dict(q, k, v) of uint16 bf16 bits [B, T*H*W, heads, D] plus metadata."""
    B = wl.B if B is None else B
    S = wl.tokens
    coords = _coords(wl.T, wl.H, wl.W)
    q = np.empty((B, S, wl.heads, wl.D), np.uint16)
    k = np.empty_like(q)
    v = np.empty_like(q)
    cfg_rng = np.random.Generator(np.random.PCG64(wl.seed))
    if wl.sigma is not None:
        sigmas = np.full(wl.heads, wl.sigma)
    else:
        sigmas = cfg_rng.uniform(1.0, 6.0, size=wl.heads)
    if wl.outlier:
        sigmas[0] = OUTLIER_HEAD0_SIGMA
    extreme = []  # (head, token) pairs scaled x30 in the outlier workload
    if wl.outlier:
        nt, nh, nw = wl.cube_grid
        cubes = cfg_rng.choice(nt * nh * nw, size=3, replace=False)
        for n_c, c in enumerate(cubes):
            ct, rem = divmod(int(c), nh * nw)
            ch, cw = divmod(rem, nw)
            head = 1 + (n_c % 2)
            cand = [((t * wl.H + h) * wl.W + w)
                    for t in range(ct * CUBE, min(wl.T, ct * CUBE + CUBE))
                    for h in range(ch * CUBE, min(wl.H, ch * CUBE + CUBE))
                    for w in range(cw * CUBE, min(wl.W, cw * CUBE + CUBE))]
            for tok in cfg_rng.choice(cand, size=min(4, len(cand)), replace=False):
                extreme.append((head, int(tok)))
    alphas = np.empty(wl.heads)
    for b in range(B):
        for h in range(wl.heads):
            rng = np.random.Generator(np.random.PCG64([wl.seed, b, h]))
            g = smooth_field(rng, coords, wl.D)
            aq = smooth_field(rng, coords, wl.D)
            ak = smooth_field(rng, coords, wl.D)
            gv = smooth_field(rng, coords, wl.D)
            qr = g + aq + NOISE * rng.standard_normal(g.shape, dtype=np.float32)
            kr = g + ak + NOISE * rng.standard_normal(g.shape, dtype=np.float32)
            vr = gv + NOISE * rng.standard_normal(g.shape, dtype=np.float32)
            alpha = math.sqrt(sigmas[h] / _logit_std(rng, qr, kr))
            alphas[h] = alpha
            qr *= alpha
            kr *= alpha
            for (eh, tok) in extreme:
                if eh == h:
                    qr[tok] *= OUTLIER_TOKEN_SCALE
                    kr[tok] *= OUTLIER_TOKEN_SCALE
            q[b, :, h, :] = bf16_bits(qr)
            k[b, :, h, :] = bf16_bits(kr)
            v[b, :, h, :] = bf16_bits(V_SCALE * vr)
    return {"q": q, "k": k, "v": v, "sigmas": sigmas, "alphas": alphas, "extreme": extreme}


def random_topk(seed: int, B: int, heads: int, N: int, topk: int) -> np.ndarray:
    """Distinct cube ids per query cube, drawn uniformly, in random order."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = np.empty((B, heads, N, topk), np.int32)
    for b in range(B):
        for h in range(heads):
            for i in range(N):
                out[b, h, i] = rng.choice(N, size=topk, replace=False)
    return out


def window_topk(cube_grid: Sequence[int], radius: Sequence[int], B: int, heads: int) -> np.ndarray:
    """Tile-level sliding-window lists (the neighbourhood |i - i'| <= r per axis
    of Sliding Tile Attention).  At the grid border the window is shifted back
    inside the grid, so every query cube lists the same number of cubes."""
    nt, nh, nw = cube_grid
    rt, rh, rw = radius
    kt, kh, kw = 2 * rt + 1, 2 * rh + 1, 2 * rw + 1
    assert kt <= nt and kh <= nh and kw <= nw
    N = nt * nh * nw
    out = np.empty((B, heads, N, kt * kh * kw), np.int32)
    for ct in range(nt):
        t0 = min(max(ct - rt, 0), nt - kt)
        for ch in range(nh):
            h0 = min(max(ch - rh, 0), nh - kh)
            for cw in range(nw):
                w0 = min(max(cw - rw, 0), nw - kw)
                ids = [((a * nh + b2) * nw + c) for a in range(t0, t0 + kt)
                       for b2 in range(h0, h0 + kh) for c in range(w0, w0 + kw)]
                out[:, :, (ct * nh + ch) * nw + cw] = np.asarray(ids, np.int32)
    return out


def sequence_inputs(wl: Workload, s_len: int):
    """Raster-order q, k, v of workload `wl` zero-padded to `s_len` tokens (a
    multiple of 128): dict(q, k, v) of bf16 bits [B, s_len, heads, D] plus
    `real` (tokens before the padding), `vbs` (int32 per 64-token slot group:
    64, then the real tokens of the last groups) and `extreme`."""
    d = make_inputs(wl)
    real = wl.tokens
    assert s_len % 128 == 0 and s_len >= real
    out = {"real": real, "extreme": d["extreme"]}
    for n in ("q", "k", "v"):
        x = np.zeros((wl.B, s_len, wl.heads, wl.D), np.uint16)
        x[:, :real] = d[n]
        out[n] = x
    out["vbs"] = np.clip(real - 64 * np.arange(s_len // 64), 0, 64).astype(np.int32)
    return out


def make_sequence_inputs(name: str):
    """sequence_inputs of a SEQUENCE_WORKLOADS entry."""
    wl, s_len = SEQUENCE_WORKLOADS[name]
    return sequence_inputs(wl, s_len)
