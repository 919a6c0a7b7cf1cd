"""GPU parity of vsa_tile / vsa_untile against the oracle: bit-exact."""
import numpy as np
import pytest
import torch

import block_sparse_video_vsa_gb300 as vsa
import oracle
from block_sparse_video_vsa_gb300 import synth
from gpu_util import to_bits, to_dev

pytestmark = pytest.mark.gpu


def rand_bits(seed, shape):
    return synth.bf16_bits(np.random.default_rng(seed).standard_normal(shape, dtype=np.float32))


@pytest.mark.parametrize("B,grid,heads,D", [
    (1, (5, 6, 10), 2, 64),      # tiny workload shape: all partial-cube kinds
    (1, (9, 16, 16), 8, 128),    # mid
    (2, (3, 5, 7), 3, 64),       # batch 2, every cube partial
    (1, (1, 1, 1), 1, 8),        # one token
    (1, (8, 8, 8), 1, 128),      # divisible: no padding
    (1, (21, 30, 52), 40, 128),  # Wan2.2 shape (full size)
])
def test_tile_untile_bit_exact(B, grid, heads, D):
    g = (B,) + grid
    S = int(np.prod(grid))
    x = rand_bits(hash(grid) % 1000, (B, S, heads, D))
    ref_t, ref_vbs = oracle.tile(x, g)
    xd = to_dev(x)
    xt, vbs = vsa.tile(xd, g)
    torch.cuda.synchronize()
    assert np.array_equal(to_bits(xt), ref_t)
    assert np.array_equal(vbs.cpu().numpy(), ref_vbs)
    y = vsa.untile(xt, g)
    torch.cuda.synchronize()
    assert np.array_equal(to_bits(y), x)
    # Untile ignores padding contents.
    xt2 = xt.clone()
    N = len(ref_vbs)
    for c in range(N):
        if ref_vbs[c] < 64:
            xt2[:, 64 * c + int(ref_vbs[c]): 64 * (c + 1)] = 7.0
    assert torch.equal(vsa.untile(xt2, g), y)


def test_tile_hunyuan_shape():
    wl = synth.WORKLOADS["hunyuan"]
    x = rand_bits(5, (1, wl.tokens, 4, 128))  # 4 heads keep the host copy small
    ref_t, ref_vbs = oracle.tile(x, wl.grid)
    xt, vbs = vsa.tile(to_dev(x), wl.grid)
    torch.cuda.synchronize()
    assert np.array_equal(to_bits(xt), ref_t)
    assert np.array_equal(vbs.cpu().numpy(), ref_vbs)
