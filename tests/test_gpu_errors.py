"""Failure detection on the GPU without faulting it.

- The bounded-wait self test waits on a barrier nobody arrives on; the wait
  must run out, report it, set the device error word and return normally.
- The index validator flags out-of-range and repeated indices and bad vbs.
"""
import numpy as np
import pytest
import torch

import block_sparse_video_vsa_gb300 as vsa
from gpu_util import i32_dev

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_reports():
    vsa.device_error(reset=True)
    assert vsa.debug_wait_timeout(2_000_000) == 1  # 2 ms
    assert vsa.device_error(reset=True) & 1
    assert vsa.device_error() == 0
    # The context is still usable afterwards.
    x = torch.ones(4, device="cuda")
    assert float((x * 2).sum()) == 8.0


def test_validator_flags():
    N, k = 10, 3
    good = np.tile(np.array([1, 4, 7], np.int32), (1, 2, N, 1))
    vbs = np.full(N, 64, np.int32)
    assert vsa.validate_indices(i32_dev(good), i32_dev(vbs)) == 0
    bad = good.copy()
    bad[0, 1, 5, 2] = N
    assert vsa.validate_indices(i32_dev(bad), i32_dev(vbs)) & 1
    dup = good.copy()
    dup[0, 0, 3, 1] = 1
    assert vsa.validate_indices(i32_dev(dup), i32_dev(vbs)) & 2
    vb = vbs.copy()
    vb[4] = 65
    assert vsa.validate_indices(i32_dev(good), i32_dev(vb)) & 4


def test_validator_with_counts_accepts_a_table_from_compressed_rows():
    """A table written by vsa_table_from_csr (-1 after each row's entries)
    validates cleanly with its counts, and still fails without them; a bad
    entry inside a row's count and a count above topk are both flagged."""
    rng = np.random.default_rng(11)
    B, heads, N, width = 1, 2, 12, 5
    rows = B * heads * N
    lengths = rng.integers(0, width + 1, size=rows)
    lengths[:2] = [0, width]
    lut_ptr = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    kv_idx = np.concatenate([rng.choice(N, size=n, replace=False) for n in lengths]).astype(np.int32)
    table, counts = vsa.table_from_csr(lut_ptr, kv_idx, width, N, shape=(B, heads, N))
    vbs = i32_dev(np.full(N, 64, np.int32))
    assert vsa.validate_indices(i32_dev(table), vbs, counts=i32_dev(counts)) == 0
    assert vsa.validate_indices(i32_dev(table), vbs) & 1  # the -1 padding, checked as entries
    bad = table.copy()
    r = np.argwhere(counts > 0)[0]
    bad[tuple(r)][0] = N
    assert vsa.validate_indices(i32_dev(bad), vbs, counts=i32_dev(counts)) & 1
    big = counts.copy()
    big.reshape(-1)[0] = width + 1
    assert vsa.validate_indices(i32_dev(table), vbs, counts=i32_dev(big)) & 8
