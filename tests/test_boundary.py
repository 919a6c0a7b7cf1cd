"""Host-only checks of the C ABI boundary (no GPU needed).

- libvsa.so builds for sm_103a, loads, and exports every entry point that
  include/vsa.h declares;
- argument validation runs before any CUDA call and returns the documented
  status codes (NULL pointers, bad sizes, unsupported D, misalignment).
Only argument combinations that fail validation are passed here: nothing in
this file launches a kernel.
"""
import ctypes
import os
import re

import pytest

import block_sparse_video_vsa_gb300 as vsa
from block_sparse_video_vsa_gb300 import build as vbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "vsa.h")
OK, INVALID, UNSUPPORTED, ALIGNMENT = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    vbuild.build()
    return vsa.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vsa_[a-z_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("vsa_tile", "vsa_untile", "vsa_coarse_select", "vsa_sparse_attn_fwd",
              "vsa_coarse_workspace_bytes", "vsa_num_cubes", "vsa_status_string",
              "vsa_validate_indices", "vsa_device_error", "vsa_debug_wait_timeout",
              "vsa_pair_cubes", "vsa_pair_workspace_bytes", "vsa_sparse_attn_fwd_paired",
              "vsa_sparse_attn_fwd_ex", "vsa_sparse_attn_fwd_gated", "vsa_coarse_attn",
              "vsa_coarse_attn_workspace_bytes", "vsa_kernel_launches", "vsa_table_from_csr",
              "vsa_validate_indices_ex", "vsa_coarse_select_noalloc", "vsa_block_select",
              "vsa_block_select_workspace_bytes", "vsa_sparse_attn_fwd_peak"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} not exported"


def test_plain_c_program_links_against_the_abi(lib, tmp_path):
    """The header is valid C99 and a C program links every entry point from
    the shared library (it calls only the host-side status strings)."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    names = declared_functions()
    src = ['#include <stdio.h>', '#include "vsa.h"', "int main(void) {",
           "    typedef void (*fn_t)(void);",
           "    const fn_t fns[] = {" + ", ".join(f"(fn_t)&{n}" for n in names) + "};",
           "    for (unsigned i = 0; i < sizeof fns / sizeof fns[0]; ++i) if (!fns[i]) return 1;",
           '    printf("%s %s\\n", vsa_status_string(VSA_OK), vsa_status_string(VSA_ERR_TIMEOUT));',
           "    return 0;", "}"]
    c_file = tmp_path / "abi.c"
    c_file.write_text("\n".join(src) + "\n")
    exe = tmp_path / "abi"
    libdir = os.path.dirname(vbuild.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-pedantic", "-I", os.path.dirname(HEADER), str(c_file),
                    "-o", str(exe), "-L", libdir, "-lvsa", f"-Wl,-rpath,{libdir}"], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.split() == ["VSA_OK", "VSA_ERR_TIMEOUT"], (r.stdout, r.stderr)


def test_status_strings(lib):
    for code, name in enumerate(["VSA_OK", "VSA_ERR_INVALID_ARG", "VSA_ERR_UNSUPPORTED", "VSA_ERR_ALIGNMENT",
                                 "VSA_ERR_INDEX_RANGE", "VSA_ERR_TIMEOUT", "VSA_ERR_CUDA"]):
        assert lib.vsa_status_string(code).decode() == name
    assert lib.vsa_status_string(99).decode() == "VSA_ERR_UNKNOWN"


def test_num_cubes(lib):
    g = vsa.VsaGrid(1, 21, 30, 52, 40, 128)
    assert lib.vsa_num_cubes(ctypes.byref(g)) == 624
    g = vsa.VsaGrid(1, 0, 30, 52, 40, 128)
    assert lib.vsa_num_cubes(ctypes.byref(g)) == -1
    assert lib.vsa_num_cubes(None) == -1


def test_workspace_bytes(lib):
    # from 256 cubes the fp32 score matrix goes through the workspace
    assert lib.vsa_coarse_workspace_bytes(1, 40, 624, 128) == 16 * 40 * 624 * 128 + 8 * 40 * 624 + 4 * 40 * 624 * 624
    assert lib.vsa_coarse_workspace_bytes(1, 2, 255, 128) == 16 * 2 * 255 * 128 + 8 * 2 * 255
    assert lib.vsa_coarse_workspace_bytes(0, 40, 624, 128) == 0
    assert lib.vsa_coarse_workspace_bytes(1, 24, 1920, 128) == (16 * 24 * 1920 * 128 + 8 * 24 * 1920
                                                               + 4 * 24 * 1920 * 1920)


A = 0x10000   # fake, never dereferenced: every call below fails validation first
MIS = 0x10008


def test_tile_validation(lib):
    g = vsa.VsaGrid(1, 5, 6, 10, 2, 64)
    assert lib.vsa_tile(None, A, A, None, None) == INVALID
    assert lib.vsa_tile(ctypes.byref(g), None, A, None, None) == INVALID
    assert lib.vsa_tile(ctypes.byref(g), A, MIS, None, None) == ALIGNMENT
    bad = vsa.VsaGrid(1, 5, 6, 10, 1, 4)  # heads * D not a multiple of 8
    assert lib.vsa_tile(ctypes.byref(bad), A, A, None, None) == UNSUPPORTED
    assert lib.vsa_untile(ctypes.byref(g), MIS, A, None) == ALIGNMENT
    assert lib.vsa_untile(ctypes.byref(g), A, None, None) == INVALID


def test_coarse_validation(lib):
    f = lib.vsa_coarse_select
    assert f(None, A, A, 1, 12, 2, 64, 3, 0.0, A, A, None) == INVALID
    assert f(A, A, A, 1, 12, 2, 64, 0, 0.0, A, A, None) == INVALID       # topk = 0
    assert f(A, A, A, 1, 12, 2, 64, 13, 0.0, A, A, None) == INVALID      # topk > ncubes
    assert f(A, A, A, 1, 12, 2, 96, 3, 0.0, A, A, None) == UNSUPPORTED   # D = 96
    assert f(A, A, A, 1, 5000, 2, 64, 3, 0.0, A, A, None) == UNSUPPORTED  # ncubes > 4096
    assert f(A, MIS, A, 1, 12, 2, 64, 3, 0.0, A, A, None) == ALIGNMENT
    assert f(A, A, A, 1, 12, 2, 64, 3, float("nan"), A, A, None) == INVALID


def test_fine_validation(lib):
    f = lib.vsa_sparse_attn_fwd
    assert f(A, A, A, A, A, 1, 12, 2, 64, 3, 0.0, None, None, None) == INVALID
    assert f(A, A, A, A, A, 1, 12, 2, 64, 0, 0.0, A, None, None) == INVALID
    assert f(A, A, A, A, A, 1, 12, 2, 64, 13, 0.0, A, None, None) == INVALID
    assert f(A, A, A, A, A, 0, 12, 2, 64, 3, 0.0, A, None, None) == INVALID
    assert f(A, A, A, A, A, 1, 12, 2, 256, 3, 0.0, A, None, None) == UNSUPPORTED
    assert f(A, A, MIS, A, A, 1, 12, 2, 64, 3, 0.0, A, None, None) == ALIGNMENT
    assert f(A, A, A, A, A, 1, 12, 2, 64, 3, 0.0, A, A + 2, None) == ALIGNMENT  # lse


def test_pairing_validation(lib):
    f = lib.vsa_pair_cubes
    assert f(None, 1, 12, 2, 3, A, A, None) == INVALID
    assert f(A, 1, 12, 2, 0, A, A, None) == INVALID       # topk = 0
    assert f(A, 1, 12, 2, 13, A, A, None) == INVALID      # topk > ncubes
    assert f(A, 1, 9000, 2, 3, A, A, None) == UNSUPPORTED  # ncubes > 8192
    assert f(A, 1, 12, 2, 3, MIS, A, None) == ALIGNMENT   # workspace
    assert f(A, 1, 12, 2, 3, A, A + 2, None) == ALIGNMENT  # pairs
    a256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    # per (b, head): bitmaps N x Wp words (Wp: N/32 rounded up to 4), candidate
    # lists N x 16 int16, partner N int16, leftover list 640 int16, its length,
    # window overlaps 640 x 128 uint16; each region 256-byte aligned
    def ws(bh, n):
        wp = ((n + 31) // 32 + 3) // 4 * 4
        return (a256(bh * n * wp * 4) + a256(bh * n * 16 * 2) + a256(bh * n * 2) + a256(bh * 640 * 2)
                + a256(bh * 4) + a256(bh * 640 * 128 * 2))
    assert lib.vsa_pair_workspace_bytes(1, 2, 12, 3) == ws(2, 12) == 512 + 768 + 256 + 2560 + 256 + 327680
    assert lib.vsa_pair_workspace_bytes(1, 40, 624, 78) == ws(40, 624)
    g = lib.vsa_sparse_attn_fwd_paired
    assert g(A, A, A, A, A, A + 2, 1, 12, 2, 64, 3, 0.0, A, None, None) == ALIGNMENT  # pairs
    assert g(A, A, A, A, A, None, 1, 12, 2, 64, 0, 0.0, A, None, None) == INVALID


def test_counts_validation(lib):
    h = lib.vsa_sparse_attn_fwd_ex
    #   qt kt vt idx counts vbs pairs  B  N  H  D  k  scale out lse stream
    assert h(A, A, A, A, A + 2, A, None, 1, 12, 2, 64, 3, 0.0, A, None, None) == ALIGNMENT  # counts
    assert h(A, A, A, A, A, A, A + 2, 1, 12, 2, 64, 3, 0.0, A, None, None) == ALIGNMENT     # pairs
    assert h(A, A, A, A, A, A, None, 1, 12, 2, 64, 13, 0.0, A, None, None) == INVALID      # topk > N
    assert h(A, A, A, A, A, A, None, 1, 12, 2, 256, 3, 0.0, A, None, None) == UNSUPPORTED


def test_coarse_attn_and_gated_validation(lib):
    f = lib.vsa_coarse_attn
    #   qt kt vt vbs  B  N  H  D  scale ws out stream
    assert f(A, A, A, A, 1, 12, 2, 64, 0.0, None, A, None) == INVALID
    assert f(A, A, A, A, 1, 12, 2, 96, 0.0, A, A, None) == UNSUPPORTED
    assert f(A, A, A, A, 1, 12, 2, 64, 0.0, MIS, A, None) == ALIGNMENT
    assert f(A, A, A, A, 1, 12, 2, 64, float("nan"), A, A, None) == INVALID
    lib.vsa_coarse_attn_workspace_bytes.restype = ctypes.c_size_t
    assert lib.vsa_coarse_attn_workspace_bytes(2, 3, 12, 64) == 3 * 2 * 3 * 12 * 64 * 4
    assert lib.vsa_coarse_attn_workspace_bytes(1, 40, 624, 128) == 3 * 40 * 624 * 128 * 4
    g = lib.vsa_sparse_attn_fwd_gated
    #   qt kt vt idx counts vbs pairs  B  N  H  D  k  scale oc gc gf out lse stream
    assert g(A, A, A, A, None, A, None, 1, 12, 2, 64, 3, 0.0, A, None, A, A, None, None) == INVALID
    assert g(A, A, A, A, None, A, None, 1, 12, 2, 64, 3, 0.0, A, A, MIS, A, None, None) == ALIGNMENT


def test_refused_calls_launch_nothing(lib):
    lib.vsa_kernel_launches.restype = ctypes.c_uint64
    n0 = lib.vsa_kernel_launches()
    assert lib.vsa_pair_cubes(None, 1, 12, 2, 3, A, A, None) == INVALID
    assert lib.vsa_sparse_attn_fwd(A, A, A, A, A, 1, 12, 2, 64, 0, 0.0, A, None, None) == INVALID
    assert lib.vsa_kernel_launches() == n0


def test_validator_and_debug_validation(lib):
    assert lib.vsa_validate_indices(None, A, 1, 1, 12, 3, A, None) == INVALID
    assert lib.vsa_validate_indices(A, A, 1, 1, 100000, 3, A, None) == UNSUPPORTED
    assert lib.vsa_validate_indices_ex(None, None, A, 1, 1, 12, 3, A, None) == INVALID
    assert lib.vsa_validate_indices_ex(A, A + 2, A, 1, 1, 12, 3, A, None) == ALIGNMENT
    assert lib.vsa_debug_wait_timeout(10, A, None) == INVALID
    assert lib.vsa_debug_wait_timeout(10 ** 6, None, None) == INVALID
    assert lib.vsa_device_error(None, 0) == INVALID


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros((1, 300, 2, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        vsa.tile(x, (1, 5, 6, 10))


def test_table_from_csr_matches_the_padded_layout():
    import numpy as np
    rng = np.random.default_rng(3)
    B, heads, N, width = 1, 3, 7, 5
    rows = B * heads * N
    lengths = rng.integers(0, width + 1, size=rows)
    lengths[:2] = [0, width]
    lut_ptr = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    kv_idx = rng.integers(0, N, size=int(lut_ptr[-1])).astype(np.int32)
    table, counts = vsa.table_from_csr(lut_ptr, kv_idx, width, N, shape=(B, heads, N))
    assert table.shape == (B, heads, N, width) and counts.shape == (B, heads, N)
    flat, cnt = table.reshape(rows, width), counts.reshape(rows)
    for r in range(rows):
        assert cnt[r] == lengths[r]
        assert flat[r, :lengths[r]].tolist() == kv_idx[lut_ptr[r]:lut_ptr[r + 1]].tolist()
        assert (flat[r, lengths[r]:] == -1).all()


def test_table_from_csr_refuses_bad_offsets(lib):
    import numpy as np
    ok_idx = np.zeros(16, np.int32)
    for bad in ([1, 2, 3], [0, 3, 2], [0, 9, 9]):  # nonzero start, decreasing, row longer than width
        with pytest.raises(vsa.VsaError):
            vsa.table_from_csr(np.array(bad, np.int64), ok_idx, 4, 6)
    table, counts = vsa.table_from_csr(np.array([0, 0, 0], np.int64), np.zeros(0, np.int32), 2, 6)
    assert (table == -1).all() and (counts == 0).all()


def test_table_from_csr_refuses_short_or_out_of_range_indices(lib):
    import ctypes
    import numpy as np
    lut_ptr = np.array([0, 2, 4], np.int64)
    with pytest.raises(ValueError, match="kv_idx"):  # the wrapper: kv_idx shorter than lut_ptr[-1]
        vsa.table_from_csr(lut_ptr, np.zeros(3, np.int32), 2, 6)
    with pytest.raises(ValueError, match="lut_ptr"):
        vsa.table_from_csr(np.array([0], np.int64), np.zeros(0, np.int32), 2, 6)
    # the C entry point itself: nnz below the last offset, and entries outside [0, ncubes)
    idx = np.array([0, 1, 2, 3], np.int32)
    table = np.empty((2, 2), np.int32)
    counts = np.empty(2, np.int32)
    args = lambda nnz, ncubes, kv: (lut_ptr.ctypes.data, kv.ctypes.data, nnz, 2, 2, ncubes,  # noqa: E731
                                    table.ctypes.data, counts.ctypes.data)
    assert lib.vsa_table_from_csr(*args(3, 6, idx)) == INVALID
    assert lib.vsa_table_from_csr(*args(4, 3, idx)) == 4  # VSA_ERR_INDEX_RANGE: entry 3 >= ncubes
    assert lib.vsa_table_from_csr(*args(4, 6, np.array([0, -1, 2, 3], np.int32))) == 4
    assert lib.vsa_table_from_csr(*args(4, 4, idx)) == 0
    assert table.tolist() == [[0, 1], [2, 3]] and counts.tolist() == [2, 2]
    with pytest.raises(vsa.VsaError):
        vsa.table_from_csr(lut_ptr, np.array([0, 1, 7, 3], np.int32), 2, 6)


def test_block_select_validation(lib):
    f = lib.vsa_block_select
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 2 + [ctypes.c_int32] * 4 + [ctypes.c_float] * 2 + [ctypes.c_void_p] * 4
    ok = (A, A, 1, 1024, 2, 64, 0.5, 0.0, A, A, A, None)
    bad = lambda i, v: tuple(v if n == i else x for n, x in enumerate(ok))  # noqa: E731
    assert f(*bad(0, None)) == INVALID
    assert f(*bad(3, 1000)) == INVALID            # S not a multiple of 128
    assert f(*bad(6, 0.0)) == INVALID             # tau outside (0, 1]
    assert f(*bad(6, 1.5)) == INVALID
    assert f(*bad(5, 96)) == UNSUPPORTED          # D
    assert f(*bad(3, 32768 + 128)) == UNSUPPORTED  # more than 256 blocks
    assert f(*bad(8, A + 4)) == ALIGNMENT
    w = lib.vsa_block_select_workspace_bytes
    w.restype = ctypes.c_size_t
    w.argtypes = [ctypes.c_int32] * 4
    assert w(1, 32768, 12, 128) == 2 * 12 * 256 * 128 * 4
    assert w(1, 1000, 12, 128) == 0
