"""The 128-token-block sequence input recipe: the Wan2.1-shape attention
call's layout ([1, 32768, 12, 128]) filled with the 21 x 30 x 52 grid's fields
in raster order and zero padding after the 32,760 real tokens."""
import numpy as np

from block_sparse_video_vsa_gb300 import synth


def test_sequence_inputs_layout_and_padding():
    d = synth.make_sequence_inputs("blocks128")
    wl, s_len = synth.SEQUENCE_WORKLOADS["blocks128"]
    assert s_len == 32768 and d["real"] == 21 * 30 * 52 == 32760
    for n in ("q", "k", "v"):
        assert d[n].shape == (1, 32768, 12, 128) and d[n].dtype == np.uint16
        assert (d[n][:, 32760:] == 0).all()
        assert (d[n][:, :32760] != 0).mean() > 0.99
    assert d["vbs"].shape == (512,) and (d["vbs"][:-1] == 64).all() and d["vbs"][-1] == 56
    again = synth.make_sequence_inputs("blocks128")
    assert np.array_equal(d["q"], again["q"])  # seeded
