"""GPU: PipelineGraph (pipeline() captured once as a CUDA graph) replays give
the eager pipeline's bits, on the inputs it was built with and on other inputs
copied into its buffers; the eager pipeline itself is checked against the
oracle in test_gpu_pipeline."""
import pytest
import torch

import block_sparse_video_vsa_gb300 as vsa
from block_sparse_video_vsa_gb300 import synth
from gpu_util import to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["mid", "wan"])
def test_graph_replay_equals_eager(name):
    wl = synth.WORKLOADS[name]
    d = synth.make_inputs(wl)
    q, k, v = (to_dev(d[n]) for n in "qkv")
    eager = [t.clone() for t in vsa.pipeline(q, k, v, wl.grid, wl.topk, wl.sm_scale)]
    g = vsa.PipelineGraph(q, k, v, wl.grid, wl.topk, wl.sm_scale)
    got = g()
    torch.cuda.synchronize()
    assert vsa.device_error(reset=True) == 0
    for a, b in zip(got, eager):
        assert torch.equal(a, b)
    # Other inputs through the same graph: the roles of q, k, v rotated.
    eager2 = [t.clone() for t in vsa.pipeline(k, v, q, wl.grid, wl.topk, wl.sm_scale)]
    got2 = g(k, v, q)
    torch.cuda.synchronize()
    assert vsa.device_error(reset=True) == 0
    for a, b in zip(got2, eager2):
        assert torch.equal(a, b)
    assert not torch.equal(got2[2], eager[2])  # the selection did change


def test_graph_refuses_other_shapes():
    wl = synth.WORKLOADS["tiny"]
    d = synth.make_inputs(wl)
    q, k, v = (to_dev(d[n]) for n in "qkv")
    g = vsa.PipelineGraph(q, k, v, wl.grid, wl.topk, wl.sm_scale)
    with pytest.raises(ValueError):
        g(q[:, :-1])
