"""The library's launches can be captured in a CUDA graph: one bench step
(flatten, both reduce-scatters, all-gather, all-reduce) captured once and
replayed gives bit-identical results to eager launches."""
import pytest
import torch

from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def test_step_graph_replay_matches_eager():
    dev = H.device()
    import bench
    stream = torch.cuda.Stream()
    wl = bench.Workload(dev, stream, n_per_rank=1 << 24)
    names = bench.STEP_KERNELS
    outs = lambda: [wl.part_f32_all, wl.params_all, wl.ar_all, wl.ipg1_all]
    part0 = wl.part_hop_all.clone()
    wl.step(names)
    stream.synchronize()
    eager = [t.clone() for t in outs()] + [wl.part_hop_all.clone()]
    wl.part_hop_all.copy_(part0)
    for t in outs():
        t.zero_()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        wl.step(names)
    # capture does not execute: reset the accumulating partition, then replay
    wl.part_hop_all.copy_(part0)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    got = [t for t in outs()] + [wl.part_hop_all]
    for a, b in zip(got, eager):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    wl.plan.close()
