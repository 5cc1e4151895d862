"""The whole step -- six launches with programmatic dependencies -- captured
once into a CUDA graph and replayed: every output equals, bit for bit, that
of the same launches issued one by one (the kernels are deterministic). The
library makes no allocation, host synchronisation or device-wide call on its
launch path once a device has been used, so a caller can put a decode loop
in a graph."""

import pytest
import torch

from gpu_util import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    return ensure_built()


OUTS = ("conv_y", "o", "res_out", "head_out")


def test_whole_step_replays_from_a_cuda_graph():
    import bench

    dev = torch.device("cuda:0")
    wl = bench.Workload(dev)
    stream = torch.cuda.Stream(dev)
    wl.step(stream)  # first use of the device: its facts are looked up here
    torch.cuda.synchronize(dev)
    wl.api.cc_check_device()
    ref = {n: getattr(wl, n).clone() for n in OUTS}

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        wl.step(torch.cuda.current_stream())
    for n in OUTS:
        getattr(wl, n).fill_(float("nan"))
    torch.cuda.synchronize(dev)
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize(dev)
    wl.api.cc_check_device()
    for n in OUTS:
        assert torch.equal(getattr(wl, n), ref[n]), f"{n} differs after graph replay"
