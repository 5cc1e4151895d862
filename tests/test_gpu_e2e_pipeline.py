"""The end-to-end chunk loop that bench.py times: pinned host inputs in, the
seven launches, pinned host outputs back, with the copies of one chunk
overlapping the kernels and copies of its neighbours on separate streams.

Consecutive chunks get different inputs (the seeded set and its negation,
alternating), and every chunk has its own host output buffers, so a stage
whose inputs were rewritten by the next chunk's copy before its kernels
finished, or whose outputs were overwritten before they were read back,
shows up as a mismatch. Each chunk's outputs must equal, bit for bit, those
of the same launches run on resident inputs with nothing overlapping (the
kernels are deterministic: fixed reduction order, no atomics)."""

import pytest
import torch

from gpu_util import ensure_built

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    return ensure_built()


def test_pipelined_chunks_match_resident_step():
    import bench

    dev = torch.device("cuda:0")
    wl = bench.Workload(dev)
    stream = torch.cuda.Stream(dev)
    wl.host_buffers()
    sets = [wl.h_in, {n: torch.neg(t).pin_memory() for n, t in wl.h_in.items()}]

    # reference outputs of each input set: resident inputs, one stream, nothing overlapping
    refs = []
    for hs in sets:
        for n, t in hs.items():
            wl.d_in[n].copy_(t)
        torch.cuda.synchronize(dev)
        wl.step(stream)
        torch.cuda.synchronize(dev)
        refs.append({n: t.cpu() for n, t in wl.d_out.items()})
    wl.api.cc_check_device()
    assert not torch.equal(refs[0]["head_out"], refs[1]["head_out"])

    chunks = 4
    outs = [{n: torch.full(t.shape, float("nan"), dtype=t.dtype).pin_memory() for n, t in wl.h_out.items()}
            for _ in range(chunks)]
    for c in range(chunks):
        wl.step_e2e(stream, h_in=sets[c % 2], h_out=outs[c])
    torch.cuda.synchronize(dev)
    wl.api.cc_check_device()
    for c in range(chunks):
        for n, ref in refs[c % 2].items():
            assert torch.equal(outs[c][n], ref), f"chunk {c}: {n} differs from the resident step"


@pytest.mark.parametrize("nbytes,ctas", [(16, 1), (4096 + 16, 3), ((1 << 20) + 48, 8), (100 << 20, 8), (64 << 20, 152)])
def test_copy_to_host_is_a_byte_copy(nbytes, ctas):
    from causal_convolution_gb300 import api

    g = torch.Generator(device="cuda").manual_seed(nbytes)
    src = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device="cuda", generator=g)
    dst = torch.zeros(nbytes, dtype=torch.uint8, pin_memory=True)
    stream = torch.cuda.Stream()
    api.cc_copy_to_host(dst, src, ctas=ctas, stream=stream)
    stream.synchronize()
    api.cc_check_device()
    assert torch.equal(dst, src.cpu())


def test_copy_to_host_rejects_what_the_device_cannot_address():
    from causal_convolution_gb300 import _lib, api

    lib = _lib.load()
    n = 1 << 16
    src = torch.ones(n, dtype=torch.uint8, device="cuda")
    pinned = torch.zeros(n, dtype=torch.uint8, pin_memory=True)
    pageable = torch.zeros(n, dtype=torch.uint8)
    dev_dst = torch.zeros(n, dtype=torch.uint8, device="cuda")
    # pageable host memory, device memory as the destination, pinned memory as
    # the source, a ragged size: rejected on the host, nothing launched
    assert lib.cc_copy_to_host(pageable.data_ptr(), src.data_ptr(), n, 8, None) == 1
    assert b"page-locked" in lib.cc_last_error()
    assert lib.cc_copy_to_host(dev_dst.data_ptr(), src.data_ptr(), n, 8, None) == 1
    assert lib.cc_copy_to_host(pinned.data_ptr(), pinned.data_ptr(), n, 8, None) == 1
    assert b"device memory" in lib.cc_last_error()
    assert lib.cc_copy_to_host(pinned.data_ptr(), src.data_ptr(), n - 8, 8, None) == 1
    with pytest.raises(ValueError):
        api.cc_copy_to_host(pageable, src)
    torch.cuda.synchronize()
    api.cc_check_device()
    assert int(pinned.sum()) == 0
