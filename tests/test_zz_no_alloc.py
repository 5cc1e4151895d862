"""cc_head_out_noalloc: the output head for callers that cannot allocate device
memory (for example a plugin whose host framework owns every device
allocation and gives it no allocator, or a latency-critical loop where a
cudaMalloc could synchronise the device), so they cannot pass the workspace
cc_head_out needs. Its g intermediate lives in the library's fixed 64 MiB
static scratch array instead.

Checked through the C ABI against cc_head_out (the existing entry point) on
the same inputs, on two calls in a row with different shapes, so a stale g
left in the shared scratch by the first call would show in the second. The
two entry points run the same deterministic kernels, so their outputs must
agree bit for bit; the second call (two carried history frames, the chunked
decode's case) is also held to the parity bar against the fp64 oracle. This
file sorts last so that a run stopping at its first failure has already run
every other test; it also passes alone in a fresh process.
"""

import numpy as np
import pytest
import torch

import oracle
from causal_convolution_gb300 import api, inputs
from gpu_util import assert_parity, ensure_built, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF16 = torch.bfloat16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    return ensure_built()


def both_entry_points(n, d, h, w, cin, seed, hist=0):
    inp = inputs.head_inputs(n, d, h, w, cin, seed=seed, device=DEV)
    x = inp["x"]
    if hist:
        x = torch.cat([inputs.history_frames(n, cin, h, w, seed + 1000, device=DEV), x], 1)
    wp = torch.empty(3 * api.HEAD_G_CH * cin, dtype=BF16, device=DEV)
    api.cc_head_prepare(inp["w"], wp)
    ref = torch.empty((n, d, h, w, api.HEAD_COUT), dtype=BF16, device=DEV)
    ws = torch.empty(api.cc_head_workspace_bytes(n, d, h, w), dtype=torch.uint8, device=DEV)
    api.cc_head_out(x, wp, inp["b"], ref, ws, hist=hist)
    got = torch.full((n, d, h, w, api.HEAD_COUT), float("nan"), dtype=BF16, device=DEV)
    api.cc_head_out_noalloc(x, wp, inp["b"], got, hist=hist)
    api.cc_check_device()
    return got, ref, x, inp


def assert_same_bits(got, ref, what):
    # the same kernels on the same inputs: identical bf16 bit patterns
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), (
        f"{what}: {(got.view(torch.int16) != ref.view(torch.int16)).sum().item()} outputs differ")


def test_noalloc_head_matches_workspace_head_on_two_calls():
    # first call: 109,824 positions, 24.6 MB of the 64 MiB scratch
    got1, ref1, _, _ = both_entry_points(1, 2, 176, 312, 64, seed=51)
    assert_same_bits(got1, ref1, "noalloc head, call 1")
    # second call in a row: a different, smaller shape with two carried
    # history frames reuses the same scratch
    got2, ref2, x2, inp2 = both_entry_points(1, 3, 9, 13, 128, seed=52, hist=2)
    assert_same_bits(got2, ref2, "noalloc head, call 2")
    xn = to_np(x2)
    want = oracle.head_out(xn[:, 2:], to_np(inp2["w"]), to_np(inp2["b"]), history=xn[:, :2])
    assert_parity(to_np(got2), want, "noalloc head, call 2, against the oracle")
    assert np.isfinite(to_np(got1)).all()


def test_noalloc_head_near_its_scratch_limit():
    # 547 x 547 = 299,209 positions: 384 below the 299,593 the scratch holds
    max_positions = api.HEAD_NOALLOC_SCRATCH_BYTES // (api.HEAD_G_CH * 2)
    assert max_positions - 384 == 547 * 547
    got, ref, _, _ = both_entry_points(1, 1, 547, 547, 64, seed=53)
    assert_same_bits(got, ref, "noalloc head at 299,209 positions")


def test_noalloc_head_rejects_more_than_its_scratch_holds():
    max_positions = api.HEAD_NOALLOC_SCRATCH_BYTES // (api.HEAD_G_CH * 2)
    w = 512
    h = max_positions // w + 1  # one frame just over the limit
    x = torch.empty((1, 1, h, w, 64), dtype=BF16, device=DEV)
    wp = torch.empty(3 * api.HEAD_G_CH * 64, dtype=BF16, device=DEV)
    b = torch.zeros(12, dtype=BF16, device=DEV)
    out = torch.empty((1, 1, h, w, 12), dtype=BF16, device=DEV)
    with pytest.raises(api.CCError) as e:
        api.cc_head_out_noalloc(x, wp, b, out)
    assert e.value.status == 1
    assert "scratch" in str(e.value)
    api.cc_check_device()
