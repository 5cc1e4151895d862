"""Attention with the softmax numerators kept on chip (cc_attn_frame_fused):
the statistics-only scores pass, then one kernel that computes S per 256-key
tile in tensor memory, turns it into E = bf16(exp2(kx*S - c_row)) in shared
memory and accumulates E v into O. Checked against the fp64 oracle's softmax
attention on ragged frames (one and several key tiles, rows past the last
full 256-row block), peaked rows, packed qkv and the full attention
configuration sampled; the statistics pass against the numerators kernel's
statistics bit for bit."""

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


def run_fused(q, k, v):
    t, hw, c = q.shape
    o = torch.full((t, hw, c), float("nan"), dtype=BF16, device=DEV)
    ws = torch.empty(api.cc_attn_fused_workspace_bytes(t, hw), dtype=torch.uint8, device=DEV)
    api.cc_attn_frame_fused(q, k, v, o, ws)
    api.cc_check_device()
    return o


@pytest.mark.parametrize("t,hw,c", [(2, 200, 256), (1, 130, 256), (1, 1, 256), (3, 64, 256), (2, 333, 1024),
                                    (1, 256, 256), (1, 257, 512), (1, 512, 256), (2, 700, 256), (1, 4200, 256)])
def test_attn_fused_small(t, hw, c):
    inp = inputs.attn_inputs(t, hw, c, seed=71, device=DEV)
    o = run_fused(inp["q"], inp["k"], inp["v"])
    ref = oracle.attn_frame(to_np(inp["q"]), to_np(inp["k"]), to_np(inp["v"]))
    assert_parity(to_np(o), ref, f"fused attention {t,hw,c}")


@pytest.mark.parametrize("gain", [4.0, 8.0])
def test_attn_fused_peaked_rows(gain):
    t, hw, c = 2, 900, 256
    inp = inputs.attn_inputs(t, hw, c, seed=72, device=DEV)
    q = (inp["q"].float() * gain).to(BF16)
    k = (inp["k"].float() * gain).to(BF16)
    o = run_fused(q, k, inp["v"])
    ref = oracle.attn_frame(to_np(q), to_np(k), to_np(inp["v"]))
    assert_parity(to_np(o), ref, f"fused attention, peaked x{gain}")


def test_attn_fused_packed_qkv_layout():
    t, hw, c = 2, 300, 256
    g = torch.Generator(device=DEV).manual_seed(73)
    qkv = torch.randn((t, hw, 3 * c), generator=g, device=DEV).to(BF16)
    q, k, v = qkv[..., :c], qkv[..., c:2 * c], qkv[..., 2 * c:]
    o = run_fused(q, k, v)
    ref = oracle.attn_frame(to_np(q), to_np(k), to_np(v))
    assert_parity(to_np(o), ref, "fused attention, packed qkv")


def test_attn_fused_close_to_the_numerators_path():
    # the same rounding points (E once, O once) as the key-tile path
    t, hw, c = 2, 1000, 512
    inp = inputs.attn_inputs(t, hw, c, seed=74, device=DEV)
    o = run_fused(inp["q"], inp["k"], inp["v"])
    o2 = torch.empty_like(o)
    ws = torch.empty(api.cc_attn_exp_workspace_bytes(t, hw), dtype=torch.uint8, device=DEV)
    api.cc_attn_frame_exp(inp["q"], inp["k"], inp["v"], o2, ws)
    api.cc_check_device()
    ref = oracle.attn_frame(to_np(inp["q"]), to_np(inp["k"]), to_np(inp["v"]))
    p_fused = assert_parity(to_np(o), ref, "fused")
    p_exp = assert_parity(to_np(o2), ref, "key tiles")
    assert p_fused["rel_l2"] < 1.5 * p_exp["rel_l2"] + 1e-4


def test_attn_scores_stats_equal_the_numerators_kernels():
    t, hw, c = 2, 600, 256
    inp = inputs.attn_inputs(t, hw, c, seed=75, device=DEV)
    tiles = api.cc_attn_exp_key_tiles(hw)
    st1 = torch.zeros((t, hw, tiles, 2), dtype=torch.float32, device=DEV)
    st2 = torch.zeros_like(st1)
    e = torch.zeros((t, hw, api.cc_attn_ld(hw)), dtype=BF16, device=DEV)
    api.cc_attn_scores_stats(inp["q"], inp["k"], st1)
    api.cc_attn_scores_exp(inp["q"], inp["k"], e, st2)
    api.cc_check_device()
    assert torch.equal(st1, st2)


def test_attn_fused_config_sampled():
    c = inputs.CONFIGS["attention"]
    inp = inputs.make_config_inputs("attention", device=DEV)
    o = run_fused(inp["q"], inp["k"], inp["v"])
    rng = np.random.default_rng(7)
    rows = [(t, i) for t in range(c.d) for i in (0, 127, 128, 255, 256, 3327, 3328, c.hw - 1)]
    rows += [(int(rng.integers(c.d)), int(rng.integers(c.hw))) for _ in range(48)]
    rows = np.array(rows)
    ref = oracle.attn_frame_rows(to_np(inp["q"]), to_np(inp["k"]), to_np(inp["v"]), rows)
    assert_parity(to_np(o)[rows[:, 0], rows[:, 1]], ref, "fused attention sampled")


def test_attn_fused_rejects_channels_not_a_multiple_of_256():
    x = torch.zeros((1, 64, 192), dtype=BF16, device=DEV)
    ws = torch.empty(api.cc_attn_fused_workspace_bytes(1, 64), dtype=torch.uint8, device=DEV)
    with pytest.raises(api.CCError) as e:
        api.cc_attn_frame_fused(x, x, x, torch.empty_like(x), ws)
    assert e.value.status == 2
    api.cc_check_device()
