"""Attention through the key-tile numerators (cc_attn_scores_exp ->
cc_attn_exp_rescale -> cc_attn_pv_exp): the scores kernel writes
E = exp2(kx*S - c_t) per 256-key tile with the row statistics (c_t, l_t), the
rescale pass puts every tile of a row on the row's largest c_t by exact
powers of two, and the PV kernel divides each output row by the row sum.
Checked against the fp64 oracle's softmax attention, with every intermediate
checked against its definition."""

import numpy as np
import pytest
import torch

import oracle
from causal_convolution_gb300 import api, inputs
from gpu_util import assert_parity, ensure_built, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF16 = torch.bfloat16
LOG2E = 1.4426950408889634


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    return ensure_built()


def run_exp(q, k, v):
    t, hw, c = q.shape
    o = torch.empty((t, hw, c), dtype=BF16, device=DEV)
    ws = torch.empty(api.cc_attn_exp_workspace_bytes(t, hw), dtype=torch.uint8, device=DEV)
    api.cc_attn_frame_exp(q, k, v, o, ws)
    api.cc_check_device()
    return o


def scaled_inputs(t, hw, c, seed, gain):
    inp = inputs.attn_inputs(t, hw, c, seed=seed, device=DEV)
    return {n: (x.float() * gain).to(BF16) if n in ("q", "k") else x for n, x in inp.items()}


@pytest.mark.parametrize("t,hw,c", [(2, 200, 64), (1, 130, 128), (3, 64, 64), (1, 1, 64), (2, 333, 1024),
                                    (1, 256, 64), (1, 257, 64), (1, 512, 128), (2, 700, 128), (1, 4200, 64),
                                    (5, 8, 64), (1, 129, 192)])
def test_attn_exp_small(t, hw, c):
    inp = inputs.attn_inputs(t, hw, c, seed=41, device=DEV)
    o = run_exp(inp["q"], inp["k"], inp["v"])
    ref = oracle.attn_frame(to_np(inp["q"]), to_np(inp["k"]), to_np(inp["v"]))
    assert_parity(to_np(o), ref, f"attention (key tiles) {t,hw,c}")


def test_attn_exp_intermediates():
    t, hw, c = 2, 600, 128
    inp = scaled_inputs(t, hw, c, 42, 2.0)
    # the keys of the second tile three times larger: its maxima sit a grain
    # (32 in log2 units) above the others' in most rows, so step 2 has tiles
    # to move
    inp["k"][:, 256:512] = (inp["k"][:, 256:512].float() * 3.0).to(BF16)
    tiles = api.cc_attn_exp_key_tiles(hw)
    assert tiles == 3
    ld = api.cc_attn_ld(hw)
    e = torch.zeros((t, hw, ld), dtype=BF16, device=DEV)
    stats = torch.zeros((t, hw, tiles, 2), dtype=torch.float32, device=DEV)
    scale = c ** -0.5
    api.cc_attn_scores_exp(inp["q"], inp["k"], e, stats, scale)
    api.cc_check_device()
    e1, st1 = to_np(e).astype(np.float64), to_np(stats).astype(np.float64)
    api.cc_attn_exp_rescale(e, stats, hw)
    api.cc_check_device()
    e2, st2 = to_np(e).astype(np.float64), to_np(stats).astype(np.float64)
    o = torch.empty((t, hw, c), dtype=BF16, device=DEV)
    api.cc_attn_pv_exp(e, stats, inp["v"], o)
    api.cc_check_device()

    # step 1 against fp64 scores
    qn, kn, vn = (to_np(inp[n]).astype(np.float64) for n in ("q", "k", "v"))
    z = np.einsum("tic,tjc->tij", qn, kn) * (scale * LOG2E)  # kx * S
    ct, lt = st1[..., 0], st1[..., 1]
    for ti in range(tiles):
        cols = slice(256 * ti, min(hw, 256 * (ti + 1)))
        zmax = z[:, :, cols].max(axis=2)
        # c_t = the tile max rounded up to a multiple of 32 (the GPU's fp32
        # scores may land the other side of a multiple only when the max is
        # that close to it)
        assert np.all(ct[:, :, ti] % 32 == 0)
        assert np.all(ct[:, :, ti] >= zmax - 1e-3) and np.all(ct[:, :, ti] < zmax + 32 + 1e-3)
        ex = np.exp2(z[:, :, cols] - ct[:, :, ti:ti + 1])
        assert np.all(ex <= 1 + 1e-3)
        np.testing.assert_allclose(lt[:, :, ti], ex.sum(axis=2), rtol=1e-4)
        # one bf16 rounding of each numerator
        assert np.all(np.abs(e1[:, :, cols] - ex) <= 2.0 ** -8 * ex + 1e-30)

    # step 2: exact powers of two, statistics moved to the row's largest c_t
    c_row = ct.max(axis=2, keepdims=True)
    alpha = np.exp2(ct - c_row)
    assert np.any(alpha < 1), "no tile needed a rescale: the case does not exercise step 2"
    a_keys = np.repeat(alpha, 256, axis=2)[:, :, :hw]
    want = e1[:, :, :hw] * a_keys
    normal = want >= 2.0 ** -126  # products below the normal range may flush
    assert np.array_equal(e2[:, :, :hw][normal], want[normal])
    assert np.all(e2[:, :, :hw][~normal] <= 2.0 ** -126)
    assert np.array_equal(st2[..., 0], np.broadcast_to(c_row, ct.shape))
    np.testing.assert_allclose(st2[..., 1], lt * alpha, rtol=1e-6)

    # the softmax the three steps realise together
    p = e2[:, :, :hw] / st2[..., 1].sum(axis=2)[:, :, None]
    assert_parity(p, oracle.attn_probs(to_np(inp["q"]), to_np(inp["k"])), "probabilities from E")
    # step 3 from the GPU's own E and statistics
    assert_parity(to_np(o), np.einsum("tij,tjc->tic", p, vn), "pv with row scale", rel_l2=2e-3)


@pytest.mark.parametrize("gain", [4.0, 8.0])
def test_attn_exp_peaked_rows(gain):
    # scores of a few hundred: tile maxima many powers of two apart, so the
    # rescale scales most tiles (some to zero) and the softmax is near one-hot
    t, hw, c = 2, 900, 128
    inp = scaled_inputs(t, hw, c, 43, gain)
    o = run_exp(inp["q"], inp["k"], inp["v"])
    ref = oracle.attn_frame(to_np(inp["q"]), to_np(inp["k"]), to_np(inp["v"]))
    assert_parity(to_np(o), ref, f"peaked attention x{gain}")


def test_attn_exp_same_as_unfused_path():
    t, hw, c = 2, 1000, 256
    inp = inputs.attn_inputs(t, hw, c, seed=44, device=DEV)
    o = run_exp(inp["q"], inp["k"], inp["v"])
    o2 = torch.empty_like(o)
    ws = torch.empty(api.cc_attn_workspace_bytes(t, hw), dtype=torch.uint8, device=DEV)
    api.cc_attn_frame(inp["q"], inp["k"], inp["v"], o2, ws)
    api.cc_check_device()
    ref = oracle.attn_frame(to_np(inp["q"]), to_np(inp["k"]), to_np(inp["v"]))
    p_exp = assert_parity(to_np(o), ref, "key tiles")
    p_unf = assert_parity(to_np(o2), ref, "unfused")
    # same rounding points (E once, O once): errors of the same size
    assert p_exp["rel_l2"] < 2 * p_unf["rel_l2"] + 1e-4


def test_attn_exp_packed_qkv_layout():
    t, hw, c = 2, 300, 128
    g = torch.Generator(device=DEV).manual_seed(5)
    qkv = torch.randn((t, hw, 3 * c), generator=g, device=DEV).to(BF16)
    q, k, v = qkv[..., :c], qkv[..., c:2 * c], qkv[..., 2 * c:]
    o = run_exp(q, k, v)
    ref = oracle.attn_frame(to_np(q), to_np(k), to_np(v))
    assert_parity(to_np(o), ref, "packed qkv (key tiles)")


def test_attn_exp_config_sampled():
    c = inputs.CONFIGS["attention"]
    inp = inputs.make_config_inputs("attention", device=DEV)
    o = run_exp(inp["q"], inp["k"], inp["v"])
    rng = np.random.default_rng(4)
    rows = [(t, i) for t in range(c.d) for i in (0, 127, 128, 255, 256, c.hw - 1)]
    rows += [(int(rng.integers(c.d)), int(rng.integers(c.hw))) for _ in range(48)]
    rows = np.array(rows)
    ref = oracle.attn_frame_rows(to_np(inp["q"]), to_np(inp["k"]), to_np(inp["v"]), rows)
    assert_parity(to_np(o)[rows[:, 0], rows[:, 1]], ref, "attention (key tiles) sampled")
