"""Seeded random shapes through every stage -- the causal conv, the
resampler (fused, spatial and temporal, and in two passes), the head (two
kernels and fused), the attention (three passes, key tiles, fused) --
each checked whole against the fp64 oracle. The shapes are small enough for
the oracle and are drawn once from a fixed generator, so a failure names a
reproducible case: ragged tails, one-row and one-column planes, several
images, partial column tiles, carried history."""

import numpy as np
import pytest
import torch

import oracle
from causal_convolution_gb300 import api
from gpu_util import assert_parity, ensure_built, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF16 = torch.bfloat16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    return ensure_built()


def _rnd(shape, g, scale=1.0):
    return (torch.randn(shape, generator=g, device=DEV) * scale).to(BF16)


def _cases(seed, k, draw):
    rng = np.random.default_rng(seed)
    return [draw(rng) for _ in range(k)]


CONV = _cases(11, 10, lambda r: (int(r.integers(1, 3)), int(r.integers(1, 4)), int(r.integers(1, 13)),
                                 int(r.integers(1, 21)), int(r.choice([64, 128, 192])),
                                 int(r.choice([16, 48, 64, 144, 272])), int(r.choice([0, 2])),
                                 bool(r.integers(0, 2))))
RESAMPLE = _cases(12, 8, lambda r: (int(r.integers(1, 3)), int(r.integers(1, 4)), int(r.integers(1, 11)),
                                    int(r.integers(1, 15)), int(r.choice([64, 128])),
                                    int(r.choice([16, 64, 96, 256])), int(r.choice([0, 2])), bool(r.integers(0, 2))))
HEAD = _cases(13, 8, lambda r: (int(r.integers(1, 3)), int(r.integers(1, 5)), int(r.integers(1, 13)),
                                int(r.integers(1, 31)), int(r.choice([64, 128, 192, 256])), int(r.choice([0, 2]))))
ATTN = _cases(14, 8, lambda r: (int(r.integers(1, 4)), int(r.integers(1, 701)), int(r.choice([64, 128, 192, 256]))))
HEAD_FUSED = _cases(15, 10, lambda r: (int(r.integers(1, 3)), int(r.integers(1, 20)), int(r.integers(1, 14)),
                                       int(r.integers(1, 75)), int(r.choice([64, 128, 192, 256])),
                                       int(r.choice([0, 2]))))
ATTN_FUSED = _cases(16, 8, lambda r: (int(r.integers(1, 4)), int(r.integers(1, 801)), int(r.choice([256, 512]))))
RESAMPLE_TWO_PASS = _cases(17, 6, lambda r: (int(r.integers(1, 3)), int(r.integers(1, 4)), int(r.integers(1, 11)),
                                             int(r.integers(1, 15)), int(r.choice([64, 128])),
                                             int(r.choice([16, 64, 96, 256])), int(r.choice([0, 2]))))
ATTN_THREE_PASS = _cases(18, 6, lambda r: (int(r.integers(1, 4)), int(r.integers(1, 701)),
                                           int(r.choice([64, 128, 192, 256]))))


@pytest.mark.parametrize("n,d,h,w,cin,cout,hist,bias", CONV)
def test_conv_random_shape(n, d, h, w, cin, cout, hist, bias):
    g = torch.Generator(device=DEV).manual_seed(n * 1000 + d * 100 + h * 10 + w)
    x = _rnd((n, d + hist, h, w, cin), g)
    wt = _rnd((cout, cin, 3, 3, 3), g, (27 * cin) ** -0.5)
    b = _rnd((cout,), g, 0.1) if bias else None
    wp = torch.empty(27 * cout * cin, dtype=BF16, device=DEV)
    api.cc_conv3d_prepare(wt, wp)
    y = torch.empty((n, d, h, w, cout), dtype=BF16, device=DEV)
    api.cc_conv3d_causal(x, wp, b, y, hist=hist)
    api.cc_check_device()
    xn = to_np(x)
    ref = oracle.causal_conv3d(xn[:, hist:], to_np(wt), to_np(b) if bias else None,
                               history=xn[:, :2] if hist else None)
    assert_parity(to_np(y), ref, f"conv {n, d, h, w, cin, cout, hist, bias}")


@pytest.mark.parametrize("n,d,hl,wl,cin,cout,hist,temporal", RESAMPLE)
def test_resample_fused_random_shape(n, d, hl, wl, cin, cout, hist, temporal):
    g = torch.Generator(device=DEV).manual_seed(n * 1000 + d * 100 + hl * 10 + wl)
    x = _rnd((n, d + hist, hl, wl, cin), g)
    wt = _rnd((cout, cin, 3, 3, 3), g, (27 * cin) ** -0.5)
    b = _rnd((cout,), g, 0.1)
    skip = _rnd((n, d, hl, wl, cout), g)
    pw = torch.empty((64 if temporal else 48) * cout * cin, dtype=BF16, device=DEV)
    (api.cc_resample_prepare_temporal if temporal else api.cc_resample_prepare)(wt, pw)
    out = torch.empty((n, 2 * d if temporal else d, 2 * hl, 2 * wl, cout), dtype=BF16, device=DEV)
    api.cc_resample_up2_fused(x, pw, b, skip, out, hist=hist, temporal=temporal)
    api.cc_check_device()
    xn = to_np(x)
    ref = oracle.resample_up2(xn[:, hist:], to_np(wt), to_np(b), to_np(skip),
                              history=xn[:, :2] if hist else None, temporal=temporal)
    assert_parity(to_np(out), ref, f"resampler {n, d, hl, wl, cin, cout, hist, temporal}")


@pytest.mark.parametrize("n,d,h,w,cin,hist", HEAD)
def test_head_random_shape(n, d, h, w, cin, hist):
    g = torch.Generator(device=DEV).manual_seed(n * 1000 + d * 100 + h * 10 + w)
    x = _rnd((n, d + hist, h, w, cin), g)
    wt = _rnd((api.HEAD_COUT, cin, 3, 3, 3), g, (27 * cin) ** -0.5)
    b = _rnd((api.HEAD_COUT,), g, 0.2)
    wp = torch.empty(3 * api.HEAD_G_CH * cin, dtype=BF16, device=DEV)
    api.cc_head_prepare(wt, wp)
    out = torch.empty((n, d, h, w, api.HEAD_COUT), dtype=BF16, device=DEV)
    ws = torch.empty(api.cc_head_workspace_bytes(n, d, h, w), dtype=torch.uint8, device=DEV)
    api.cc_head_out(x, wp, b, out, ws, hist=hist)
    api.cc_check_device()
    xn = to_np(x)
    ref = oracle.head_out(xn[:, hist:], to_np(wt), to_np(b), history=xn[:, :2] if hist else None)
    assert_parity(to_np(out), ref, f"head {n, d, h, w, cin, hist}")
    assert float(out.abs().max()) <= 1.0


@pytest.mark.parametrize("t,hw,c", ATTN)
def test_attention_key_tiles_random_shape(t, hw, c):
    g = torch.Generator(device=DEV).manual_seed(t * 10000 + hw * 10 + c)
    q, k, v = (_rnd((t, hw, c), g) for _ in range(3))
    o = torch.empty((t, hw, c), dtype=BF16, device=DEV)
    ws = torch.empty(api.cc_attn_exp_workspace_bytes(t, hw), dtype=torch.uint8, device=DEV)
    api.cc_attn_frame_exp(q, k, v, o, ws)
    api.cc_check_device()
    ref = oracle.attn_frame(to_np(q), to_np(k), to_np(v))
    assert_parity(to_np(o), ref, f"attention {t, hw, c}")


@pytest.mark.parametrize("n,d,h,w,cin,hist", HEAD_FUSED)
def test_head_fused_random_shape(n, d, h, w, cin, hist):
    g = torch.Generator(device=DEV).manual_seed(n * 1000 + d * 100 + h * 10 + w + 7)
    x = _rnd((n, d + hist, h, w, cin), g, 2.0)
    wt = _rnd((api.HEAD_COUT, cin, 3, 3, 3), g, (27 * cin) ** -0.5)
    b = _rnd((api.HEAD_COUT,), g, 0.2)
    wp = torch.empty(3 * api.HEAD_G_CH * cin, dtype=BF16, device=DEV)
    api.cc_head_prepare(wt, wp)
    out = torch.empty((n, d, h, w, api.HEAD_COUT), dtype=BF16, device=DEV)
    api.cc_head_out_fused(x, wp, b, out, hist=hist)
    api.cc_check_device()
    xn = to_np(x)
    ref = oracle.head_out(xn[:, hist:], to_np(wt), to_np(b), history=xn[:, :2] if hist else None)
    assert_parity(to_np(out), ref, f"fused head {n, d, h, w, cin, hist}")


@pytest.mark.parametrize("t,hw,c", ATTN_FUSED)
def test_attention_fused_random_shape(t, hw, c):
    g = torch.Generator(device=DEV).manual_seed(t * 10000 + hw * 10 + c + 3)
    q, k, v = (_rnd((t, hw, c), g) for _ in range(3))
    o = torch.empty((t, hw, c), dtype=BF16, device=DEV)
    ws = torch.empty(api.cc_attn_fused_workspace_bytes(t, hw), dtype=torch.uint8, device=DEV)
    api.cc_attn_frame_fused(q, k, v, o, ws)
    api.cc_check_device()
    ref = oracle.attn_frame(to_np(q), to_np(k), to_np(v))
    assert_parity(to_np(o), ref, f"fused attention {t, hw, c}")


@pytest.mark.parametrize("n,d,hl,wl,cin,cout,hist", RESAMPLE_TWO_PASS)
def test_resample_two_pass_random_shape(n, d, hl, wl, cin, cout, hist):
    g = torch.Generator(device=DEV).manual_seed(n * 1000 + d * 100 + hl * 10 + wl + 11)
    x = _rnd((n, d + hist, hl, wl, cin), g)
    wt = _rnd((cout, cin, 3, 3, 3), g, (27 * cin) ** -0.5)
    b = _rnd((cout,), g, 0.1)
    skip = _rnd((n, d, hl, wl, cout), g)
    pw = torch.empty(48 * cout * cin, dtype=BF16, device=DEV)
    api.cc_resample_prepare(wt, pw)
    out = torch.empty((n, d, 2 * hl, 2 * wl, cout), dtype=BF16, device=DEV)
    ws = torch.empty(api.cc_resample_workspace_bytes(n, d, hl, wl, cout), dtype=torch.uint8, device=DEV)
    api.cc_resample_up2(x, pw, b, skip, out, ws, hist=hist)
    api.cc_check_device()
    xn = to_np(x)
    ref = oracle.resample_up2(xn[:, hist:], to_np(wt), to_np(b), to_np(skip), history=xn[:, :2] if hist else None)
    assert_parity(to_np(out), ref, f"two-pass resampler {n, d, hl, wl, cin, cout, hist}")


@pytest.mark.parametrize("t,hw,c", ATTN_THREE_PASS)
def test_attention_three_pass_random_shape(t, hw, c):
    g = torch.Generator(device=DEV).manual_seed(t * 10000 + hw * 10 + c + 5)
    q, k, v = (_rnd((t, hw, c), g) for _ in range(3))
    o = torch.empty((t, hw, c), dtype=BF16, device=DEV)
    ws = torch.empty(api.cc_attn_workspace_bytes(t, hw), dtype=torch.uint8, device=DEV)
    api.cc_attn_frame(q, k, v, o, ws)
    api.cc_check_device()
    ref = oracle.attn_frame(to_np(q), to_np(k), to_np(v))
    assert_parity(to_np(o), ref, f"three-pass attention {t, hw, c}")
