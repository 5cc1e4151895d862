"""Pins of the fp64 oracle against things other than itself.

Each test fixes the oracle to brute-force loops, a library routine, a closed
form or an invariant of the definitions, chosen so that a plausible slip in
the oracle (a dropped tap, a wrong sign or offset, a transposed weight, a
softmax over the wrong axis) fails at least one of them.
"""

import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

RNG = np.random.default_rng(12345)


def rnd(*shape):
    return RNG.standard_normal(shape)


# ---------------------------------------------------------------- conv ----

def brute_conv(x, w, b):
    """Pure-Python loops over the causal 3x3x3 definition (separate code)."""
    n, d, h, wd, cin = x.shape
    cout = w.shape[0]
    y = [[[[[0.0] * cout for _ in range(wd)] for _ in range(h)] for _ in range(d)] for _ in range(n)]
    for nn, t, hh, ww, co in itertools.product(range(n), range(d), range(h), range(wd), range(cout)):
        acc = float(b[co])
        for ci, kt, kh, kw in itertools.product(range(cin), range(3), range(3), range(3)):
            ts, hs, ws = t + kt - 2, hh + kh - 1, ww + kw - 1
            if ts < 0 or hs < 0 or hs >= h or ws < 0 or ws >= wd:
                continue
            acc += float(w[co, ci, kt, kh, kw]) * float(x[nn, ts, hs, ws, ci])
        y[nn][t][hh][ww][co] = acc
    return np.array(y)


def torch_conv(x, w, b):
    """Library routine: torch conv3d (cross-correlation) on the causally padded input."""
    xt = torch.from_numpy(np.ascontiguousarray(x)).permute(0, 4, 1, 2, 3)
    xt = F.pad(xt, (1, 1, 1, 1, 2, 0))
    y = F.conv3d(xt, torch.from_numpy(w), None if b is None else torch.from_numpy(b))
    return y.permute(0, 2, 3, 4, 1).numpy()


def test_conv_brute_force_2x3x4():
    x = rnd(1, 2, 3, 4, 2)
    w = rnd(3, 2, 3, 3, 3)  # Cout != Cin catches a transposed weight
    b = rnd(3)
    np.testing.assert_allclose(oracle.causal_conv3d(x, w, b), brute_conv(x, w, b), rtol=0, atol=1e-12)


def test_conv_brute_force_batch2():
    x = rnd(2, 3, 2, 3, 2)
    w = rnd(2, 2, 3, 3, 3)
    b = rnd(2)
    np.testing.assert_allclose(oracle.causal_conv3d(x, w, b), brute_conv(x, w, b), rtol=0, atol=1e-12)


def test_conv_matches_torch_conv3d():
    x = rnd(1, 4, 5, 6, 8)
    w = rnd(6, 8, 3, 3, 3)
    b = rnd(6)
    np.testing.assert_allclose(oracle.causal_conv3d(x, w, b), torch_conv(x, w, b), rtol=0, atol=1e-11)


def test_conv_identity_tap():
    # only tap (kt=2, kh=1, kw=1) set to the identity: reads frame t itself
    c = 5
    x = rnd(1, 3, 4, 5, c)
    w = np.zeros((c, c, 3, 3, 3))
    w[:, :, 2, 1, 1] = np.eye(c)
    np.testing.assert_array_equal(oracle.causal_conv3d(x, w, None), x)


def test_conv_centre_tap_is_one_frame_delay():
    # the literal centre tap (1,1,1) reads frame t-1 under causal alignment
    c = 3
    x = rnd(1, 4, 3, 3, c)
    w = np.zeros((c, c, 3, 3, 3))
    w[:, :, 1, 1, 1] = np.eye(c)
    y = oracle.causal_conv3d(x, w, None)
    np.testing.assert_array_equal(y[:, 0], 0.0)
    np.testing.assert_array_equal(y[:, 1:], x[:, :-1])


def test_conv_shift_taps_move_the_right_way():
    # tap (2, 0, 2) reads x[t, h-1, w+1]
    c = 2
    x = rnd(1, 2, 4, 5, c)
    w = np.zeros((c, c, 3, 3, 3))
    w[:, :, 2, 0, 2] = np.eye(c)
    y = oracle.causal_conv3d(x, w, None)
    np.testing.assert_array_equal(y[:, :, 1:, :-1], x[:, :, :-1, 1:])
    np.testing.assert_array_equal(y[:, :, 0], 0.0)
    np.testing.assert_array_equal(y[:, :, :, -1], 0.0)


def test_conv_constant_input_closed_form():
    # x == 1: interior output = b + sum of all weights; a corner of frame 0
    # sees only kt=2 and the 2x2 in-plane taps
    x = np.ones((1, 3, 4, 4, 2))
    w = rnd(3, 2, 3, 3, 3)
    b = rnd(3)
    y = oracle.causal_conv3d(x, w, b)
    np.testing.assert_allclose(y[0, 2, 1, 1], b + w.sum(axis=(1, 2, 3, 4)), atol=1e-12)
    np.testing.assert_allclose(y[0, 0, 0, 0], b + w[:, :, 2, 1:, 1:].sum(axis=(1, 2, 3)), atol=1e-12)


def test_conv_causality():
    x = rnd(1, 5, 3, 4, 3)
    w = rnd(3, 3, 3, 3, 3)
    b = rnd(3)
    y0 = oracle.causal_conv3d(x, w, b)
    x2 = x.copy()
    x2[:, 3] += 1.0
    y1 = oracle.causal_conv3d(x2, w, b)
    np.testing.assert_array_equal(y0[:, :3], y1[:, :3])
    assert np.abs(y0[:, 3] - y1[:, 3]).max() > 1e-3


def test_conv_linearity():
    x1, x2 = rnd(1, 2, 3, 3, 2), rnd(1, 2, 3, 3, 2)
    w1, w2 = rnd(2, 2, 3, 3, 3), rnd(2, 2, 3, 3, 3)
    f = lambda x, w: oracle.causal_conv3d(x, w, None)
    np.testing.assert_allclose(f(2 * x1 - x2, w1), 2 * f(x1, w1) - f(x2, w1), atol=1e-12)
    np.testing.assert_allclose(f(x1, w1 + 3 * w2), f(x1, w1) + 3 * f(x1, w2), atol=1e-12)


def test_conv_history_frames_are_the_frames_before():
    x = rnd(1, 3, 3, 4, 2)
    hist = rnd(1, 2, 3, 4, 2)
    w = rnd(2, 2, 3, 3, 3)
    b = rnd(2)
    full = oracle.causal_conv3d(np.concatenate([hist, x], axis=1), w, b)
    np.testing.assert_allclose(oracle.causal_conv3d(x, w, b, history=hist), full[:, 2:], atol=1e-12)


def test_conv_sampled_matches_full():
    x = rnd(2, 3, 4, 5, 4)
    w = rnd(3, 4, 3, 3, 3)
    b = rnd(3)
    hist = rnd(2, 2, 4, 5, 4)
    pts = np.array(list(itertools.product(range(2), range(3), range(4), range(5))))
    for hh in (None, hist):
        full = oracle.causal_conv3d(x, w, b, history=hh)
        at = oracle.causal_conv3d_at(x, w, b, pts, history=hh)
        np.testing.assert_allclose(at, full[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]], atol=1e-12)


# ----------------------------------------------------------- resampler ----

def torch_resample(x, w, b, s):
    """Library routines: nearest interpolate x2 in (h, w), torch conv3d, then the shortcut."""
    up = lambda a: F.interpolate(torch.from_numpy(a).permute(0, 4, 1, 2, 3), scale_factor=(1, 2, 2), mode="nearest")
    y = F.conv3d(F.pad(up(x), (1, 1, 1, 1, 2, 0)), torch.from_numpy(w), torch.from_numpy(b)) + up(s)
    return y.permute(0, 2, 3, 4, 1).numpy()


def test_resample_direct_matches_torch():
    x, s = rnd(1, 2, 3, 4, 4), rnd(1, 2, 3, 4, 4)
    w, b = rnd(4, 4, 3, 3, 3), rnd(4)
    np.testing.assert_allclose(oracle.resample_up2(x, w, b, s), torch_resample(x, w, b, s), atol=1e-11)


def test_resample_four_phase_matches_direct_toy():
    # the toy configuration's shapes: [1,64,2,8,12] -> [1,64,2,16,24]
    x, s = rnd(1, 2, 8, 12, 64), rnd(1, 2, 8, 12, 64)
    w, b = rnd(64, 64, 3, 3, 3) / math.sqrt(27 * 64), rnd(64)
    direct = oracle.resample_up2(x, w, b, s)
    assert direct.shape == (1, 2, 16, 24, 64)
    np.testing.assert_allclose(oracle.resample_up2_four_phase(x, w, b, s), direct, rtol=0, atol=1e-12)


def test_resample_phase_kernels_sum_every_tap_once():
    # over the four phases each original tap appears exactly 4 times in total
    # (once per phase), so summing all phase kernels gives 4 x the row/col sums
    w = rnd(3, 2, 3, 3, 3)
    pk = oracle.resample_phase_kernels(w)
    np.testing.assert_allclose(pk.sum(axis=(0, 4, 5)), 4 * w.sum(axis=(3, 4)), atol=1e-12)
    # phase (0,0), tap (a=1,b=1) sums the lower-right 2x2 block
    np.testing.assert_allclose(pk[0, :, :, :, 1, 1], w[:, :, :, 1:, 1:].sum(axis=(3, 4)), atol=1e-12)


def test_resample_identity_tap():
    c = 4
    x, s = rnd(1, 2, 3, 5, c), rnd(1, 2, 3, 5, c)
    w = np.zeros((c, c, 3, 3, 3))
    w[:, :, 2, 1, 1] = np.eye(c)
    b = rnd(c)
    up = lambda a: np.repeat(np.repeat(a, 2, axis=2), 2, axis=3)
    np.testing.assert_allclose(oracle.resample_up2(x, w, b, s), up(x) + b + up(s), atol=1e-12)
    np.testing.assert_allclose(oracle.resample_up2_four_phase(x, w, b, s), up(x) + b + up(s), atol=1e-12)


def test_resample_sampled_matches_full():
    x, s = rnd(1, 3, 3, 4, 3), rnd(1, 3, 3, 4, 3)
    w, b = rnd(3, 3, 3, 3, 3), rnd(3)
    full = oracle.resample_up2(x, w, b, s)
    pts = np.array(list(itertools.product(range(1), range(3), range(6), range(8))))
    at = oracle.resample_up2_at(x, w, b, s, pts)
    np.testing.assert_allclose(at, full[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]], atol=1e-12)


# ----------------------------------------------------------- attention ----

def brute_attn(q, k, v, scale):
    t, hw, c = q.shape
    out = np.zeros_like(q)
    for f in range(t):
        for i in range(hw):
            s = [sum(q[f, i, cc] * k[f, j, cc] for cc in range(c)) * scale for j in range(hw)]
            m = max(s)
            e = [math.exp(sj - m) for sj in s]
            z = sum(e)
            for cc in range(c):
                out[f, i, cc] = sum(e[j] / z * v[f, j, cc] for j in range(hw))
    return out


def test_attn_brute_force_hw5_c4():
    q, k, v = rnd(2, 5, 4), rnd(2, 5, 4), rnd(2, 5, 4)
    np.testing.assert_allclose(oracle.attn_frame(q, k, v), brute_attn(q, k, v, 0.5), atol=1e-12)


def test_attn_matches_torch_sdpa():
    q, k, v = rnd(3, 37, 16), rnd(3, 37, 16), rnd(3, 37, 16)
    ref = F.scaled_dot_product_attention(*(torch.from_numpy(a)[None] for a in (q, k, v)))[0].numpy()
    np.testing.assert_allclose(oracle.attn_frame(q, k, v), ref, atol=1e-12)


def test_attn_rows_sum_to_one_and_scale_default():
    q, k = rnd(2, 33, 64) * 4, rnd(2, 33, 64) * 4
    p = oracle.attn_probs(q, k)
    np.testing.assert_allclose(p.sum(axis=-1), 1.0, atol=1e-12)
    assert (p >= 0).all()
    # the default scale is 1/sqrt(C): 1/8 here
    np.testing.assert_allclose(p, oracle.attn_probs(q, k, 1.0 / 8.0), atol=0)
    # softmax is over keys: P[i, :] depends on q_i only
    q2 = q.copy()
    q2[:, 5] += 1.0
    p2 = oracle.attn_probs(q2, k)
    np.testing.assert_array_equal(np.delete(p, 5, axis=1), np.delete(p2, 5, axis=1))


def test_attn_zero_query_gives_mean_of_values():
    q, k, v = np.zeros((2, 11, 8)), rnd(2, 11, 8), rnd(2, 11, 8)
    o = oracle.attn_frame(q, k, v)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=1, keepdims=True), o.shape), atol=1e-12)


def test_attn_constant_values_give_constant_output():
    q, k = rnd(1, 9, 8), rnd(1, 9, 8)
    v = np.full((1, 9, 8), 0.37)
    np.testing.assert_allclose(oracle.attn_frame(q, k, v), 0.37, atol=1e-12)


def test_attn_key_value_permutation_invariance():
    q, k, v = rnd(1, 13, 8), rnd(1, 13, 8), rnd(1, 13, 8)
    perm = RNG.permutation(13)
    np.testing.assert_allclose(oracle.attn_frame(q, k[:, perm], v[:, perm]), oracle.attn_frame(q, k, v), atol=1e-12)


def test_attn_rows_sampled_matches_full():
    q, k, v = rnd(2, 17, 8), rnd(2, 17, 8), rnd(2, 17, 8)
    rows = np.array([[0, 0], [1, 16], [1, 3]])
    np.testing.assert_allclose(oracle.attn_frame_rows(q, k, v, rows), oracle.attn_frame(q, k, v)[rows[:, 0], rows[:, 1]], atol=1e-12)


# ---------------------------------------------------------------- head ----

def test_head_matches_torch_conv_clamp():
    x = rnd(1, 3, 5, 6, 16) * 3
    w, b = rnd(12, 16, 3, 3, 3), rnd(12)
    np.testing.assert_allclose(oracle.head_out(x, w, b), np.clip(torch_conv(x, w, b), -1, 1), atol=1e-11)


def test_head_two_stage_equals_direct():
    x = rnd(1, 3, 5, 6, 16)
    w, b = rnd(12, 16, 3, 3, 3) * 0.05, rnd(12) * 0.1
    np.testing.assert_allclose(oracle.head_two_stage(x, w, b), oracle.head_out(x, w, b), rtol=0, atol=1e-12)


def test_head_zero_weight_gives_clamped_bias():
    x = rnd(1, 2, 3, 3, 8)
    b = np.array([-3.0, -1.0, -0.5, 0.0, 0.25, 1.0, 2.0, 0.9, -0.9, 5.0, -5.0, 0.1])
    y = oracle.head_out(x, np.zeros((12, 8, 3, 3, 3)), b)
    np.testing.assert_array_equal(y, np.broadcast_to(np.clip(b, -1, 1), y.shape))


def test_head_output_is_bounded():
    x = rnd(1, 2, 4, 4, 8) * 10
    y = oracle.head_out(x, rnd(12, 8, 3, 3, 3), rnd(12))
    assert np.abs(y).max() <= 1.0
    assert (np.abs(y) == 1.0).any()


def test_head_sampled_matches_full():
    x = rnd(1, 3, 4, 5, 8)
    w, b = rnd(12, 8, 3, 3, 3) * 0.1, rnd(12) * 0.1
    pts = np.array(list(itertools.product(range(1), range(3), range(4), range(5))))
    np.testing.assert_allclose(oracle.head_out_at(x, w, b, pts), oracle.head_out(x, w, b)[0].reshape(-1, 12), atol=1e-12)


def test_resample_four_phase_matches_direct_with_history():
    x, s, hist = rnd(1, 2, 3, 4, 6), rnd(1, 2, 3, 4, 6), rnd(1, 2, 3, 4, 6)
    w, b = rnd(5, 6, 3, 3, 3), rnd(5)
    s = rnd(1, 2, 3, 4, 5)
    np.testing.assert_allclose(oracle.resample_up2_four_phase(x, w, b, s, history=hist),
                               oracle.resample_up2(x, w, b, s, history=hist), rtol=0, atol=1e-12)


def test_head_two_stage_equals_direct_with_history():
    x, hist = rnd(1, 2, 4, 5, 8), rnd(1, 2, 4, 5, 8)
    w, b = rnd(12, 8, 3, 3, 3) * 0.05, rnd(12) * 0.1
    np.testing.assert_allclose(oracle.head_two_stage(x, w, b, history=hist), oracle.head_out(x, w, b, history=hist),
                               rtol=0, atol=1e-12)


def test_interleave_places_each_phase_on_its_parity():
    ph = rnd(4, 1, 2, 3, 4, 2)
    b, s = rnd(2), rnd(1, 2, 3, 4, 2)
    out = oracle.resample_interleave(ph, b, s)
    # output row 2i+1, column 2j is phase 2*1+0 = 2
    np.testing.assert_array_equal(out[0, 1, 2 * 2 + 1, 2 * 3, :], ph[2, 0, 1, 2, 3] + b + s[0, 1, 2, 3])
    np.testing.assert_array_equal(out[0, 0, 0, 1, :], ph[1, 0, 0, 0, 0] + b + s[0, 0, 0, 0])


# ------------------------------------------------- temporal resampler ----

def torch_resample_temporal(x, w, b, s):
    """Library routines: nearest interpolate x2 in (t, h, w), torch conv3d, shortcut likewise."""
    up = lambda a: F.interpolate(torch.from_numpy(a).permute(0, 4, 1, 2, 3), scale_factor=(2, 2, 2), mode="nearest")
    y = F.conv3d(F.pad(up(x), (1, 1, 1, 1, 2, 0)), torch.from_numpy(w), torch.from_numpy(b)) + up(s)
    return y.permute(0, 2, 3, 4, 1).numpy()


def test_resample_temporal_direct_matches_torch():
    x, s = rnd(1, 3, 3, 4, 4), rnd(1, 3, 3, 4, 4)
    w, b = rnd(4, 4, 3, 3, 3), rnd(4)
    got = oracle.resample_up2(x, w, b, s, temporal=True)
    assert got.shape == (1, 6, 6, 8, 4)
    np.testing.assert_allclose(got, torch_resample_temporal(x, w, b, s), atol=1e-11)


def test_resample_temporal_eight_phase_matches_direct():
    x, s = rnd(1, 3, 4, 5, 8), rnd(1, 3, 4, 5, 6)
    w, b = rnd(6, 8, 3, 3, 3), rnd(6)
    hist = rnd(1, 2, 4, 5, 8)
    for hh in (None, hist):
        np.testing.assert_allclose(oracle.resample_up2_temporal_eight_phase(x, w, b, s, history=hh),
                                   oracle.resample_up2(x, w, b, s, history=hh, temporal=True), rtol=0, atol=1e-12)


def test_resample_temporal_history_uses_last_frame_only():
    # nearest x2 in time puts low-resolution frame -1 at both up-sampled frames
    # -2 and -1, so history frame -2 cannot matter
    x, s = rnd(1, 2, 3, 3, 4), rnd(1, 2, 3, 3, 4)
    w, b = rnd(4, 4, 3, 3, 3), rnd(4)
    h1, h2 = rnd(1, 2, 3, 3, 4), rnd(1, 2, 3, 3, 4)
    h2[:, 1] = h1[:, 1]
    np.testing.assert_array_equal(oracle.resample_up2(x, w, b, s, history=h1, temporal=True),
                                  oracle.resample_up2(x, w, b, s, history=h2, temporal=True))
    full = oracle.resample_up2(np.concatenate([h1[:, 1:], x], 1), w, b, np.concatenate([s[:, :1], s], 1),
                               temporal=True)
    np.testing.assert_allclose(oracle.resample_up2(x, w, b, s, history=h1, temporal=True), full[:, 2:], atol=1e-12)


def test_resample_temporal_sampled_matches_full():
    x, s = rnd(1, 2, 3, 4, 3), rnd(1, 2, 3, 4, 3)
    w, b = rnd(3, 3, 3, 3, 3), rnd(3)
    hist = rnd(1, 2, 3, 4, 3)
    pts = np.array(list(itertools.product(range(1), range(4), range(6), range(8))))
    for hh in (None, hist):
        full = oracle.resample_up2(x, w, b, s, history=hh, temporal=True)
        at = oracle.resample_up2_at(x, w, b, s, pts, history=hh, temporal=True)
        np.testing.assert_allclose(at, full[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]], atol=1e-12)
