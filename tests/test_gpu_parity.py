"""GPU parity: every entry point of the C ABI against the fp64 oracle on the
same seeded bf16 inputs.

Small cases run the whole output through the oracle and are shaped to span
several 128-row tiles with a ragged tail (and partial column tiles); the
full-size configurations compare sampled outputs (tile boundaries, every
corner and edge of every frame, and random positions) that the oracle
computes one by one. The bar is the one stated for this stack: relative L2
error <= 4e-3 and max |d| <= 2^-6 * max |ref| per output tensor; pure data
movement (weight repacks) is compared bit for bit.
"""

import numpy as np
import pytest
import torch

import oracle
from causal_convolution_gb300 import api, inputs
from gpu_util import assert_parity, edge_points, ensure_built, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF16 = torch.bfloat16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    return ensure_built()


def empty(*shape, dtype=BF16):
    return torch.empty(shape, dtype=dtype, device=DEV)


# ------------------------------------------------------------ im2col probe --

def im2col_expected(x, lower, upper, start, offsets, c0):
    """128 pixels walked W-fastest through the bounding box from `start`, each
    read at pixel + offsets (zero outside the tensor)."""
    n, d_in, h, w, _ = x.shape
    box = [(lower[0], w - 1 + upper[0]), (lower[1], h - 1 + upper[1]), (lower[2], d_in - 1 + upper[2])]
    pw, ph, pd, pn = start
    out = np.zeros((128, 64), np.float32)
    for p in range(128):
        iw, ih, idd = pw + offsets[0], ph + offsets[1], pd + offsets[2]
        if 0 <= pn < n and 0 <= idd < d_in and 0 <= ih < h and 0 <= iw < w:
            out[p] = x[pn, idd, ih, iw, c0:c0 + 64]
        pw += 1
        if pw > box[0][1]:
            pw = box[0][0]
            ph += 1
        if ph > box[1][1]:
            ph = box[1][0]
            pd += 1
        if pd > box[2][1]:
            pd = box[2][0]
            pn += 1
    return out


@pytest.mark.parametrize("lower,upper,start,offsets,c0", [
    ((-1, -1, -2), (-1, -1, -2), (-1, -1, -2, 0), (0, 0, 0), 0),
    ((-1, -1, -2), (-1, -1, -2), (-1, -1, -2, 0), (2, 1, 2), 64),
    ((-1, -1, -2), (-1, -1, -2), (0, 1, -1, 0), (1, 2, 1), 0),
    ((-1, -1, 0), (-1, -1, -2), (-1, -1, 0, 0), (1, 1, 2), 64),
])
def test_im2col_tile_matches_definition(lower, upper, start, offsets, c0):
    g = torch.Generator(device=DEV).manual_seed(5)
    x = torch.randn((2, 3, 5, 7, 128), generator=g, device=DEV).to(BF16)
    tile = empty(128, 64)
    api.cc_debug_im2col_tile(x, tile, lower, upper, c0, start, offsets)
    api.cc_check_device()
    got = to_np(tile)
    exp = im2col_expected(to_np(x), lower, upper, start, offsets, c0)
    if not np.array_equal(got, exp):
        alt = im2col_expected(to_np(x), lower[::-1], upper[::-1], start, offsets, c0)
        raise AssertionError(f"im2col tile differs from the definition; matches reversed corner order: "
                             f"{np.array_equal(got, alt)}; first bad pixel: {int(np.argmax(np.any(got != exp, 1)))}")


# ------------------------------------------------------------------- conv --

def run_conv(n, d, h, w, cin, cout, hist, seed=11, with_bias=True):
    inp = inputs.conv_inputs(n, d, h, w, cin, cout, seed, device=DEV, history=bool(hist))
    x = torch.cat([inp["hist"], inp["x"]], 1).contiguous() if hist else inp["x"]
    wp = empty(27 * cout * cin)
    api.cc_conv3d_prepare(inp["w"], wp)
    y = empty(n, d, h, w, cout)
    api.cc_conv3d_causal(x, wp, inp["b"] if with_bias else None, y, hist=hist)
    api.cc_check_device()
    return inp, wp, y


def test_conv3d_prepare_is_a_pure_repack():
    inp = inputs.conv_inputs(1, 1, 1, 1, 64, 48, seed=3, device=DEV)
    wp = empty(27 * 48 * 64)
    api.cc_conv3d_prepare(inp["w"], wp)
    ref = inp["w"].permute(2, 3, 4, 0, 1).reshape(-1)
    assert torch.equal(wp.view(torch.int16), ref.contiguous().view(torch.int16))


@pytest.mark.parametrize("n,d,h,w,cin,cout,hist,bias", [
    (1, 3, 5, 9, 64, 64, 0, True),       # 135 rows: two tiles, ragged tail
    (2, 2, 6, 11, 128, 272, 0, True),    # two images; partial column tile (272 = 256 + 16)
    (1, 3, 4, 7, 64, 32, 2, True),       # carried history frames
    (1, 2, 3, 5, 192, 64, 0, False),     # no bias
    (1, 1, 1, 1, 64, 16, 0, True),       # a single position
    (1, 3, 1, 200, 64, 64, 0, True),     # one-row planes: every tap row above and below is padding
    (1, 3, 200, 1, 64, 64, 0, True),     # one-column planes
    (1, 1, 6, 9, 1024, 16, 2, True),     # one frame after two carried frames; K = 27,648, N = 16
])
def test_conv3d_causal_small(n, d, h, w, cin, cout, hist, bias):
    inp, _, y = run_conv(n, d, h, w, cin, cout, hist, with_bias=bias)
    ref = oracle.causal_conv3d(to_np(inp["x"]), to_np(inp["w"]), to_np(inp["b"]) if bias else None,
                               history=to_np(inp["hist"]) if hist else None)
    assert_parity(to_np(y), ref, f"conv {n,d,h,w,cin,cout,hist}")


@pytest.mark.parametrize("n,d,h,w", [
    (2, 3, 8, 20),    # 480 rows per image: 256-row pair tiles straddle frames and the image boundary
    (1, 5, 16, 16),   # 256 rows per frame: every pair tile inside one frame
    (3, 2, 5, 7),     # 70 rows per image: every pair tile spans several images
])
def test_conv3d_zero_history_taps_skipped_per_tile(n, d, h, w):
    # with zero history a pair tile skips the leading taps that read only the
    # zero frames before frame 0 for all of its rows; the result must not
    # change, whatever frames and images the tile spans
    inp, _, y = run_conv(n, d, h, w, 64, 64, 0)
    ref = oracle.causal_conv3d(to_np(inp["x"]), to_np(inp["w"]), to_np(inp["b"]))
    assert_parity(to_np(y), ref, f"conv {n,d,h,w}")


def test_epilogue_with_16_byte_aligned_outputs():
    # outputs (and the shortcut) 16 bytes past a 32-byte boundary: the
    # epilogue falls back from its 32-byte accesses to 16-byte ones
    def shifted(*shape):
        buf = torch.empty(int(np.prod(shape)) + 8, dtype=BF16, device=DEV)
        t = buf[8:].view(*shape)
        assert t.data_ptr() % 32 == 16
        return t

    inp = inputs.conv_inputs(1, 2, 6, 11, 64, 48, seed=21, device=DEV)
    wp = empty(27 * 48 * 64)
    api.cc_conv3d_prepare(inp["w"], wp)
    y = shifted(1, 2, 6, 11, 48)
    api.cc_conv3d_causal(inp["x"], wp, inp["b"], y)
    api.cc_check_device()
    assert_parity(to_np(y), oracle.causal_conv3d(to_np(inp["x"]), to_np(inp["w"]), to_np(inp["b"])), "conv, shifted y")

    r = inputs.resample_inputs(1, 2, 5, 9, 64, seed=22, device=DEV)
    pw = prepare_resample(r["w"])
    skip = shifted(1, 2, 5, 9, 64)
    skip.copy_(r["skip"])
    out = shifted(1, 2, 10, 18, 64)
    api.cc_resample_up2_fused(r["x"], pw, r["b"], skip, out)
    api.cc_check_device()
    ref = oracle.resample_up2(to_np(r["x"]), to_np(r["w"]), to_np(r["b"]), to_np(r["skip"]))
    assert_parity(to_np(out), ref, "fused resampler, shifted out and skip")


def test_conv3d_mid_block_config_sampled():
    c = inputs.CONFIGS["mid_conv"]
    inp = inputs.make_config_inputs("mid_conv", device=DEV)
    wp = empty(27 * c.cout * c.c)
    api.cc_conv3d_prepare(inp["w"], wp)
    y = empty(c.n, c.d, c.h, c.w, c.cout)
    api.cc_conv3d_causal(inp["x"], wp, inp["b"], y)
    api.cc_check_device()
    pts = edge_points(c.n, c.d, c.h, c.w, 160, np.random.default_rng(1))
    ref = oracle.causal_conv3d_at(to_np(inp["x"]), to_np(inp["w"]), to_np(inp["b"]), pts)
    yy = to_np(y)[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]]
    assert_parity(yy, ref, "mid_conv sampled")


def test_conv3d_output_guard_bands_untouched():
    n, d, h, w, cin, cout = 1, 2, 5, 6, 64, 48
    inp = inputs.conv_inputs(n, d, h, w, cin, cout, 4, device=DEV)
    wp = empty(27 * cout * cin)
    api.cc_conv3d_prepare(inp["w"], wp)
    size = n * d * h * w * cout
    guard = 4096
    buf = torch.full((size + 2 * guard,), 12345, dtype=torch.int16, device=DEV)
    y = buf[guard:guard + size].view(BF16).view(n, d, h, w, cout)
    api.cc_conv3d_causal(inp["x"], wp, inp["b"], y)
    api.cc_check_device()
    assert bool((buf[:guard] == 12345).all()) and bool((buf[guard + size:] == 12345).all())
    ref = oracle.causal_conv3d(to_np(inp["x"]), to_np(inp["w"]), to_np(inp["b"]))
    assert_parity(to_np(y), ref, "conv in guarded buffer")


# -------------------------------------------------------------- resampler --

def prepare_resample(w):
    cout, cin = w.shape[:2]
    pw = empty(48 * cout * cin)
    api.cc_resample_prepare(w, pw)
    return pw


def test_resample_prepare_matches_oracle_phase_kernels():
    inp = inputs.resample_inputs(1, 1, 1, 1, 64, seed=8, device=DEV)
    pw = prepare_resample(inp["w"])
    pk = oracle.resample_phase_kernels(to_np(inp["w"]))  # [4, co, ci, kt, a, b]
    ref = pk.transpose(0, 3, 4, 5, 1, 2).reshape(-1)     # [phase][(kt*2+a)*2+b][co][ci]
    got = to_np(pw).astype(np.float64)
    # fp32 sums of at most four bf16 taps, rounded once: within bf16's half ulp
    np.testing.assert_allclose(got, ref, rtol=2.0 ** -8, atol=1e-30)


def run_resample(x, w, b, skip, hist=0):
    n, dd, hl, wl, cin = x.shape
    d = dd - hist
    cout = w.shape[0]
    pw = prepare_resample(w)
    out = empty(n, d, 2 * hl, 2 * wl, cout)
    ws = torch.empty(api.cc_resample_workspace_bytes(n, d, hl, wl, cout), dtype=torch.uint8, device=DEV)
    api.cc_resample_up2(x, pw, b, skip, out, ws, hist=hist)
    api.cc_check_device()
    return pw, out, ws


def test_resample_toy_config_full():
    inp = inputs.make_config_inputs("toy_resampler", device=DEV)
    _, out, _ = run_resample(inp["x"], inp["w"], inp["b"], inp["skip"])
    ref = oracle.resample_up2(to_np(inp["x"]), to_np(inp["w"]), to_np(inp["b"]), to_np(inp["skip"]))
    assert out.shape == (1, 2, 16, 24, 64)
    assert_parity(to_np(out), ref, "toy resampler")


@pytest.mark.parametrize("n,d,hl,wl,cin,cout,hist", [
    (1, 3, 5, 7, 64, 128, 0),
    (2, 2, 3, 4, 128, 64, 2),
    (1, 2, 9, 13, 64, 272, 0),
])
def test_resample_small(n, d, hl, wl, cin, cout, hist):
    g = torch.Generator(device=DEV).manual_seed(21)
    x = torch.randn((n, d + hist, hl, wl, cin), generator=g, device=DEV).to(BF16)
    w = (torch.randn((cout, cin, 3, 3, 3), generator=g, device=DEV) / (27 * cin) ** 0.5).to(BF16)
    b = (torch.randn((cout,), generator=g, device=DEV) * 0.1).to(BF16)
    s = torch.randn((n, d, hl, wl, cout), generator=g, device=DEV).to(BF16)
    _, out, _ = run_resample(x, w, b, s, hist)
    xn = to_np(x)
    ref = oracle.resample_up2(xn[:, hist:], to_np(w), to_np(b), to_np(s), history=xn[:, :2] if hist else None)
    assert_parity(to_np(out), ref, f"resampler {n,d,hl,wl,cin,cout,hist}")


def test_resample_stages_separately():
    n, d, hl, wl, cin, cout = 1, 2, 6, 10, 64, 64
    inp = inputs.resample_inputs(n, d, hl, wl, cin, seed=9, device=DEV)
    pw = prepare_resample(inp["w"])
    phases = empty(4, n, d, hl, wl, cout)
    api.cc_resample_phase_conv(inp["x"], pw, phases)
    api.cc_check_device()
    pk = to_np(pw).reshape(4, 3, 2, 2, cout, cin).transpose(0, 4, 5, 1, 2, 3)
    ref = oracle.resample_phase_conv(to_np(inp["x"]), pk)
    for ph in range(4):
        assert_parity(to_np(phases[ph]), ref[ph], f"phase {ph}")
    out = empty(n, d, 2 * hl, 2 * wl, cout)
    api.cc_resample_interleave(phases, inp["b"], inp["skip"], out)
    api.cc_check_device()
    ref_out = oracle.resample_interleave(to_np(phases), to_np(inp["b"]), to_np(inp["skip"]))
    assert_parity(to_np(out), ref_out, "interleave", rel_l2=3e-3)


def test_resample_config_sampled():
    c = inputs.CONFIGS["resampler"]
    inp = inputs.make_config_inputs("resampler", device=DEV)
    _, out, _ = run_resample(inp["x"], inp["w"], inp["b"], inp["skip"])
    pts = edge_points(c.n, c.d, 2 * c.h, 2 * c.w, 160, np.random.default_rng(2))
    ref = oracle.resample_up2_at(to_np(inp["x"]), to_np(inp["w"]), to_np(inp["b"]), to_np(inp["skip"]), pts)
    got = to_np(out)[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]]
    assert_parity(got, ref, "resampler sampled")


# -------------------------------------------------------------- attention --

def run_attn(q, k, v):
    t, hw, c = q.shape
    o = empty(t, hw, c)
    ws = torch.empty(api.cc_attn_workspace_bytes(t, hw), dtype=torch.uint8, device=DEV)
    api.cc_attn_frame(q, k, v, o, ws)
    api.cc_check_device()
    return o


@pytest.mark.parametrize("t,hw,c", [(2, 200, 64), (1, 130, 128), (3, 64, 64), (1, 1, 64), (2, 333, 1024),
                                    (1, 4200, 64)])
def test_attn_small(t, hw, c):
    inp = inputs.attn_inputs(t, hw, c, seed=31, device=DEV)
    o = run_attn(inp["q"], inp["k"], inp["v"])
    ref = oracle.attn_frame(to_np(inp["q"]), to_np(inp["k"]), to_np(inp["v"]))
    assert_parity(to_np(o), ref, f"attention {t,hw,c}")


def test_attn_packed_qkv_layout():
    t, hw, c = 2, 150, 128
    g = torch.Generator(device=DEV).manual_seed(4)
    qkv = torch.randn((t, hw, 3 * c), generator=g, device=DEV).to(BF16)
    q, k, v = qkv[..., :c], qkv[..., c:2 * c], qkv[..., 2 * c:]
    o = run_attn(q, k, v)
    ref = oracle.attn_frame(to_np(q), to_np(k), to_np(v))
    assert_parity(to_np(o), ref, "packed qkv")


def test_attn_stages_separately():
    t, hw, c = 2, 260, 128
    inp = inputs.attn_inputs(t, hw, c, seed=32, device=DEV)
    ld = api.cc_attn_ld(hw)
    s = empty(t, hw, ld, dtype=torch.float32)
    api.cc_attn_scores(inp["q"], inp["k"], s)
    p = empty(t, hw, ld)
    api.cc_attn_softmax(s, p, hw, c ** -0.5)
    o = empty(t, hw, c)
    api.cc_attn_pv(p, inp["v"], o, hw)
    api.cc_check_device()
    qn, kn, vn = to_np(inp["q"]), to_np(inp["k"]), to_np(inp["v"])
    s_ref = np.einsum("tic,tjc->tij", qn.astype(np.float64), kn.astype(np.float64))
    assert_parity(to_np(s)[:, :, :hw], s_ref, "scores", rel_l2=1e-5, max_frac=1e-5)
    pn = to_np(p)
    assert_parity(pn[:, :, :hw], oracle.attn_probs(qn, kn), "probabilities")
    assert np.all(pn[:, :, hw:] == 0)
    # O from the GPU's own P: isolates the PV product
    o_ref = np.einsum("tij,tjc->tic", pn[:, :, :hw].astype(np.float64), vn.astype(np.float64))
    assert_parity(to_np(o), o_ref, "pv", rel_l2=2e-3)


def test_attn_config_sampled():
    c = inputs.CONFIGS["attention"]
    inp = inputs.make_config_inputs("attention", device=DEV)
    o = run_attn(inp["q"], inp["k"], inp["v"])
    rng = np.random.default_rng(3)
    rows = [(t, i) for t in range(c.d) for i in (0, 127, 128, c.hw - 1)]
    rows += [(int(rng.integers(c.d)), int(rng.integers(c.hw))) for _ in range(48)]
    rows = np.array(rows)
    ref = oracle.attn_frame_rows(to_np(inp["q"]), to_np(inp["k"]), to_np(inp["v"]), rows)
    assert_parity(to_np(o)[rows[:, 0], rows[:, 1]], ref, "attention sampled")


# ------------------------------------------------------------------- head --

def run_head(x, w, b, hist=0):
    n, dd, h, ww, cin = x.shape
    d = dd - hist
    wp = empty(3 * api.HEAD_G_CH * cin)
    api.cc_head_prepare(w, wp)
    out = empty(n, d, h, ww, api.HEAD_COUT)
    ws = torch.empty(api.cc_head_workspace_bytes(n, d, h, ww), dtype=torch.uint8, device=DEV)
    api.cc_head_out(x, wp, b, out, ws, hist=hist)
    api.cc_check_device()
    return wp, out, ws


@pytest.mark.parametrize("n,d,h,w,cin,hist", [
    (1, 3, 10, 14, 64, 0),
    (1, 2, 8, 16, 128, 0),    # plane of 128: frame-interleaved tile order
    (2, 2, 8, 16, 64, 0),
    (1, 2, 5, 9, 64, 2),
])
def test_head_small(n, d, h, w, cin, hist):
    g = torch.Generator(device=DEV).manual_seed(41)
    x = (torch.randn((n, d + hist, h, w, cin), generator=g, device=DEV) * 2).to(BF16)
    wt = (torch.randn((12, cin, 3, 3, 3), generator=g, device=DEV) / (27 * cin) ** 0.5).to(BF16)
    b = (torch.randn((12,), generator=g, device=DEV) * 0.3).to(BF16)
    _, out, _ = run_head(x, wt, b, hist)
    xn = to_np(x)
    ref = oracle.head_out(xn[:, hist:], to_np(wt), to_np(b), history=xn[:, :2] if hist else None)
    assert_parity(to_np(out), ref, f"head {n,d,h,w,cin,hist}")
    assert float(out.abs().max()) <= 1.0


@pytest.mark.parametrize("n,d,h,w,cin,hist", [
    (3, 7, 24, 40, 64, 0),     # 12 tile pairs x 7 frames = 84 items: shares of 1-2 cross tile pairs
    (2, 15, 16, 48, 64, 2),    # 6 x 15 = 90 items, carried history at every share start
    (1, 16, 32, 80, 128, 0),   # 10 x 16 = 160 items, shares of 2-3 frames
])
def test_head_work_split_across_tile_pairs(n, d, h, w, cin, hist):
    # more (tile pair, output frame) items than CTA pairs: shares start and
    # end inside a tile pair's frames and re-read the frames before them.
    # x has the head configuration's unit scale: at twice that scale the bf16
    # g of the two-stage design alone (an fp64 model of its two roundings)
    # puts the largest of ~10^5 outputs 0.017 off, above 2^-6 of the clamped
    # maximum 1.0, whatever the kernel does.
    g = torch.Generator(device=DEV).manual_seed(44)
    x = torch.randn((n, d + hist, h, w, cin), generator=g, device=DEV).to(BF16)
    wt = (torch.randn((12, cin, 3, 3, 3), generator=g, device=DEV) / (27 * cin) ** 0.5).to(BF16)
    b = (torch.randn((12,), generator=g, device=DEV) * 0.3).to(BF16)
    _, out, _ = run_head(x, wt, b, hist)
    xn = to_np(x)
    ref = oracle.head_out(xn[:, hist:], to_np(wt), to_np(b), history=xn[:, :2] if hist else None)
    assert_parity(to_np(out), ref, f"head {n,d,h,w,cin,hist}")


def test_head_stages_separately():
    inp = inputs.head_inputs(1, 2, 6, 9, 64, seed=42, device=DEV)
    wp = empty(3 * api.HEAD_G_CH * 64)
    api.cc_head_prepare(inp["w"], wp)
    gbuf = empty(1, 2, 6, 9, api.HEAD_G_CH)
    api.cc_head_temporal(inp["x"], wp, gbuf)
    api.cc_check_device()
    g_ref = oracle.head_stage_a(to_np(inp["x"]), to_np(inp["w"]))
    gn = to_np(gbuf)
    assert_parity(gn[..., :108], g_ref, "head stage A")
    assert np.all(gn[..., 108:] == 0)
    out = empty(1, 2, 6, 9, 12)
    api.cc_head_stencil(gbuf, inp["b"], out)
    api.cc_check_device()
    assert_parity(to_np(out), oracle.head_stage_b(gn, to_np(inp["b"])), "head stage B", rel_l2=3e-3)


def test_head_prepare_is_a_pure_repack():
    inp = inputs.head_inputs(1, 1, 1, 1, 64, seed=43, device=DEV)
    wp = empty(3 * api.HEAD_G_CH * 64)
    api.cc_head_prepare(inp["w"], wp)
    w = inp["w"]  # [12, cin, 3, 3, 3]
    ref = torch.zeros((3, api.HEAD_G_CH, 64), dtype=BF16, device=DEV)
    ref[:, :108] = w.permute(2, 3, 4, 0, 1).reshape(3, 108, 64)
    assert torch.equal(wp.view(3, api.HEAD_G_CH, 64).view(torch.int16), ref.view(torch.int16))


def test_head_config_sampled():
    c = inputs.CONFIGS["head"]
    inp = inputs.make_config_inputs("head", device=DEV)
    _, out, _ = run_head(inp["x"], inp["w"], inp["b"])
    pts = edge_points(c.n, c.d, c.h, c.w, 400, np.random.default_rng(4))
    ref = oracle.head_out_at(to_np(inp["x"]), to_np(inp["w"]), to_np(inp["b"]), pts)
    got = to_np(out)[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]]
    assert_parity(got, ref, "head sampled")


# --------------------------------------------------------- failure paths --

def test_unsupported_and_invalid_requests_raise():
    x = empty(1, 1, 2, 2, 96)
    wp = empty(27 * 16 * 96)
    y = empty(1, 1, 2, 2, 16)
    with pytest.raises(api.CCError) as e:
        api.cc_conv3d_causal(x, wp, None, y)
    assert e.value.status == 2
    inp = inputs.resample_inputs(1, 1, 2, 2, 64, seed=1, device=DEV)
    pw = prepare_resample(inp["w"])
    out = empty(1, 1, 4, 4, 64)
    ws = torch.empty(16, dtype=torch.uint8, device=DEV)
    with pytest.raises(api.CCError) as e:
        api.cc_resample_up2(inp["x"], pw, inp["b"], inp["skip"], out, ws)
    assert e.value.status == 1
    api.cc_check_device()


def test_empty_tensors_are_a_no_op():
    # zero frames, rows or positions: every entry point returns at once
    wp = empty(27 * 64 * 64)
    api.cc_conv3d_causal(empty(1, 2, 4, 4, 64), wp, None, empty(1, 0, 4, 4, 64), hist=2)
    api.cc_conv3d_causal(empty(0, 3, 4, 4, 64), wp, None, empty(0, 3, 4, 4, 64))
    pw = empty(48 * 64 * 64)
    b, skip = empty(64), empty(1, 3, 0, 4, 64)
    api.cc_resample_up2_fused(empty(1, 3, 0, 4, 64), pw, b, skip, empty(1, 3, 0, 8, 64))
    api.cc_resample_up2(empty(1, 3, 0, 4, 64), pw, b, skip, empty(1, 3, 0, 8, 64),
                        torch.empty(0, dtype=torch.uint8, device=DEV))
    q = empty(2, 0, 64)
    api.cc_attn_frame_exp(q, q, q, empty(2, 0, 64), torch.empty(0, dtype=torch.uint8, device=DEV))
    api.cc_attn_frame(q, q, q, empty(2, 0, 64), torch.empty(0, dtype=torch.uint8, device=DEV))
    hw = empty(3 * api.HEAD_G_CH * 64)
    api.cc_head_out(empty(1, 0, 4, 4, 64), hw, empty(12), empty(1, 0, 4, 4, 12),
                    torch.empty(0, dtype=torch.uint8, device=DEV))
    api.cc_head_out_noalloc(empty(1, 2, 4, 0, 64), hw, empty(12), empty(1, 0, 4, 0, 12), hist=2)
    api.cc_check_device()
    # the library is still usable afterwards
    inp, _, y = run_conv(1, 2, 3, 5, 64, 16, 0)
    assert_parity(to_np(y), oracle.causal_conv3d(to_np(inp["x"]), to_np(inp["w"]), to_np(inp["b"])), "conv after")


def test_kernel_wait_timeout_is_reported_and_cleared():
    api.cc_debug_wait_timeout(2_000_000)
    with pytest.raises(api.CCError) as e:
        api.cc_check_device()
    assert e.value.status == 4
    api.cc_check_device()  # the word was cleared; the context is still usable
    inp, _, y = run_conv(1, 1, 2, 3, 64, 16, 0)
    ref = oracle.causal_conv3d(to_np(inp["x"]), to_np(inp["w"]), to_np(inp["b"]))
    assert_parity(to_np(y), ref, "conv after a timeout")


def test_bad_tile_order_is_reported_and_skipped():
    # entry 0 of the pair tiles' walking order is the pair row tile 0 (rows
    # 0-255: the zero-history tiles of frame 0 come first, in plain order);
    # the self test replaces it by a row tile that does not exist
    n, d, h, w, cin, cout = 1, 3, 16, 32, 64, 64
    inp = inputs.conv_inputs(n, d, h, w, cin, cout, 41, device=DEV)
    wp = empty(27 * cout * cin)
    api.cc_conv3d_prepare(inp["w"], wp)
    y = torch.full((n, d, h, w, cout), float("nan"), dtype=BF16, device=DEV)
    api.cc_debug_conv_bad_tile_order(inp["x"], wp, y, 0)
    with pytest.raises(api.CCError) as e:
        api.cc_check_device()
    assert e.value.status == 5
    api.cc_check_device()  # the word was cleared; the context is still usable
    rows = to_np(y).reshape(-1, cout)
    assert np.isnan(rows[:256]).all(), "the skipped tile's rows were written"
    ref = oracle.causal_conv3d(to_np(inp["x"]), to_np(inp["w"]), None).reshape(-1, cout)
    assert_parity(rows[256:], ref[256:], "conv rows of the other tiles")
    with pytest.raises(api.CCError) as e:
        api.cc_debug_conv_bad_tile_order(inp["x"], wp, y, 6)  # 1536 rows: pair row tiles 0-5
    assert e.value.status == 1
    api.cc_check_device()


# ------------------------------------------------------ fused resampler --

def run_resample_fused(x, w, b, skip, hist=0):
    n, dd, hl, wl, cin = x.shape
    d = dd - hist
    cout = w.shape[0]
    pw = prepare_resample(w)
    out = empty(n, d, 2 * hl, 2 * wl, cout)
    api.cc_resample_up2_fused(x, pw, b, skip, out, hist=hist)
    api.cc_check_device()
    return out


def test_resample_fused_toy_config_full():
    inp = inputs.make_config_inputs("toy_resampler", device=DEV)
    out = run_resample_fused(inp["x"], inp["w"], inp["b"], inp["skip"])
    ref = oracle.resample_up2(to_np(inp["x"]), to_np(inp["w"]), to_np(inp["b"]), to_np(inp["skip"]))
    assert_parity(to_np(out), ref, "toy resampler, fused")


@pytest.mark.parametrize("n,d,hl,wl,cin,cout,hist", [
    (1, 3, 5, 7, 64, 128, 0),
    (2, 2, 3, 4, 128, 64, 2),
    (1, 2, 9, 13, 64, 272, 0),
    (1, 1, 1, 1, 64, 16, 0),     # a single low-resolution pixel (single-CTA path)
    (1, 2, 1, 150, 64, 64, 0),   # one-row low-resolution planes
    (1, 1, 12, 11, 128, 16, 2),  # one frame after two carried frames, N = 16
])
def test_resample_fused_small(n, d, hl, wl, cin, cout, hist):
    g = torch.Generator(device=DEV).manual_seed(22)
    x = torch.randn((n, d + hist, hl, wl, cin), generator=g, device=DEV).to(BF16)
    w = (torch.randn((cout, cin, 3, 3, 3), generator=g, device=DEV) / (27 * cin) ** 0.5).to(BF16)
    b = (torch.randn((cout,), generator=g, device=DEV) * 0.1).to(BF16)
    s = torch.randn((n, d, hl, wl, cout), generator=g, device=DEV).to(BF16)
    out = run_resample_fused(x, w, b, s, hist)
    xn = to_np(x)
    ref = oracle.resample_up2(xn[:, hist:], to_np(w), to_np(b), to_np(s), history=xn[:, :2] if hist else None)
    assert_parity(to_np(out), ref, f"fused resampler {n,d,hl,wl,cin,cout,hist}")


@pytest.mark.parametrize("n,d,hl,wl,temporal", [(2, 3, 8, 20, False), (1, 5, 16, 16, False), (2, 3, 8, 20, True)])
def test_resample_fused_zero_history_taps_skipped_per_tile(n, d, hl, wl, temporal):
    g = torch.Generator(device=DEV).manual_seed(29)
    cin = cout = 64
    x = torch.randn((n, d, hl, wl, cin), generator=g, device=DEV).to(BF16)
    w = (torch.randn((cout, cin, 3, 3, 3), generator=g, device=DEV) / (27 * cin) ** 0.5).to(BF16)
    b = (torch.randn((cout,), generator=g, device=DEV) * 0.1).to(BF16)
    s = torch.randn((n, d, hl, wl, cout), generator=g, device=DEV).to(BF16)
    pw = empty((64 if temporal else 48) * cout * cin)
    (api.cc_resample_prepare_temporal if temporal else api.cc_resample_prepare)(w, pw)
    out = empty(n, 2 * d if temporal else d, 2 * hl, 2 * wl, cout)
    api.cc_resample_up2_fused(x, pw, b, s, out, temporal=temporal)
    api.cc_check_device()
    ref = oracle.resample_up2(to_np(x), to_np(w), to_np(b), to_np(s), temporal=temporal)
    assert_parity(to_np(out), ref, f"fused resampler {n,d,hl,wl,temporal}")


def test_resample_fused_matches_two_pass():
    inp = inputs.resample_inputs(1, 2, 6, 10, 128, seed=23, device=DEV)
    _, two_pass, _ = run_resample(inp["x"], inp["w"], inp["b"], inp["skip"])
    fused = run_resample_fused(inp["x"], inp["w"], inp["b"], inp["skip"])
    # the two-pass path rounds the phases to bf16 once more; both meet the bar
    assert_parity(to_np(fused), to_np(two_pass), "fused vs two-pass", rel_l2=4e-3)


def test_resample_fused_config_sampled():
    c = inputs.CONFIGS["resampler"]
    inp = inputs.make_config_inputs("resampler", device=DEV)
    out = run_resample_fused(inp["x"], inp["w"], inp["b"], inp["skip"])
    pts = edge_points(c.n, c.d, 2 * c.h, 2 * c.w, 160, np.random.default_rng(5))
    ref = oracle.resample_up2_at(to_np(inp["x"]), to_np(inp["w"]), to_np(inp["b"]), to_np(inp["skip"]), pts)
    got = to_np(out)[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]]
    assert_parity(got, ref, "fused resampler sampled")


# --------------------------------------------- temporal resampler (x2 in time) --

def test_resample_prepare_temporal_matches_oracle():
    inp = inputs.resample_inputs(1, 1, 1, 1, 64, seed=24, device=DEV)
    pw = empty(64 * 64 * 64)
    api.cc_resample_prepare_temporal(inp["w"], pw)
    pk = oracle.resample_phase_kernels_temporal(to_np(inp["w"]))  # [8, co, ci, a, b, c]
    ref = pk.transpose(0, 3, 4, 5, 1, 2).reshape(-1)               # [phase][(a*2+b)*2+c][co][ci]
    np.testing.assert_allclose(to_np(pw).astype(np.float64), ref, rtol=2.0 ** -8, atol=1e-30)


def run_resample_temporal(x, w, b, skip, hist=0):
    n, dd, hl, wl, cin = x.shape
    d = dd - hist
    cout = w.shape[0]
    pw = empty(64 * cout * cin)
    api.cc_resample_prepare_temporal(w, pw)
    out = empty(n, 2 * d, 2 * hl, 2 * wl, cout)
    api.cc_resample_up2_fused(x, pw, b, skip, out, hist=hist, temporal=True)
    api.cc_check_device()
    return out


@pytest.mark.parametrize("n,d,hl,wl,cin,cout,hist", [
    (1, 2, 8, 12, 64, 64, 0),
    (1, 3, 5, 7, 64, 128, 2),
    (2, 2, 3, 4, 128, 64, 0),
    (1, 1, 1, 1, 64, 16, 2),
])
def test_resample_temporal_small(n, d, hl, wl, cin, cout, hist):
    g = torch.Generator(device=DEV).manual_seed(25)
    x = torch.randn((n, d + hist, hl, wl, cin), generator=g, device=DEV).to(BF16)
    w = (torch.randn((cout, cin, 3, 3, 3), generator=g, device=DEV) / (27 * cin) ** 0.5).to(BF16)
    b = (torch.randn((cout,), generator=g, device=DEV) * 0.1).to(BF16)
    s = torch.randn((n, d, hl, wl, cout), generator=g, device=DEV).to(BF16)
    out = run_resample_temporal(x, w, b, s, hist)
    xn = to_np(x)
    ref = oracle.resample_up2(xn[:, hist:], to_np(w), to_np(b), to_np(s), history=xn[:, :2] if hist else None,
                              temporal=True)
    assert out.shape == (n, 2 * d, 2 * hl, 2 * wl, cout)
    assert_parity(to_np(out), ref, f"temporal resampler {n,d,hl,wl,cin,cout,hist}")


def test_resample_temporal_sampled_large():
    # an up-block-sized case: 512 channels, 4 latent frames at 44x78 -> 8 x 88x156
    inp = inputs.resample_inputs(1, 4, 44, 78, 512, seed=26, device=DEV)
    out = run_resample_temporal(inp["x"], inp["w"], inp["b"], inp["skip"])
    pts = edge_points(1, 8, 88, 156, 120, np.random.default_rng(6))
    ref = oracle.resample_up2_at(to_np(inp["x"]), to_np(inp["w"]), to_np(inp["b"]), to_np(inp["skip"]), pts,
                                 temporal=True)
    got = to_np(out)[pts[:, 0], pts[:, 1], pts[:, 2], pts[:, 3]]
    assert_parity(got, ref, "temporal resampler sampled")


# ------------------------------------------ chunked streaming with history --
# A long video is decoded in chunks; each chunk after the first carries the
# previous chunk's last two input frames as history (hist = 2). The result
# must equal one call over all frames, bit for bit (same sums in the same order).

def test_conv_chunked_streaming_equals_one_call():
    n, d, h, w, c = 1, 8, 6, 10, 128
    inp = inputs.conv_inputs(n, d, h, w, c, c, seed=27, device=DEV)
    wp = empty(27 * c * c)
    api.cc_conv3d_prepare(inp["w"], wp)
    full = empty(n, d, h, w, c)
    api.cc_conv3d_causal(inp["x"], wp, inp["b"], full)
    y0, y1 = empty(n, 4, h, w, c), empty(n, 4, h, w, c)
    api.cc_conv3d_causal(inp["x"][:, :4].contiguous(), wp, inp["b"], y0, hist=0)
    api.cc_conv3d_causal(inp["x"][:, 2:].contiguous(), wp, inp["b"], y1, hist=2)
    api.cc_check_device()
    assert torch.equal(torch.cat([y0, y1], 1), full)


def test_head_chunked_streaming_equals_one_call():
    n, d, h, w, c = 1, 8, 8, 20, 64
    inp = inputs.head_inputs(n, d, h, w, c, seed=28, device=DEV)
    wp = empty(3 * api.HEAD_G_CH * c)
    api.cc_head_prepare(inp["w"], wp)
    ws = torch.empty(api.cc_head_workspace_bytes(n, d, h, w), dtype=torch.uint8, device=DEV)
    full = empty(n, d, h, w, 12)
    api.cc_head_out(inp["x"], wp, inp["b"], full, ws)
    y0, y1 = empty(n, 4, h, w, 12), empty(n, 4, h, w, 12)
    api.cc_head_out(inp["x"][:, :4].contiguous(), wp, inp["b"], y0, ws, hist=0)
    api.cc_head_out(inp["x"][:, 2:].contiguous(), wp, inp["b"], y1, ws, hist=2)
    api.cc_check_device()
    assert torch.equal(torch.cat([y0, y1], 1), full)


@pytest.mark.parametrize("temporal", [False, True])
def test_resample_chunked_streaming_equals_one_call(temporal):
    n, d, hl, wl, c = 1, 8, 6, 9, 64
    inp = inputs.resample_inputs(n, d, hl, wl, c, seed=29, device=DEV)
    pw = empty((64 if temporal else 48) * c * c)
    (api.cc_resample_prepare_temporal if temporal else api.cc_resample_prepare)(inp["w"], pw)
    ft = 2 if temporal else 1
    full = empty(n, ft * d, 2 * hl, 2 * wl, c)
    api.cc_resample_up2_fused(inp["x"], pw, inp["b"], inp["skip"], full, temporal=temporal)
    y0, y1 = empty(n, ft * 4, 2 * hl, 2 * wl, c), empty(n, ft * 4, 2 * hl, 2 * wl, c)
    api.cc_resample_up2_fused(inp["x"][:, :4].contiguous(), pw, inp["b"], inp["skip"][:, :4].contiguous(), y0,
                              hist=0, temporal=temporal)
    api.cc_resample_up2_fused(inp["x"][:, 2:].contiguous(), pw, inp["b"], inp["skip"][:, 4:].contiguous(), y1,
                              hist=2, temporal=temporal)
    api.cc_check_device()
    assert torch.equal(torch.cat([y0, y1], 1), full)


# ------------------------------------- dependent launches on one stream --

def test_dependent_chain_on_one_stream_matches_synchronised_run():
    # conv -> fused resampler -> head, each reading the previous output, queued
    # back to back on one stream (the kernels are launched with programmatic
    # serialization and wait for their predecessor before the first global
    # access); the result must equal, bit for bit, the same launches with the
    # host synchronising after each
    g = torch.Generator(device=DEV).manual_seed(71)
    n, d, h, w, c = 1, 3, 24, 40, 64
    x = torch.randn((n, d, h, w, c), generator=g, device=DEV).to(BF16)
    wc = (torch.randn((c, c, 3, 3, 3), generator=g, device=DEV) / (27 * c) ** 0.5).to(BF16)
    bc = (torch.randn((c,), generator=g, device=DEV) * 0.1).to(BF16)
    wr = (torch.randn((c, c, 3, 3, 3), generator=g, device=DEV) / (27 * c) ** 0.5).to(BF16)
    br = (torch.randn((c,), generator=g, device=DEV) * 0.1).to(BF16)
    wh = (torch.randn((12, c, 3, 3, 3), generator=g, device=DEV) / (27 * c) ** 0.5).to(BF16)
    bh = (torch.randn((12,), generator=g, device=DEV) * 0.1).to(BF16)
    wpc = empty(27 * c * c)
    api.cc_conv3d_prepare(wc, wpc)
    pw = empty(48 * c * c)
    api.cc_resample_prepare(wr, pw)
    wph = empty(3 * api.HEAD_G_CH * c)
    api.cc_head_prepare(wh, wph)
    torch.cuda.synchronize()

    def chain(sync):
        y = empty(n, d, h, w, c)
        up = empty(n, d, 2 * h, 2 * w, c)
        out = empty(n, d, 2 * h, 2 * w, api.HEAD_COUT)
        ws = torch.empty(api.cc_head_workspace_bytes(n, d, 2 * h, 2 * w), dtype=torch.uint8, device=DEV)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            api.cc_conv3d_causal(x, wpc, bc, y, stream=s)
            if sync:
                s.synchronize()
            api.cc_resample_up2_fused(y, pw, br, y, up, stream=s)
            if sync:
                s.synchronize()
            api.cc_head_out(up, wph, bh, out, ws, stream=s)
        s.synchronize()
        api.cc_check_device()
        return y, up, out

    a, b = chain(False), chain(True)
    for name, u, v in zip(("conv", "resampler", "head"), a, b):
        assert torch.equal(u, v), f"{name}: the queued chain differs from the synchronised one"


def test_two_streams_at_once_match_one_after_the_other():
    # independent stages queued on two streams at the same time (their
    # persistent kernels then share the SMs and the device error word) give
    # the same bits as the same calls one after the other on one stream
    g = torch.Generator(device=DEV).manual_seed(72)
    n, d, h, w, c = 1, 3, 24, 40, 64
    x = torch.randn((n, d, h, w, c), generator=g, device=DEV).to(BF16)
    wc = (torch.randn((c, c, 3, 3, 3), generator=g, device=DEV) / (27 * c) ** 0.5).to(BF16)
    bc = (torch.randn((c,), generator=g, device=DEV) * 0.1).to(BF16)
    wr = (torch.randn((c, c, 3, 3, 3), generator=g, device=DEV) / (27 * c) ** 0.5).to(BF16)
    skip = torch.randn((n, d, h, w, c), generator=g, device=DEV).to(BF16)
    wh = (torch.randn((12, c, 3, 3, 3), generator=g, device=DEV) / (27 * c) ** 0.5).to(BF16)
    bh = (torch.randn((12,), generator=g, device=DEV) * 0.1).to(BF16)
    t, hw, ca = 2, 500, 128
    q, k, v = (torch.randn((t, hw, ca), generator=g, device=DEV).to(BF16) for _ in range(3))
    wpc = empty(27 * c * c)
    api.cc_conv3d_prepare(wc, wpc)
    pw = empty(48 * c * c)
    api.cc_resample_prepare(wr, pw)
    wph = empty(3 * api.HEAD_G_CH * c)
    api.cc_head_prepare(wh, wph)
    torch.cuda.synchronize()

    def run(two_streams):
        y = empty(n, d, h, w, c)
        hd = empty(n, d, h, w, api.HEAD_COUT)
        up = empty(n, d, 2 * h, 2 * w, c)
        o = empty(t, hw, ca)
        ws = torch.empty(api.cc_attn_exp_workspace_bytes(t, hw), dtype=torch.uint8, device=DEV)
        sa = torch.cuda.Stream()
        sb = torch.cuda.Stream() if two_streams else sa
        api.cc_conv3d_causal(x, wpc, bc, y, stream=sa)
        api.cc_attn_frame_exp(q, k, v, o, ws, stream=sb)
        api.cc_head_out_fused(x, wph, bh, hd, stream=sa)
        api.cc_resample_up2_fused(x, pw, bc, skip, up, stream=sb)
        sa.synchronize()
        sb.synchronize()
        api.cc_check_device()
        return y, o, hd, up

    a, b = run(True), run(False)
    for name, u, v in zip(("conv", "attention", "head", "resampler"), a, b):
        assert torch.equal(u.view(torch.int16), v.view(torch.int16)), f"{name}: two streams differ from one"
