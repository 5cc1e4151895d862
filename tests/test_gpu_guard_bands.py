"""Memory canaries around every output of every entry point. compute-sanitizer
is not available on the test machines, so each output (and each workspace)
sits inside a larger buffer whose guard bands, 4096 elements before and
after, hold a sentinel bit pattern; after the call and a device check, the
bands must be unchanged, the inputs must be bit-identical to what they were,
and, for the row-strided attention buffers, the padding columns past HW must
hold what the header says: untouched for E, zeros for P, and for S untouched
past the 16-byte piece that holds a row's last score. Shapes are
ragged on purpose: partial tiles in every dimension, two images, carried
history frames."""

import math

import pytest
import torch

from causal_convolution_gb300 import api
from gpu_util import ensure_built

pytestmark = pytest.mark.gpu
DEV = "cuda"
BF16 = torch.bfloat16
GUARD = 4096
SENTINEL = {BF16: (torch.int16, 0x7FA5), torch.float32: (torch.int32, 0x7FC0A5A5), torch.uint8: (torch.uint8, 0xA5)}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    return ensure_built()


class Guarded:
    """A tensor of `shape` in the middle of a buffer whose GUARD elements on
    either side (and the tensor itself) start as the sentinel."""

    def __init__(self, shape, dtype=BF16):
        self.dtype = dtype
        self.n = math.prod(shape)
        self.buf = torch.empty(self.n + 2 * GUARD, dtype=dtype, device=DEV)
        self.bits, self.pattern = SENTINEL[dtype]
        self.buf.view(self.bits).fill_(self.pattern)
        self.t = self.buf[GUARD:GUARD + self.n].view(shape)

    def bands_intact(self) -> bool:
        b = self.buf.view(self.bits)
        return bool(torch.all(b[:GUARD] == self.pattern)) and bool(torch.all(b[GUARD + self.n:] == self.pattern))

    def untouched(self, view) -> bool:
        return bool(torch.all(view.contiguous().view(self.bits) == self.pattern))


def rnd(shape, seed, scale=1.0):
    g = torch.Generator(device=DEV).manual_seed(seed)
    return (torch.randn(shape, generator=g, device=DEV) * scale).to(BF16)


def bits(x):
    return x.contiguous().view(SENTINEL[x.dtype][0])


def call_and_check(fn, inputs, outputs, what):
    before = [bits(x).clone() for x in inputs]
    fn()
    api.cc_check_device()
    for i, (x, x0) in enumerate(zip(inputs, before)):
        assert torch.equal(bits(x), x0), f"{what}: input {i} was modified"
    for i, o in enumerate(outputs):
        assert o.bands_intact(), f"{what}: output {i} written outside its bounds"


def finite(t):
    return bool(torch.isfinite(t.float()).all())


# ------------------------------------------------------------------ prepare --

@pytest.mark.parametrize("kind", ["conv", "resample", "resample_temporal", "head"])
def test_prepare_kernels_write_only_their_output(kind):
    cout, cin = (12, 128) if kind == "head" else (80, 64)
    w = rnd((cout, cin, 3, 3, 3), 1, 0.05)
    per = {"conv": 27 * cout * cin, "resample": 48 * cout * cin, "resample_temporal": 64 * cout * cin,
           "head": 3 * api.HEAD_G_CH * cin}[kind]
    wp = Guarded((per,))
    fn = {"conv": api.cc_conv3d_prepare, "resample": api.cc_resample_prepare,
          "resample_temporal": api.cc_resample_prepare_temporal, "head": api.cc_head_prepare}[kind]
    call_and_check(lambda: fn(w, wp.t), [w], [wp], f"{kind} prepare")


# --------------------------------------------------------------------- conv --

@pytest.mark.parametrize("hist", [0, 2])
def test_conv_writes_only_its_output(hist):
    n, d, h, w, cin, cout = 2, 3, 5, 7, 64, 80
    x = rnd((n, d + hist, h, w, cin), 2)
    wp = rnd((27 * cout * cin,), 3, 0.02)
    b = rnd((cout,), 4, 0.1)
    y = Guarded((n, d, h, w, cout))
    call_and_check(lambda: api.cc_conv3d_causal(x, wp, b, y.t, hist=hist), [x, wp, b], [y], f"conv hist={hist}")
    assert finite(y.t)


# ---------------------------------------------------------------- resampler --

@pytest.mark.parametrize("hist,temporal", [(0, False), (2, False), (0, True), (2, True)])
def test_fused_resampler_writes_only_its_output(hist, temporal):
    n, d, hl, wl, cin, cout = 2, 2, 5, 7, 64, 80
    x = rnd((n, d + hist, hl, wl, cin), 5)
    pw = rnd(((64 if temporal else 48) * cout * cin,), 6, 0.02)
    b = rnd((cout,), 7, 0.1)
    skip = rnd((n, d, hl, wl, cout), 8)
    out = Guarded((n, 2 * d if temporal else d, 2 * hl, 2 * wl, cout))
    call_and_check(lambda: api.cc_resample_up2_fused(x, pw, b, skip, out.t, hist=hist, temporal=temporal),
                   [x, pw, b, skip], [out], f"fused resampler hist={hist} temporal={temporal}")
    assert finite(out.t)


def test_two_pass_resampler_writes_only_its_outputs():
    n, d, hl, wl, cin, cout, hist = 2, 2, 5, 7, 64, 80, 2
    x = rnd((n, d + hist, hl, wl, cin), 9)
    pw = rnd((48 * cout * cin,), 10, 0.02)
    b = rnd((cout,), 11, 0.1)
    skip = rnd((n, d, hl, wl, cout), 12)
    phases = Guarded((4, n, d, hl, wl, cout))
    call_and_check(lambda: api.cc_resample_phase_conv(x, pw, phases.t, hist=hist), [x, pw], [phases], "phase convs")
    out = Guarded((n, d, 2 * hl, 2 * wl, cout))
    call_and_check(lambda: api.cc_resample_interleave(phases.t, b, skip, out.t), [phases.t, b, skip], [out],
                   "interleave")
    ws = Guarded((api.cc_resample_workspace_bytes(n, d, hl, wl, cout),), torch.uint8)
    out2 = Guarded((n, d, 2 * hl, 2 * wl, cout))
    call_and_check(lambda: api.cc_resample_up2(x, pw, b, skip, out2.t, ws.t, hist=hist), [x, pw, b, skip],
                   [out2, ws], "composite resampler")
    assert finite(out.t) and torch.equal(bits(out.t), bits(out2.t))


# ---------------------------------------------------------------- attention --

T, HW, C = 2, 333, 128


def qkv(c=C, seed=13):
    return rnd((T, HW, c), seed), rnd((T, HW, c), seed + 1), rnd((T, HW, c), seed + 2)


LD = 352  # row stride of S, P and E: 19 columns past HW = 333


def test_three_pass_attention_writes_only_its_outputs():
    q, k, v = qkv()
    s = Guarded((T, HW, LD), torch.float32)
    call_and_check(lambda: api.cc_attn_scores(q, k, s.t), [q, k], [s], "scores")
    # S leaves through tensor stores, which end a row on a 16-byte boundary:
    # columns 333-335 may hold zeros, the rest of the padding is untouched
    assert s.untouched(s.t[:, :, 336:]), "scores: padding columns written past the row's last 16 bytes"
    p = Guarded((T, HW, LD))
    call_and_check(lambda: api.cc_attn_softmax(s.t, p.t, HW, C ** -0.5), [s.t], [p], "softmax")
    assert torch.all(p.t[:, :, HW:] == 0), "softmax: padding columns of P are not zero"
    o = Guarded((T, HW, C))
    call_and_check(lambda: api.cc_attn_pv(p.t, v, o.t, HW), [p.t, v], [o], "PV")
    ws = Guarded((api.cc_attn_workspace_bytes(T, HW),), torch.uint8)
    o2 = Guarded((T, HW, C))
    call_and_check(lambda: api.cc_attn_frame(q, k, v, o2.t, ws.t), [q, k, v], [o2, ws], "composite attention")
    assert finite(p.t) and finite(o.t) and torch.equal(bits(o.t), bits(o2.t))


def test_key_tile_attention_writes_only_its_outputs():
    q, k, v = qkv(seed=16)
    tiles = api.cc_attn_exp_key_tiles(HW)
    e = Guarded((T, HW, LD))
    st = Guarded((T, HW, tiles, 2), torch.float32)
    call_and_check(lambda: api.cc_attn_scores_exp(q, k, e.t, st.t), [q, k], [e, st], "numerators")
    assert e.untouched(e.t[:, :, HW:]), "numerators: padding columns written"
    call_and_check(lambda: api.cc_attn_exp_rescale(e.t, st.t, HW), [], [e, st], "rescale")
    assert e.untouched(e.t[:, :, HW:]), "rescale: padding columns written"
    o = Guarded((T, HW, C))
    call_and_check(lambda: api.cc_attn_pv_exp(e.t, st.t, v, o.t), [e.t, st.t, v], [o], "PV with row scale")
    ws = Guarded((api.cc_attn_exp_workspace_bytes(T, HW),), torch.uint8)
    o2 = Guarded((T, HW, C))
    call_and_check(lambda: api.cc_attn_frame_exp(q, k, v, o2.t, ws.t), [q, k, v], [o2, ws],
                   "composite key-tile attention")
    assert finite(e.t[:, :, :HW]) and finite(o.t) and torch.equal(bits(o.t), bits(o2.t))


def test_numerators_through_tensor_stores_stay_in_their_rows():
    # a row stride of 344 elements is not a multiple of 16, so E leaves
    # through staged TMA tensor stores instead of 32-byte stores from
    # registers: the same values, and nothing written past the 16-byte piece
    # that holds a row's last key (keys 333-335 may hold zeros)
    q, k, _ = qkv(seed=25)
    tiles = api.cc_attn_exp_key_tiles(HW)
    e1, st1 = Guarded((T, HW, LD)), Guarded((T, HW, tiles, 2), torch.float32)
    call_and_check(lambda: api.cc_attn_scores_exp(q, k, e1.t, st1.t), [q, k], [e1, st1], "numerators, direct stores")
    e2, st2 = Guarded((T, HW, 344)), Guarded((T, HW, tiles, 2), torch.float32)
    call_and_check(lambda: api.cc_attn_scores_exp(q, k, e2.t, st2.t), [q, k], [e2, st2], "numerators, tensor stores")
    assert e2.untouched(e2.t[:, :, 336:]), "numerators: padding columns written past the row's last 16 bytes"
    assert torch.equal(bits(e1.t[:, :, :HW]), bits(e2.t[:, :, :HW])) and torch.equal(bits(st1.t), bits(st2.t))


def test_fused_attention_writes_only_its_outputs():
    q, k, v = qkv(c=256, seed=19)
    tiles = api.cc_attn_exp_key_tiles(HW)
    st = Guarded((T, HW, tiles, 2), torch.float32)
    call_and_check(lambda: api.cc_attn_scores_stats(q, k, st.t), [q, k], [st], "statistics pass")
    ws = Guarded((api.cc_attn_fused_workspace_bytes(T, HW),), torch.uint8)
    o = Guarded((T, HW, 256))
    call_and_check(lambda: api.cc_attn_frame_fused(q, k, v, o.t, ws.t), [q, k, v], [o, ws], "fused attention")
    assert finite(o.t)


# --------------------------------------------------------------------- head --

@pytest.mark.parametrize("hist", [0, 2])
def test_head_entry_points_write_only_their_outputs(hist):
    n, d, h, w, cin = 2, 3, 5, 37, 128
    x = rnd((n, d + hist, h, w, cin), 22)
    wp = rnd((3 * api.HEAD_G_CH * cin,), 23, 0.05)
    b = rnd((api.HEAD_COUT,), 24, 0.2)
    g = Guarded((n, d, h, w, api.HEAD_G_CH))
    call_and_check(lambda: api.cc_head_temporal(x, wp, g.t, hist=hist), [x, wp], [g], "head stage A")
    out = Guarded((n, d, h, w, api.HEAD_COUT))
    call_and_check(lambda: api.cc_head_stencil(g.t, b, out.t), [g.t, b], [out], "head stencil")
    ws = Guarded((api.cc_head_workspace_bytes(n, d, h, w),), torch.uint8)
    out2 = Guarded((n, d, h, w, api.HEAD_COUT))
    call_and_check(lambda: api.cc_head_out(x, wp, b, out2.t, ws.t, hist=hist), [x, wp, b], [out2, ws],
                   "composite head")
    out3 = Guarded((n, d, h, w, api.HEAD_COUT))
    call_and_check(lambda: api.cc_head_out_fused(x, wp, b, out3.t, hist=hist), [x, wp, b], [out3], "fused head")
    out4 = Guarded((n, d, h, w, api.HEAD_COUT))
    call_and_check(lambda: api.cc_head_out_noalloc(x, wp, b, out4.t, hist=hist), [x, wp, b], [out4],
                   "no-workspace head")
    assert finite(out3.t) and torch.equal(bits(out.t), bits(out2.t)) and torch.equal(bits(out2.t), bits(out4.t))
