"""Python binding of the C ABI (include/cc.h): the same entry points under the
same names, taking torch CUDA tensors instead of raw pointers.

Argument marshalling only: each function checks that its tensors are CUDA,
contiguous and of the expected dtype, reads the sizes off their shapes, and
calls the library on the current (or given) stream. All compute runs in
libcc.so's kernels. A non-OK status raises ``CCError`` with the library's
message.
"""

from __future__ import annotations

import torch

from . import _lib

__all__ = [
    "CCError", "cc_version", "cc_check_device",
    "cc_conv3d_prepare", "cc_conv3d_causal",
    "cc_resample_prepare", "cc_resample_workspace_bytes", "cc_resample_phase_conv", "cc_resample_interleave",
    "cc_resample_up2", "cc_resample_up2_fused", "cc_resample_prepare_temporal",
    "cc_attn_ld", "cc_attn_workspace_bytes", "cc_attn_scores", "cc_attn_softmax", "cc_attn_pv", "cc_attn_frame",
    "cc_attn_exp_key_tiles", "cc_attn_exp_workspace_bytes", "cc_attn_scores_exp", "cc_attn_exp_rescale",
    "cc_attn_pv_exp", "cc_attn_frame_exp",
    "cc_head_prepare", "cc_head_workspace_bytes", "cc_head_temporal", "cc_head_stencil", "cc_head_out",
    "cc_attn_scores_stats", "cc_attn_fused_workspace_bytes", "cc_attn_frame_fused",
    "cc_head_out_fused", "cc_head_out_noalloc", "HEAD_NOALLOC_SCRATCH_BYTES", "cc_copy_to_host",
    "cc_debug_im2col_tile", "cc_debug_wait_timeout", "cc_debug_conv_bad_tile_order",
    "HEAD_COUT", "HEAD_G_CH",
]

HEAD_COUT = 12
HEAD_G_CH = 112
HEAD_NOALLOC_SCRATCH_BYTES = 64 << 20  # CC_HEAD_NOALLOC_SCRATCH_BYTES

STATUS = {0: "CC_OK", 1: "CC_ERR_INVALID", 2: "CC_ERR_UNSUPPORTED", 3: "CC_ERR_CUDA", 4: "CC_ERR_TIMEOUT",
          5: "CC_ERR_DEVICE"}


class CCError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def _check(st: int) -> None:
    if st != 0:
        msg = _lib.load().cc_last_error()
        raise CCError(st, msg.decode() if msg else "")


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: torch.Tensor | None, dtype=torch.bfloat16, name: str = "tensor") -> int | None:
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name}: must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return t.data_ptr()


def cc_version() -> int:
    return _lib.load().cc_version()


def cc_check_device(stream=None) -> None:
    _check(_lib.load().cc_check_device(_stream(stream)))


# ------------------------------------------------------- causal 3x3x3 conv --

def cc_conv3d_prepare(w: torch.Tensor, wp: torch.Tensor, stream=None) -> None:
    cout, cin = w.shape[:2]
    if tuple(w.shape) != (cout, cin, 3, 3, 3) or wp.numel() != 27 * cout * cin:
        raise ValueError("conv3d_prepare: w must be [Cout,Cin,3,3,3] and wp hold 27*Cout*Cin elements")
    _check(_lib.load().cc_conv3d_prepare(_ptr(w, name="w"), _ptr(wp, name="wp"), cout, cin, _stream(stream)))


def cc_conv3d_causal(x, wp, bias, y, hist: int = 0, stream=None) -> None:
    n, d, h, w, cout = y.shape
    cin = x.shape[-1]
    if tuple(x.shape) != (n, d + hist, h, w, cin):
        raise ValueError(f"conv3d_causal: x {tuple(x.shape)} does not match y {tuple(y.shape)} with hist={hist}")
    if wp.numel() != 27 * cout * cin:
        raise ValueError("conv3d_causal: wp must hold 27*Cout*Cin elements")
    if bias is not None and bias.numel() != cout:
        raise ValueError("conv3d_causal: bias must hold Cout elements")
    _check(_lib.load().cc_conv3d_causal(_ptr(x, name="x"), _ptr(wp, name="wp"), _ptr(bias, name="bias"),
                                        _ptr(y, name="y"), n, d, h, w, cin, cout, hist, _stream(stream)))


# ------------------------------------------------------- spatial resampler --

def cc_resample_prepare(w, pw, stream=None) -> None:
    cout, cin = w.shape[:2]
    if tuple(w.shape) != (cout, cin, 3, 3, 3) or pw.numel() != 48 * cout * cin:
        raise ValueError("resample_prepare: w must be [Cout,Cin,3,3,3] and pw hold 48*Cout*Cin elements")
    _check(_lib.load().cc_resample_prepare(_ptr(w, name="w"), _ptr(pw, name="pw"), cout, cin, _stream(stream)))


def cc_resample_workspace_bytes(n: int, d: int, hl: int, wl: int, cout: int) -> int:
    return _lib.load().cc_resample_workspace_bytes(n, d, hl, wl, cout)


def cc_resample_phase_conv(x, pw, phases, hist: int = 0, stream=None) -> None:
    four, n, d, hl, wl, cout = phases.shape
    cin = x.shape[-1]
    if four != 4 or tuple(x.shape) != (n, d + hist, hl, wl, cin) or pw.numel() != 48 * cout * cin:
        raise ValueError("resample_phase_conv: phases must be [4,N,D,HL,WL,Cout] matching x and pw")
    _check(_lib.load().cc_resample_phase_conv(_ptr(x, name="x"), _ptr(pw, name="pw"), _ptr(phases, name="phases"),
                                              n, d, hl, wl, cin, cout, hist, _stream(stream)))


def cc_resample_interleave(phases, bias, skip, out, stream=None) -> None:
    four, n, d, hl, wl, c = phases.shape
    if four != 4 or tuple(skip.shape) != (n, d, hl, wl, c) or tuple(out.shape) != (n, d, 2 * hl, 2 * wl, c) \
            or bias.numel() != c:
        raise ValueError("resample_interleave: shapes do not match")
    _check(_lib.load().cc_resample_interleave(_ptr(phases, name="phases"), _ptr(bias, name="bias"),
                                              _ptr(skip, name="skip"), _ptr(out, name="out"), n, d, hl, wl, c,
                                              _stream(stream)))


def cc_resample_up2(x, pw, bias, skip, out, ws, hist: int = 0, stream=None) -> None:
    n, d, h2, w2, cout = out.shape
    hl, wl = h2 // 2, w2 // 2
    cin = x.shape[-1]
    if h2 != 2 * hl or w2 != 2 * wl or tuple(x.shape) != (n, d + hist, hl, wl, cin):
        raise ValueError("resample_up2: out must be [N,D,2HL,2WL,Cout] of x [N,D+hist,HL,WL,Cin]")
    if tuple(skip.shape) != (n, d, hl, wl, cout) or bias.numel() != cout or pw.numel() != 48 * cout * cin:
        raise ValueError("resample_up2: skip, bias or pw shape mismatch")
    _check(_lib.load().cc_resample_up2(_ptr(x, name="x"), _ptr(pw, name="pw"), _ptr(bias, name="bias"),
                                       _ptr(skip, name="skip"), _ptr(out, name="out"), n, d, hl, wl, cin, cout, hist,
                                       _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream(stream)))


def cc_resample_prepare_temporal(w, pw, stream=None) -> None:
    cout, cin = w.shape[:2]
    if tuple(w.shape) != (cout, cin, 3, 3, 3) or pw.numel() != 64 * cout * cin:
        raise ValueError("resample_prepare_temporal: w must be [Cout,Cin,3,3,3] and pw hold 64*Cout*Cin elements")
    _check(_lib.load().cc_resample_prepare_temporal(_ptr(w, name="w"), _ptr(pw, name="pw"), cout, cin,
                                                    _stream(stream)))


def cc_resample_up2_fused(x, pw, bias, skip, out, hist: int = 0, temporal: bool = False, stream=None) -> None:
    n, d2, h2, w2, cout = out.shape
    hl, wl = h2 // 2, w2 // 2
    d = d2 // 2 if temporal else d2
    cin = x.shape[-1]
    if h2 != 2 * hl or w2 != 2 * wl or (temporal and d2 != 2 * d) or tuple(x.shape) != (n, d + hist, hl, wl, cin):
        raise ValueError("resample_up2_fused: out must be [N,(2)D,2HL,2WL,Cout] of x [N,D+hist,HL,WL,Cin]")
    taps = 64 if temporal else 48
    if tuple(skip.shape) != (n, d, hl, wl, cout) or bias.numel() != cout or pw.numel() != taps * cout * cin:
        raise ValueError("resample_up2_fused: skip, bias or pw shape mismatch")
    _check(_lib.load().cc_resample_up2_fused(_ptr(x, name="x"), _ptr(pw, name="pw"), _ptr(bias, name="bias"),
                                             _ptr(skip, name="skip"), _ptr(out, name="out"), n, d, hl, wl, cin, cout,
                                             hist, 1 if temporal else 0, _stream(stream)))


# ------------------------------------------------------ per-frame attention --

def cc_attn_ld(hw: int) -> int:
    return _lib.load().cc_attn_ld(hw)


def cc_attn_workspace_bytes(t: int, hw: int) -> int:
    return _lib.load().cc_attn_workspace_bytes(t, hw)


def _rows(t: torch.Tensor, name: str):
    """(T, HW, C, ld) of a [T, HW, C] tensor whose rows may be strided (packed qkv slices)."""
    if t.dim() != 3 or (t.numel() and (t.stride(2) != 1 or t.stride(0) != t.shape[1] * t.stride(1))):
        raise ValueError(f"{name}: expected [T,HW,C] with unit channel stride and frame stride HW*ld")
    if t.device.type != "cuda" or t.dtype != torch.bfloat16:
        raise ValueError(f"{name}: expected a bf16 CUDA tensor")
    return t.shape[0], t.shape[1], t.shape[2], t.stride(1)


def cc_attn_scores(q, k, s, stream=None) -> None:
    t, hw, c, ld_q = _rows(q, "q")
    _, _, _, ld_k = _rows(k, "k")
    if tuple(k.shape) != (t, hw, c) or s.dim() != 3 or s.shape[0] != t or s.shape[1] != hw:
        raise ValueError("attn_scores: shapes do not match")
    _check(_lib.load().cc_attn_scores(q.data_ptr(), k.data_ptr(), _ptr(s, torch.float32, "s"), t, hw, c, ld_q, ld_k,
                                      s.shape[2], _stream(stream)))


def cc_attn_softmax(s, p, hw: int, scale: float, stream=None) -> None:
    t = s.shape[0]
    if s.dim() != 3 or p.dim() != 3 or s.shape[:2] != (t, hw) or p.shape[:2] != (t, hw):
        raise ValueError("attn_softmax: s and p must be [T,HW,ld]")
    _check(_lib.load().cc_attn_softmax(_ptr(s, torch.float32, "s"), _ptr(p, name="p"), t, hw, s.shape[2], p.shape[2],
                                       float(scale), _stream(stream)))


def cc_attn_pv(p, v, o, hw: int, stream=None) -> None:
    t, _, c, ld_v = _rows(v, "v")
    _, _, _, ld_o = _rows(o, "o")
    if p.dim() != 3 or p.shape[:2] != (t, hw):
        raise ValueError("attn_pv: p must be [T,HW,ld]")
    _check(_lib.load().cc_attn_pv(_ptr(p, name="p"), v.data_ptr(), o.data_ptr(), t, hw, c, p.shape[2], ld_v, ld_o,
                                  _stream(stream)))


def cc_attn_frame(q, k, v, o, ws, scale: float | None = None, stream=None) -> None:
    t, hw, c, ld_q = _rows(q, "q")
    _, _, _, ld_k = _rows(k, "k")
    _, _, _, ld_v = _rows(v, "v")
    _, _, _, ld_o = _rows(o, "o")
    if not (tuple(k.shape) == tuple(v.shape) == tuple(o.shape) == (t, hw, c)):
        raise ValueError("attn_frame: q, k, v, o must share [T,HW,C]")
    if scale is None:
        scale = c ** -0.5
    _check(_lib.load().cc_attn_frame(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), t, hw, c, ld_q, ld_k,
                                     ld_v, ld_o, float(scale), _ptr(ws, torch.uint8, "ws"), ws.numel(),
                                     _stream(stream)))


def cc_attn_exp_key_tiles(hw: int) -> int:
    return _lib.load().cc_attn_exp_key_tiles(hw)


def cc_attn_exp_workspace_bytes(t: int, hw: int) -> int:
    return _lib.load().cc_attn_exp_workspace_bytes(t, hw)


def cc_attn_scores_exp(q, k, e, stats, scale: float | None = None, stream=None) -> None:
    """e: bf16 [T, HW, ld]; stats: fp32 [T, HW, key_tiles, 2] (pairs c_t, l_t)."""
    t, hw, c, ld_q = _rows(q, "q")
    _, _, _, ld_k = _rows(k, "k")
    tiles = cc_attn_exp_key_tiles(hw)
    if tuple(k.shape) != (t, hw, c) or e.dim() != 3 or tuple(e.shape[:2]) != (t, hw):
        raise ValueError("attn_scores_exp: shapes do not match")
    if tuple(stats.shape) != (t, hw, tiles, 2):
        raise ValueError(f"attn_scores_exp: stats must be [T,HW,{tiles},2]")
    if scale is None:
        scale = c ** -0.5
    _check(_lib.load().cc_attn_scores_exp(q.data_ptr(), k.data_ptr(), _ptr(e, name="e"),
                                          _ptr(stats, torch.float32, "stats"), t, hw, c, ld_q, ld_k, e.shape[2],
                                          float(scale), _stream(stream)))


def cc_attn_exp_rescale(e, stats, hw: int, stream=None) -> None:
    t = e.shape[0]
    if e.dim() != 3 or tuple(e.shape[:2]) != (t, hw) or tuple(stats.shape) != (t, hw, cc_attn_exp_key_tiles(hw), 2):
        raise ValueError("attn_exp_rescale: e must be [T,HW,ld] and stats [T,HW,key_tiles,2]")
    _check(_lib.load().cc_attn_exp_rescale(_ptr(e, name="e"), _ptr(stats, torch.float32, "stats"), t, hw, e.shape[2],
                                           _stream(stream)))


def cc_attn_pv_exp(e, stats, v, o, stream=None) -> None:
    t, hw, c, ld_v = _rows(v, "v")
    _, _, _, ld_o = _rows(o, "o")
    if e.dim() != 3 or tuple(e.shape[:2]) != (t, hw) or tuple(stats.shape) != (t, hw, cc_attn_exp_key_tiles(hw), 2):
        raise ValueError("attn_pv_exp: e must be [T,HW,ld] and stats [T,HW,key_tiles,2]")
    _check(_lib.load().cc_attn_pv_exp(_ptr(e, name="e"), _ptr(stats, torch.float32, "stats"), v.data_ptr(),
                                      o.data_ptr(), t, hw, c, e.shape[2], ld_v, ld_o, _stream(stream)))


def cc_attn_frame_exp(q, k, v, o, ws, scale: float | None = None, stream=None) -> None:
    t, hw, c, ld_q = _rows(q, "q")
    _, _, _, ld_k = _rows(k, "k")
    _, _, _, ld_v = _rows(v, "v")
    _, _, _, ld_o = _rows(o, "o")
    if not (tuple(k.shape) == tuple(v.shape) == tuple(o.shape) == (t, hw, c)):
        raise ValueError("attn_frame_exp: q, k, v, o must share [T,HW,C]")
    if scale is None:
        scale = c ** -0.5
    _check(_lib.load().cc_attn_frame_exp(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), t, hw, c, ld_q, ld_k,
                                         ld_v, ld_o, float(scale), _ptr(ws, torch.uint8, "ws"), ws.numel(),
                                         _stream(stream)))


def cc_attn_scores_stats(q, k, stats, scale: float | None = None, stream=None) -> None:
    """stats: fp32 [T, HW, key_tiles, 2] (pairs c_t, l_t); E is not written."""
    t, hw, c, ld_q = _rows(q, "q")
    _, _, _, ld_k = _rows(k, "k")
    tiles = cc_attn_exp_key_tiles(hw)
    if tuple(k.shape) != (t, hw, c) or tuple(stats.shape) != (t, hw, tiles, 2):
        raise ValueError(f"attn_scores_stats: k must be [T,HW,C] and stats [T,HW,{tiles},2]")
    if scale is None:
        scale = c ** -0.5
    _check(_lib.load().cc_attn_scores_stats(q.data_ptr(), k.data_ptr(), _ptr(stats, torch.float32, "stats"), t, hw,
                                            c, ld_q, ld_k, float(scale), _stream(stream)))


def cc_attn_fused_workspace_bytes(t: int, hw: int) -> int:
    return _lib.load().cc_attn_fused_workspace_bytes(t, hw)


def cc_attn_frame_fused(q, k, v, o, ws, scale: float | None = None, stream=None) -> None:
    """Attention with the numerators kept on chip (statistics pass + one kernel)."""
    t, hw, c, ld_q = _rows(q, "q")
    _, _, _, ld_k = _rows(k, "k")
    _, _, _, ld_v = _rows(v, "v")
    _, _, _, ld_o = _rows(o, "o")
    if not (tuple(k.shape) == tuple(v.shape) == tuple(o.shape) == (t, hw, c)):
        raise ValueError("attn_frame_fused: q, k, v, o must share [T,HW,C]")
    if scale is None:
        scale = c ** -0.5
    _check(_lib.load().cc_attn_frame_fused(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), t, hw, c, ld_q,
                                           ld_k, ld_v, ld_o, float(scale), _ptr(ws, torch.uint8, "ws"), ws.numel(),
                                           _stream(stream)))


# -------------------------------------------------------------- output head --

def cc_head_prepare(w, wp, stream=None) -> None:
    cin = w.shape[1]
    if tuple(w.shape) != (HEAD_COUT, cin, 3, 3, 3) or wp.numel() != 3 * HEAD_G_CH * cin:
        raise ValueError("head_prepare: w must be [12,Cin,3,3,3] and wp hold 3*112*Cin elements")
    _check(_lib.load().cc_head_prepare(_ptr(w, name="w"), _ptr(wp, name="wp"), cin, _stream(stream)))


def cc_head_workspace_bytes(n: int, d: int, h: int, w: int) -> int:
    return _lib.load().cc_head_workspace_bytes(n, d, h, w)


def cc_head_temporal(x, wp, g, hist: int = 0, stream=None) -> None:
    n, d, h, w, ch = g.shape
    cin = x.shape[-1]
    if ch != HEAD_G_CH or tuple(x.shape) != (n, d + hist, h, w, cin) or wp.numel() != 3 * HEAD_G_CH * cin:
        raise ValueError("head_temporal: g must be [N,D,H,W,112] matching x and wp")
    _check(_lib.load().cc_head_temporal(_ptr(x, name="x"), _ptr(wp, name="wp"), _ptr(g, name="g"), n, d, h, w, cin,
                                        hist, _stream(stream)))


def cc_head_stencil(g, bias, out, stream=None) -> None:
    n, d, h, w, c = out.shape
    if c != HEAD_COUT or tuple(g.shape) != (n, d, h, w, HEAD_G_CH) or bias.numel() != HEAD_COUT:
        raise ValueError("head_stencil: g must be [N,D,H,W,112] and out [N,D,H,W,12]")
    _check(_lib.load().cc_head_stencil(_ptr(g, name="g"), _ptr(bias, name="bias"), _ptr(out, name="out"), n, d, h, w,
                                       _stream(stream)))


def cc_head_out(x, wp, bias, out, ws, hist: int = 0, stream=None) -> None:
    n, d, h, w, c = out.shape
    cin = x.shape[-1]
    if c != HEAD_COUT or tuple(x.shape) != (n, d + hist, h, w, cin) or bias.numel() != HEAD_COUT:
        raise ValueError("head_out: out must be [N,D,H,W,12] of x [N,D+hist,H,W,Cin]")
    _check(_lib.load().cc_head_out(_ptr(x, name="x"), _ptr(wp, name="wp"), _ptr(bias, name="bias"),
                                   _ptr(out, name="out"), n, d, h, w, cin, hist, _ptr(ws, torch.uint8, "ws"),
                                   ws.numel(), _stream(stream)))


def cc_head_out_fused(x, wp, bias, out, hist: int = 0, stream=None) -> None:
    """The whole head in one kernel (g kept in fp32 on chip), no workspace."""
    n, d, h, w, c = out.shape
    cin = x.shape[-1]
    if c != HEAD_COUT or tuple(x.shape) != (n, d + hist, h, w, cin) or bias.numel() != HEAD_COUT:
        raise ValueError("head_out_fused: out must be [N,D,H,W,12] of x [N,D+hist,H,W,Cin]")
    _check(_lib.load().cc_head_out_fused(_ptr(x, name="x"), _ptr(wp, name="wp"), _ptr(bias, name="bias"),
                                         _ptr(out, name="out"), n, d, h, w, cin, hist, _stream(stream)))


def cc_head_out_noalloc(x, wp, bias, out, hist: int = 0, stream=None) -> None:
    """cc_head_out without a workspace, for callers that cannot allocate device
    memory: g lives in the library's fixed 64 MiB static scratch (at most
    299,593 output positions per call; calls that overlap on the GPU race on
    it, so keep them on one stream)."""
    n, d, h, w, c = out.shape
    cin = x.shape[-1]
    if c != HEAD_COUT or tuple(x.shape) != (n, d + hist, h, w, cin) or bias.numel() != HEAD_COUT:
        raise ValueError("head_out_noalloc: out must be [N,D,H,W,12] of x [N,D+hist,H,W,Cin]")
    _check(_lib.load().cc_head_out_noalloc(_ptr(x, name="x"), _ptr(wp, name="wp"), _ptr(bias, name="bias"),
                                           _ptr(out, name="out"), n, d, h, w, cin, hist, _stream(stream)))


# -------------------------------------------------------- result read-back --

def cc_copy_to_host(dst: torch.Tensor, src: torch.Tensor, ctas: int = 8, stream=None) -> None:
    """Copies the CUDA tensor `src` into the pinned CPU tensor `dst` (same
    number of bytes, both contiguous) with a copy kernel of `ctas` CTAs."""
    if not isinstance(dst, torch.Tensor) or not isinstance(src, torch.Tensor):
        raise TypeError("copy_to_host: expected torch tensors")
    if dst.device.type != "cpu" or not dst.is_pinned():
        raise ValueError("copy_to_host: dst must be a pinned CPU tensor")
    if src.device.type != "cuda":
        raise ValueError("copy_to_host: src must be a CUDA tensor")
    if not (dst.is_contiguous() and src.is_contiguous()):
        raise ValueError("copy_to_host: tensors must be contiguous")
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("copy_to_host: dst and src hold different numbers of bytes")
    _check(_lib.load().cc_copy_to_host(dst.data_ptr(), src.data_ptr(), nbytes, int(ctas), _stream(stream)))


# ------------------------------------------------------------- self tests --

def cc_debug_im2col_tile(x, tile, lower, upper, c0, start, offsets, stream=None) -> None:
    n, d_in, h, w, c = x.shape
    if tile.numel() != 128 * 64:
        raise ValueError("debug_im2col_tile: tile must hold 128*64 elements")
    _check(_lib.load().cc_debug_im2col_tile(_ptr(x, name="x"), _ptr(tile, name="tile"), n, d_in, h, w, c, *lower,
                                            *upper, c0, *start, *offsets, _stream(stream)))


def cc_debug_wait_timeout(limit_ns: int, stream=None) -> None:
    _check(_lib.load().cc_debug_wait_timeout(int(limit_ns), _stream(stream)))


def cc_debug_conv_bad_tile_order(x, wp, y, entry: int, stream=None) -> None:
    n, d, h, w, cout = y.shape
    cin = x.shape[-1]
    if tuple(x.shape) != (n, d, h, w, cin) or wp.numel() != 27 * cout * cin:
        raise ValueError("debug_conv_bad_tile_order: x must be [N,D,H,W,Cin] of y and wp hold 27*Cout*Cin elements")
    _check(_lib.load().cc_debug_conv_bad_tile_order(_ptr(x, name="x"), _ptr(wp, name="wp"), _ptr(y, name="y"), n, d,
                                                    h, w, cin, cout, int(entry), _stream(stream)))
