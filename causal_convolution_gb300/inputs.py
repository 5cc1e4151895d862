"""Seeded synthetic inputs for the causal-convolution stack.

This module holds random draws, scaling by a standard deviation, the bf16
rounding of the drawn values and the move to channels-last -- nothing of the
method's arithmetic. The CUDA path's tests and bench and the oracle's tests
all take their inputs from here, so both sides see identical tensors.

Recipe (per configuration): a ``torch.Generator`` on ``device`` seeded with the
configuration's seed; ``torch.randn`` in fp32 over the LOGICAL shapes, in the
order x, weight, bias, shortcut source (attention: q, k, v); each draw times
its standard deviation, rounded to bf16, then made channels-last
``[N, D, H, W, C]``. "N(0, s)" in the configuration text is read as variance
s: weights have std sqrt(1 / (27 * C_in)), biases sqrt(var).
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch

__all__ = ["CONFIGS", "Config", "conv_inputs", "resample_inputs", "attn_inputs", "head_inputs", "make_config_inputs"]


@dataclass(frozen=True)
class Config:
    name: str
    kind: str  # "conv" | "resample" | "attn" | "head"
    seed: int
    n: int = 1
    c: int = 0          # input channels (attention: head dim)
    cout: int = 0
    d: int = 0          # latent frames (attention: frames T)
    h: int = 0
    w: int = 0
    hw: int = 0         # attention positions per frame
    bias_var: float = 0.0


CONFIGS = {
    "toy_resampler": Config("toy_resampler", "resample", 0, 1, 64, 64, 2, 8, 12, bias_var=0.1),
    "mid_conv": Config("mid_conv", "conv", 1, 1, 1024, 1024, 4, 44, 78, bias_var=0.02),
    "resampler": Config("resampler", "resample", 2, 1, 512, 512, 8, 88, 156, bias_var=0.02),
    "attention": Config("attention", "attn", 3, c=1024, d=4, hw=3432),
    "head": Config("head", "head", 4, 1, 256, 12, 16, 352, 624, bias_var=0.05),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _act(g, n, c, d, h, w, device, std=1.0) -> torch.Tensor:
    x = torch.randn((n, c, d, h, w), generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16).permute(0, 2, 3, 4, 1).contiguous()


def _weight(g, cout, cin, device) -> torch.Tensor:
    w = torch.randn((cout, cin, 3, 3, 3), generator=g, device=device, dtype=torch.float32)
    return (w * math.sqrt(1.0 / (27.0 * cin))).to(torch.bfloat16).contiguous()


def _bias(g, cout, var, device) -> torch.Tensor:
    b = torch.randn((cout,), generator=g, device=device, dtype=torch.float32)
    return (b * math.sqrt(var)).to(torch.bfloat16).contiguous()


def conv_inputs(n, d, h, w, cin, cout, seed, bias_var=0.02, device="cpu", history=False):
    """x [N,D,H,W,Cin], weight [Cout,Cin,3,3,3], bias [Cout] (all bf16);
    with ``history`` also two history frames [N,2,H,W,Cin] drawn last."""
    g = _gen(seed, device)
    out = {"x": _act(g, n, cin, d, h, w, device), "w": _weight(g, cout, cin, device), "b": _bias(g, cout, bias_var, device)}
    if history:
        out["hist"] = _act(g, n, cin, 2, h, w, device)
    return out


def history_frames(n, c, h, w, seed, device="cpu"):
    """Two N(0,1) frames [N, 2, H, W, C] bf16 to carry in front of a chunk's
    input (the previous chunk's last two frames in a streamed decode)."""
    return _act(_gen(seed, device), n, c, 2, h, w, device)


def resample_inputs(n, d, hl, wl, c, seed, bias_var=0.02, device="cpu"):
    """x [N,D,HL,WL,C], weight [C,C,3,3,3], bias [C], skip [N,D,HL,WL,C]."""
    g = _gen(seed, device)
    x = _act(g, n, c, d, hl, wl, device)
    w = _weight(g, c, c, device)
    b = _bias(g, c, bias_var, device)
    s = _act(g, n, c, d, hl, wl, device)
    return {"x": x, "w": w, "b": b, "skip": s}


def attn_inputs(t, hw, c, seed, device="cpu"):
    """q, k, v [T, HW, C] bf16, N(0, 1)."""
    g = _gen(seed, device)
    mk = lambda: torch.randn((t, hw, c), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    q = mk()
    k = mk()
    v = mk()
    return {"q": q, "k": k, "v": v}


def head_inputs(n, d, h, w, cin, seed, bias_var=0.05, cout=12, device="cpu"):
    """x [N,D,H,W,Cin], weight [12,Cin,3,3,3], bias [12]."""
    g = _gen(seed, device)
    return {"x": _act(g, n, cin, d, h, w, device), "w": _weight(g, cout, cin, device), "b": _bias(g, cout, bias_var, device)}


def make_config_inputs(name: str, device="cpu"):
    """Inputs of one named configuration (see ``CONFIGS``)."""
    c = CONFIGS[name]
    if c.kind == "conv":
        return conv_inputs(c.n, c.d, c.h, c.w, c.c, c.cout, c.seed, c.bias_var, device)
    if c.kind == "resample":
        return resample_inputs(c.n, c.d, c.h, c.w, c.c, c.seed, c.bias_var, device)
    if c.kind == "attn":
        return attn_inputs(c.d, c.hw, c.c, c.seed, device)
    if c.kind == "head":
        return head_inputs(c.n, c.d, c.h, c.w, c.c, c.seed, c.bias_var, c.cout, device)
    raise ValueError(name)
