"""Benchmark of the causal-convolution stack on GB300.

One step = one 4-latent-frame chunk through all four stages of the hot path
at the configured sizes, every kernel launched through the C ABI:

  mid-block causal conv 1024->1024 @ 4x44x78          (1 launch)
  attention, 4 frames x 3432 positions x C=1024       (scores, softmax, PV)
  resampler 512->512 @ 8x88x156 -> 8x176x312          (phase convs, interleave)
  output head 256->12 @ 16x352x624                    (one fused kernel)

`value` is milliseconds per chunk for the whole job (with N GPUs each rank
decodes its own chunk: value = max-over-ranks step time / N). Inputs are
synthetic (seeded), resident in HBM; the per-step working set (~4.3 GB) is
far larger than L2, so every step's reads come from DRAM (no explicit flush).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from causal_convolution_gb300 import inputs as cc_inputs  # noqa: E402

METRIC = "causal-conv TFLOP/s (% of bf16 peak); resampler HBM GB/s; ms per 4-frame chunk"
WORKLOAD = ("one 4-latent-frame chunk through the four stages: causal conv 1024->1024 @ 4x44x78; "
            "attention 4x3432xC1024; resampler 512->512 @ 8x88x156 -> 8x176x312; head 256->12 @ 16x352x624")

# The step: every row of the hot path, with the resampler's phase convs and
# interleave (rows a4, a5) fused into one kernel, the attention (rows a6-a8)
# through the key-tile numerators (no fp32 S round trip) and the head's two
# stages (rows a9, a10) fused into one kernel (g never leaves the chip).
KERNELS = ["conv3d_causal", "attn_scores_exp", "attn_exp_rescale", "attn_pv_exp", "resample_up2_fused",
           "head_out_fused"]
# Rows a4, a5, a6-a8 and a9, a10 as the separate passes of the reference
# design, timed in their own loop after the step (not part of the step's time).
ROW_KERNELS = ["resample_phase_conv", "resample_interleave", "attn_scores", "attn_softmax", "attn_pv",
               "head_temporal", "head_stencil", "attn_frame_fused"]


def real_taps(frames: int, taps_per_offset: int) -> int:
    """Taps, summed over output frames 0..frames-1, that read a real input
    frame when the two frames before frame 0 are zeros (temporal offsets 0, 1,
    2 read frames t-2, t-1, t): frame 0 has one real offset, frame 1 two."""
    return taps_per_offset * sum(min(3, t + 1) for t in range(frames))


def algorithmic_work(rescale_bytes: float = 0.0):
    """Per-launch algorithmic work of every kernel: (bound, amount, unit).
    The convolutions count the multiply-adds of taps that read a real input
    frame: with zero history the products with the zero frames before frame
    0 are exact zeros, which the GEMM skips per tile.
    rescale_bytes: what the rescale pass must move for the workload's inputs
    (it reads and writes only the key tiles not yet on their row's scale)."""
    cv = cc_inputs.CONFIGS["mid_conv"]
    at = cc_inputs.CONFIGS["attention"]
    rs = cc_inputs.CONFIGS["resampler"]
    hd = cc_inputs.CONFIGS["head"]
    m_conv = cv.n * cv.d * cv.h * cv.w
    m_res = rs.n * rs.d * rs.h * rs.w
    m_head = hd.n * hd.d * hd.h * hd.w
    t, hw, c = at.d, at.hw, at.c
    ld = (hw + 7) // 8 * 8
    return {
        "conv3d_causal": ("tensor", 2.0 * (m_conv // cv.d) * cv.cout * real_taps(cv.d, 9) * cv.c, "flop"),
        "attn_scores": ("tensor", 2.0 * t * hw * hw * c, "flop"),
        "attn_softmax": ("hbm", t * hw * hw * 4.0 + t * hw * ld * 2.0, "byte"),
        "attn_pv": ("tensor", 2.0 * t * hw * hw * c, "flop"),
        "attn_scores_exp": ("tensor", 2.0 * t * hw * hw * c, "flop"),
        "attn_exp_rescale": ("hbm", rescale_bytes, "byte"),
        "attn_pv_exp": ("tensor", 2.0 * t * hw * hw * c, "flop"),
        "resample_phase_conv": ("tensor", 2.0 * 4 * (m_res // rs.d) * rs.cout * real_taps(rs.d, 4) * rs.c, "flop"),
        "resample_up2_fused": ("tensor", 2.0 * 4 * (m_res // rs.d) * rs.cout * real_taps(rs.d, 4) * rs.c, "flop"),
        "resample_interleave": ("hbm", (4 + 1 + 4) * m_res * rs.c * 2.0, "byte"),
        "head_temporal": ("hbm", m_head * hd.c * 2.0 + m_head * 112 * 2.0, "byte"),
        "head_stencil": ("hbm", m_head * 112 * 2.0 + m_head * 12 * 2.0, "byte"),
        # x read once, the 12-channel output written once; g stays on chip
        # (its multiply-adds, nearly as binding: head_tensor_work)
        "head_out_fused": ("hbm", m_head * hd.c * 2.0 + m_head * 12 * 2.0, "byte"),
        # the attention's useful products (its S is computed C/256 + 1 times)
        "attn_frame_fused": ("tensor", 4.0 * t * hw * hw * c, "flop"),
    }


def head_tensor_work():
    """The fused head's multiply-adds: (useful, executed) flops per launch.
    Useful: the 12-channel 3x3x3 conv over real input frames (the products
    with the causal zero frames are skipped, as in the convolutions).
    Executed: what its MMAs run -- 112 accumulator columns for 108 used, and
    each 32-column block recomputes its two halo columns (strips of 30
    interior columns: ceil(W/30) blocks of 32 columns per row), plus one g row
    above each strip's first block (every strip is one segment here)."""
    hd = cc_inputs.CONFIGS["head"]
    plane = hd.h * hd.w
    useful = 2.0 * plane * 12 * real_taps(hd.d, 9) * hd.c
    strips = -(-hd.w // 30)
    blocks_rows = -(-(hd.h + 2) // 4) * 4  # g rows the blocks of one strip cover
    # every input frame's block feeds the outputs that read it: 3 d - 3 frame pairs
    executed = 2.0 * hd.n * (strips * 32) * blocks_rows * 112 * (3 * hd.d - 3) * hd.c
    return useful, executed


# The source files each kernel is built from (for tying ncu counters to code).
_GEMM_SRC = ["csrc/cc_gemm.cuh", "csrc/cc_gemm_pair.cuh", "csrc/cc_ptx.cuh", "csrc/cc_gemm_launch.cuh",
             "csrc/cc_host.h", "csrc/host.cu"]
KERNEL_SOURCES = {
    "conv3d_causal": _GEMM_SRC + ["csrc/conv.cu"],
    "resample_phase_conv": _GEMM_SRC + ["csrc/conv.cu"],
    "resample_up2_fused": _GEMM_SRC + ["csrc/conv.cu"],
    "head_temporal": _GEMM_SRC + ["csrc/head.cu"],
    "attn_scores": _GEMM_SRC + ["csrc/attn.cu"],
    "attn_pv": _GEMM_SRC + ["csrc/attn.cu"],
    "attn_softmax": ["csrc/attn.cu"],
    "attn_scores_exp": _GEMM_SRC + ["csrc/attn.cu"],
    "attn_exp_rescale": ["csrc/attn.cu", "csrc/cc_gemm.cuh"],
    "attn_pv_exp": _GEMM_SRC + ["csrc/attn.cu"],
    "resample_interleave": ["csrc/passes.cu"],
    "head_stencil": ["csrc/passes.cu"],
    "head_out_fused": _GEMM_SRC + ["csrc/head_fused.cu"],
    "attn_frame_fused": _GEMM_SRC + ["csrc/attn.cu", "csrc/attn_fused.cu"],
}


def kernel_source_hash(kernel: str) -> str:
    """sha256 over the sources `kernel` is built from."""
    import hashlib
    hsh = hashlib.sha256()
    for rel in sorted(KERNEL_SOURCES[kernel]):
        hsh.update(rel.encode())
        with open(os.path.join(ROOT, "causal_convolution_gb300", rel), "rb") as f:
            hsh.update(f.read())
    return hsh.hexdigest()


def measured_traffic():
    """Per-launch DRAM bytes (read + write) from committed ncu captures, for
    the kernels whose sources are unchanged since their capture."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return {}
    return {k: v["dram_bytes"] for k, v in t.get("kernels", {}).items()
            if k in KERNEL_SOURCES and v.get("source_sha256") == kernel_source_hash(k)}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# CTAs of the read-back copy kernel in the end-to-end loop: 4-16 gave the
# same chunk time (10.46-10.53 ms), 2 a little more, the copy engine 10.86.
E2E_READBACK_CTAS = 8

# ------------------------------------------------------------------ clocks --

class ClockSampler:
    """nvidia-smi samples (every 50 ms) of this GPU while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw.instant,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.samples = []
        self.proc = None
        self.thread = None
        sel = []
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            sel = []
        self.cmd = ["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 7:
                self.samples.append(parts)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm, mx, watts, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in self.samples:
            try:
                sm.append(float(s[0]))
                mx.append(float(s[1]))
            except ValueError:
                continue
            try:
                watts.append(float(s[2]))
            except ValueError:
                pass
            for name, val in zip(names, s[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_median": round(statistics.median(watts), 1) if watts else None,
                "power_w_max": round(max(watts), 1) if watts else None}


# ---------------------------------------------------------------- workload --

class Workload:
    """All inputs, prepared weights, workspaces and outputs of one chunk, on one GPU."""

    STAGE_OF = {"conv3d_causal": "conv", "attn_scores_exp": "attn", "attn_exp_rescale": "attn", "attn_pv_exp": "attn",
                "resample_up2_fused": "res", "head_out_fused": "head", "resample_phase_conv": "res",
                "resample_interleave": "res", "attn_scores": "attn", "attn_softmax": "attn", "attn_pv": "attn",
                "head_temporal": "head", "head_stencil": "head", "attn_frame_fused": "attn"}

    def __init__(self, device, stages=("conv", "attn", "res", "head"), history=True):
        from causal_convolution_gb300 import api
        self.api = api
        self.dev = device
        bf = torch.bfloat16
        E = lambda *s, dt=bf: torch.empty(s, dtype=dt, device=device)
        mk = cc_inputs.make_config_inputs

        cv = cc_inputs.CONFIGS["mid_conv"]
        at = cc_inputs.CONFIGS["attention"]
        rs = cc_inputs.CONFIGS["resampler"]
        hd = cc_inputs.CONFIGS["head"]
        self.cv, self.at, self.rs, self.hd = cv, at, rs, hd
        self.scale = at.c ** -0.5
        hf = cc_inputs.history_frames
        if "conv" in stages:
            i = mk("mid_conv", device)
            self.conv_x, self.conv_b = i["x"], i["b"]
            self.conv_wp = E(27 * cv.cout * cv.c)
            api.cc_conv3d_prepare(i["w"], self.conv_wp)
            self.conv_y = E(cv.n, cv.d, cv.h, cv.w, cv.cout)

        if "attn" in stages:
            i = mk("attention", device)
            self.q, self.k, self.v = i["q"], i["k"], i["v"]
            self.ld = api.cc_attn_ld(at.hw)
            self.s = E(at.d, at.hw, self.ld, dt=torch.float32)
            self.p = E(at.d, at.hw, self.ld)
            self.o = E(at.d, at.hw, at.c)
            self.e = E(at.d, at.hw, self.ld)
            self.st = E(at.d, at.hw, api.cc_attn_exp_key_tiles(at.hw), 2, dt=torch.float32)
            self.fws = E(api.cc_attn_fused_workspace_bytes(at.d, at.hw), dt=torch.uint8)

        if "res" in stages:
            i = mk("resampler", device)
            self.res_x, self.res_b, self.res_skip = i["x"], i["b"], i["skip"]
            self.res_pw = E(48 * rs.cout * rs.c)
            api.cc_resample_prepare(i["w"], self.res_pw)
            self.phases = E(4, rs.n, rs.d, rs.h, rs.w, rs.cout)
            self.res_out = E(rs.n, rs.d, 2 * rs.h, 2 * rs.w, rs.cout)

        if "head" in stages:
            i = mk("head", device)
            self.head_x, self.head_b = i["x"], i["b"]
            self.head_wp = E(3 * api.HEAD_G_CH * hd.c)
            api.cc_head_prepare(i["w"], self.head_wp)
            self.g = E(hd.n, hd.d, hd.h, hd.w, api.HEAD_G_CH)
            self.head_out = E(hd.n, hd.d, hd.h, hd.w, api.HEAD_COUT)

        # a later chunk of a streamed decode: the causal stages get the previous
        # chunk's last two input frames in front (hist = 2) instead of zeros
        if history:
            self.conv_xh = torch.cat([hf(cv.n, cv.c, cv.h, cv.w, 101, device), self.conv_x], 1)
            self.res_xh = torch.cat([hf(rs.n, rs.c, rs.h, rs.w, 102, device), self.res_x], 1)
            self.head_xh = torch.cat([hf(hd.n, hd.c, hd.h, hd.w, 104, device), self.head_x], 1)
        torch.cuda.synchronize(device)
        api.cc_check_device()

    def launches(self, stream, hist: int = 0):
        """The hot path as (stage, launch) pairs in launch order, one per entry
        of KERNELS; hist = 2 feeds the causal stages two carried history frames."""
        a = self.api
        pick = lambda name: getattr(self, name + ("h" if hist else ""), None)
        cx, rx, hx = pick("conv_x"), pick("res_x"), pick("head_x")
        return (
            ("conv", lambda: a.cc_conv3d_causal(cx, self.conv_wp, self.conv_b, self.conv_y, hist=hist, stream=stream)),
            ("attn", lambda: a.cc_attn_scores_exp(self.q, self.k, self.e, self.st, self.scale, stream=stream)),
            ("attn", lambda: a.cc_attn_exp_rescale(self.e, self.st, self.at.hw, stream=stream)),
            ("attn", lambda: a.cc_attn_pv_exp(self.e, self.st, self.v, self.o, stream=stream)),
            ("res", lambda: a.cc_resample_up2_fused(rx, self.res_pw, self.res_b, self.res_skip, self.res_out,
                                                    hist=hist, stream=stream)),
            ("head", lambda: a.cc_head_out_fused(hx, self.head_wp, self.head_b, self.head_out, hist=hist,
                                                 stream=stream)),
        )

    def step(self, stream, ev=None, hist: int = 0, around=None):
        """The whole hot path once. With `ev` (len(KERNELS)+1 events) each launch is bracketed;
        with `around` = (j, before, after) only launch j is. An event between two launches costs
        the later one its overlap with the earlier (programmatic dependent launch): ~4.6 us each."""
        if ev is not None:
            ev[0].record(stream)
        for j, (_, launch) in enumerate(self.launches(stream, hist)):
            if around is not None and j == around[0]:
                around[1].record(stream)
            launch()
            if ev is not None:
                ev[j + 1].record(stream)
            if around is not None and j == around[0]:
                around[2].record(stream)

    def row_launches(self, stream):
        """Rows a4, a5 as two passes through the phase tensors, rows a6-a8 as
        three passes through fp32 S and bf16 P, and rows a9, a10 as two passes
        through the bf16 g, one launch per entry of ROW_KERNELS."""
        a = self.api
        return (
            lambda: a.cc_resample_phase_conv(self.res_x, self.res_pw, self.phases, stream=stream),
            lambda: a.cc_resample_interleave(self.phases, self.res_b, self.res_skip, self.res_out, stream=stream),
            lambda: a.cc_attn_scores(self.q, self.k, self.s, stream=stream),
            lambda: a.cc_attn_softmax(self.s, self.p, self.at.hw, self.scale, stream=stream),
            lambda: a.cc_attn_pv(self.p, self.v, self.o, self.at.hw, stream=stream),
            lambda: a.cc_head_temporal(self.head_x, self.head_wp, self.g, stream=stream),
            lambda: a.cc_head_stencil(self.g, self.head_b, self.head_out, stream=stream),
            lambda: a.cc_attn_frame_fused(self.q, self.k, self.v, self.o, self.fws, self.scale, stream=stream),
        )

    def rows(self, stream, ev):
        """The ROW_KERNELS launches, each bracketed by events (len(ROW_KERNELS)+1)."""
        launches = self.row_launches(stream)
        ev[0].record(stream)
        for j, launch in enumerate(launches):
            launch()
            ev[j + 1].record(stream)

    def rescale_bytes(self, stream) -> float:
        """Bytes the rescale pass moves for these inputs: each key tile whose
        c_t is below its row's largest is read and written once (bf16), and
        every row's statistics are read (8 bytes per tile) and those of the
        rescaled tiles written."""
        self.api.cc_attn_scores_exp(self.q, self.k, self.e, self.st, self.scale, stream=stream)
        torch.cuda.synchronize(self.dev)
        st = self.st.cpu().numpy()
        c = st[..., 0]
        moved = c < c.max(axis=2, keepdims=True)
        tiles = c.shape[2]
        keys = np.minimum(256, self.at.hw - 256 * np.arange(tiles))  # keys per tile (last one partial)
        return float(2 * 2 * (moved * keys).sum() + 8 * c.size + 8 * moved.sum())

    # ---- end to end through host buffers -------------------------------
    # Stages in launch order: (inputs copied in, launches, outputs copied back).
    STAGES = (("conv", ("conv_x",), ("conv_y",)),
              ("attn", ("q", "k", "v"), ("o",)),
              ("res", ("res_x", "res_skip"), ("res_out",)),
              ("head", ("head_x",), ("head_out",)))

    def host_buffers(self):
        pin = lambda t: torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t)
        self.d_in = {"conv_x": self.conv_x, "q": self.q, "k": self.k, "v": self.v, "res_x": self.res_x,
                     "res_skip": self.res_skip, "head_x": self.head_x}
        self.d_out = {"conv_y": self.conv_y, "o": self.o, "res_out": self.res_out, "head_out": self.head_out}
        self.h_in = {n: pin(t) for n, t in self.d_in.items()}
        self.h_out = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in self.d_out.items()}
        # one copy-in stream (more streams gave no more host-link bandwidth) and
        # one read-back stream
        self.s_h2d = torch.cuda.Stream(self.dev)
        self.s_d2h = torch.cuda.Stream(self.dev)
        nst = len(self.STAGES)
        self.ev_in = [torch.cuda.Event() for _ in range(nst)]    # stage inputs landed
        self.ev_used = [torch.cuda.Event() for _ in range(nst)]  # stage kernels done
        self.ev_out = [torch.cuda.Event() for _ in range(nst)]   # stage outputs read back
        self.e2e_primed = False
        h2d = sum(t.numel() * t.element_size() for t in self.h_in.values())
        d2h = sum(t.numel() * t.element_size() for t in self.h_out.values())
        return h2d, d2h

    def step_e2e(self, stream, h_in=None, h_out=None):
        """One chunk from pinned host inputs (`h_in`, default the ones
        `host_buffers` made) to pinned host outputs (`h_out`): the same
        seven launches as `step`. Inputs go in stage by stage on the copy-in
        stream, each stage's launches wait only for their own inputs, and each
        output goes back as soon as its stage ends, so copies overlap compute
        (and the previous chunk's copies) but never a buffer still in use:
        a stage's inputs are rewritten only after its kernels of the previous
        chunk have finished, and its outputs only after they were read back."""
        h_in = self.h_in if h_in is None else h_in
        h_out = self.h_out if h_out is None else h_out
        launches = self.launches(stream)
        for i, (_, ins, _) in enumerate(self.STAGES):
            if self.e2e_primed:
                self.s_h2d.wait_event(self.ev_used[i])
            with torch.cuda.stream(self.s_h2d):
                for name in ins:
                    self.d_in[name].copy_(h_in[name], non_blocking=True)
            self.ev_in[i].record(self.s_h2d)
        for i, (stage, _, outs) in enumerate(self.STAGES):
            stream.wait_event(self.ev_in[i])
            if self.e2e_primed:
                stream.wait_event(self.ev_out[i])
            for st, launch in launches:
                if st == stage:
                    launch()
            self.ev_used[i].record(stream)
            self.s_d2h.wait_event(self.ev_used[i])
            # read back by the library's copy kernel (a few CTAs storing to
            # the mapped pinned buffers): beside the copy-engine copy-in it
            # leaves that copy nearly its whole link bandwidth
            for name in outs:
                self.api.cc_copy_to_host(h_out[name], self.d_out[name], ctas=E2E_READBACK_CTAS, stream=self.s_d2h)
            self.ev_out[i].record(self.s_d2h)
        self.e2e_primed = True


# -------------------------------------------------------------- CPU oracle --

# outputs per oracle call for conv, attention, resampler, head: large enough
# that each call's setup (the conv widens and slices 27 weight taps of 8 MB
# per call) is a small part of its time
ORACLE_BATCH = (512, 1024, 2048, 8192)


def oracle_sample_step(cpu, budget_s: float, rng, per_config=None):
    """Times the fp64 oracle on a bounded sample of each stage's outputs and
    extrapolates by output count to ms per chunk. Returns (ms_per_chunk,
    seconds spent, description). With a dict `per_config`, each stage's
    figures go into it: seconds per chunk (extrapolated), outputs sampled,
    outputs in the configuration, the sampled fraction and seconds spent."""
    import oracle

    total_ms = 0.0
    spent = 0.0
    desc = []
    per_stage = budget_s / 4.0

    def timed(fn, total, batch):
        """Calls of `batch` sampled outputs until the stage's share of the
        budget is spent (at least one) or the configuration's outputs are all
        counted; returns (points, seconds, ms per chunk). The batch is fixed
        per stage (the last call may be shorter), so the per-call setup is
        spread over the same number of outputs whatever the budget."""
        npts, dt = 0, 0.0
        # until the stage's share of the budget is spent, or as many outputs
        # as the configuration has were timed
        while npts == 0 or (dt < per_stage and npts < total):
            b = min(batch, total - npts)  # the last call stops at the configuration's count
            t0 = time.perf_counter()
            fn(b)
            dt += time.perf_counter() - t0
            npts += b
        return npts, dt, dt / npts * total * 1e3

    stages = []
    cv = cc_inputs.CONFIGS["mid_conv"]
    stages.append(("conv", cv.n * cv.d * cv.h * cv.w,
                   lambda P: oracle.causal_conv3d_at(cpu["conv_x"], cpu["conv_w"], cpu["conv_b"],
                                                     _pts(rng, P, cv.n, cv.d, cv.h, cv.w))))
    at = cc_inputs.CONFIGS["attention"]
    stages.append(("attention", at.d * at.hw,
                   lambda P: oracle.attn_frame_rows(cpu["q"], cpu["k"], cpu["v"],
                                                    np.stack([rng.integers(0, at.d, P), rng.integers(0, at.hw, P)], 1))))
    rs = cc_inputs.CONFIGS["resampler"]
    stages.append(("resampler", rs.n * rs.d * 4 * rs.h * rs.w,
                   lambda P: oracle.resample_up2_at(cpu["res_x"], cpu["res_w"], cpu["res_b"], cpu["res_skip"],
                                                    _pts(rng, P, rs.n, rs.d, 2 * rs.h, 2 * rs.w))))
    hd = cc_inputs.CONFIGS["head"]
    hf = cpu["head_x"].shape[1]  # frames held on the host (the first ones)
    stages.append(("head", hd.n * hd.d * hd.h * hd.w,
                   lambda P: oracle.head_out_at(cpu["head_x"], cpu["head_w"], cpu["head_b"],
                                                _pts(rng, P, hd.n, hf, hd.h, hd.w))))
    for (name, total, fn), batch in zip(stages, ORACLE_BATCH):
        npts, dt, ms = timed(fn, total, batch)
        spent += dt
        total_ms += ms
        desc.append(f"{name}: {npts} of {total} outputs in batches of {batch}")
        if per_config is not None:
            per_config[name] = {"seconds_per_chunk": round(ms * 1e-3, 3), "outputs_sampled": npts,
                                "outputs_per_chunk": total, "fraction_sampled": round(npts / total, 6),
                                "seconds_spent": round(dt, 3)}
    return total_ms, spent, "; ".join(desc) + " (extrapolated by output count)"


def oracle_toy_resampler(per_config):
    """The toy resampler configuration through the fp64 oracle in full (it
    finishes in well under a second): wall-clock seconds, nothing sampled."""
    import oracle

    i = cc_inputs.make_config_inputs("toy_resampler", "cpu")
    f = lambda t: t.double().numpy()
    args = (f(i["x"]), f(i["w"]), f(i["b"]), f(i["skip"]))
    t0 = time.perf_counter()
    out = oracle.resample_up2(*args)
    dt = time.perf_counter() - t0
    per_config["toy_resampler"] = {"seconds_per_chunk": round(dt, 4), "outputs_sampled": int(out.size // out.shape[-1]),
                                   "outputs_per_chunk": int(out.size // out.shape[-1]), "fraction_sampled": 1.0,
                                   "seconds_spent": round(dt, 4)}


def _pts(rng, p, n, d, h, w):
    return np.stack([rng.integers(0, n, p), rng.integers(0, d, p), rng.integers(0, h, p), rng.integers(0, w, p)], 1)


def host_inputs(device, head_frames=3):
    """The oracle's inputs on the host, already float64 (the oracle widens its
    inputs on every call otherwise); the head keeps its first frames only:
    sampled outputs there need frames t-2..t, all held."""
    f = lambda t: t.double().cpu().numpy()
    out = {}
    i = cc_inputs.make_config_inputs("mid_conv", device)
    out.update(conv_x=f(i["x"]), conv_w=f(i["w"]), conv_b=f(i["b"]))
    i = cc_inputs.make_config_inputs("attention", device)
    out.update(q=f(i["q"]), k=f(i["k"]), v=f(i["v"]))
    i = cc_inputs.make_config_inputs("resampler", device)
    out.update(res_x=f(i["x"]), res_w=f(i["w"]), res_b=f(i["b"]), res_skip=f(i["skip"]))
    i = cc_inputs.make_config_inputs("head", device)
    out.update(head_x=f(i["x"][:, :head_frames]), head_w=f(i["w"]), head_b=f(i["b"]))
    return out


def cpu_threads():
    """Threads the oracle's numpy matmuls run on (the BLAS pool), else the
    host's CPU count."""
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads") for d in threadpool_info() if d.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        try:
            return int(os.environ[var])
        except (KeyError, ValueError):
            pass
    return os.cpu_count() or 1


def host_facts():
    """nproc (CPUs this process may run on), the host's CPU count and the
    thread counts the oracle's libraries are set to use."""
    try:
        nproc = len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        nproc = os.cpu_count() or 1
    return {"nproc": nproc, "cpu_count": os.cpu_count(), "blas_threads": cpu_threads(),
            "omp_num_threads": os.environ.get("OMP_NUM_THREADS")}


# -------------------------------------------------------------------- main --

def config_dict(n_gpus):
    return {"workload": WORKLOAD, "chunks_per_step": n_gpus, "global_batch": n_gpus, "seq_len": 4,
            "parallelism": f"replicas{n_gpus}" if n_gpus > 1 else "single",
            "l2": "per-step working set ~4.3 GB > 126 MB L2: inputs larger than L2, no explicit flush"}


def max_over_ranks(value: float, device) -> float:
    """The maximum of `value` over all ranks (identity without a process group)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def run_reference(args):
    ws, rank, local = dist_setup()
    if rank != 0:
        return 0
    device = "cuda:0" if torch.cuda.is_available() else "cpu"
    cpu = host_inputs(device)
    rng = np.random.default_rng(0)
    # each step a bounded sample: the whole run stays near --ref-total-s
    step_s = min(args.ref_step_s, args.ref_total_s / (args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample_step(cpu, step_s, rng)
    vals, spent, desc = [], 0.0, ""
    per_config = {}
    t0 = time.perf_counter()
    for _ in range(args.steps):
        v, s, desc = oracle_sample_step(cpu, step_s, rng, per_config)
        vals.append(v)
        spent += s
    wall = time.perf_counter() - t0
    oracle_toy_resampler(per_config)
    value = float(np.mean(vals)) / max(args.gpus, 1)
    cores = cpu_threads()
    line = {"metric": METRIC, "value": value, "unit": "ms", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": wall * 1e3 / args.steps, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(args.gpus), "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "ms", "cores": cores, "kind": "oracle",
                             "sample": f"per step: {desc}; fp64 numpy oracle on {cores} host threads",
                             "per_config_last_step": per_config, **host_facts()},
            "e2e": {"value": value, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_profile_kernel(args):
    """One kernel of the step on its bench workload, nothing else launched
    after the set-up: `ncu -k regex:<kernel> -s <warmup> -c 1` then captures
    exactly one launch."""
    torch.cuda.set_device(0)
    device = torch.device("cuda:0")
    from causal_convolution_gb300 import _lib
    if not os.path.exists(_lib.LIB_PATH):
        from causal_convolution_gb300 import build
        build.build()
    wl = Workload(device, stages=(Workload.STAGE_OF[args.profile_kernel],), history=False)
    stream = torch.cuda.Stream(device)
    names = KERNELS + ROW_KERNELS
    launches = [launch for _, launch in wl.launches(stream)] + list(wl.row_launches(stream))
    launch = launches[names.index(args.profile_kernel)]
    if args.profile_kernel == "attn_pv_exp":  # its inputs: E and statistics from the scores kernel
        wl.api.cc_attn_scores_exp(wl.q, wl.k, wl.e, wl.st, wl.scale, stream=stream)
        wl.api.cc_attn_exp_rescale(wl.e, wl.st, wl.at.hw, stream=stream)
    elif args.profile_kernel == "attn_pv":
        wl.api.cc_attn_scores(wl.q, wl.k, wl.s, stream=stream)
        wl.api.cc_attn_softmax(wl.s, wl.p, wl.at.hw, wl.scale, stream=stream)
    torch.cuda.synchronize(device)
    for _ in range(args.warmup + args.steps):
        launch()
    torch.cuda.synchronize(device)
    wl.api.cc_check_device()
    print(f"profile-kernel {args.profile_kernel}: {args.warmup + args.steps} launches", flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget-s", type=float, default=16.0)
    ap.add_argument("--ref-step-s", type=float, default=4.0)
    ap.add_argument("--ref-total-s", type=float, default=150.0)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--profile-kernel", choices=KERNELS + ROW_KERNELS, default=None,
                    help="launch only this kernel of the step, warmup + steps times, and print nothing else "
                         "(the target of one-kernel ncu captures)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.profile_kernel:
        return run_profile_kernel(args)

    ws, rank, local = dist_setup()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    torch.cuda.set_device(local)
    device = torch.device(f"cuda:{local}")

    from causal_convolution_gb300 import _lib
    if not os.path.exists(_lib.LIB_PATH):
        from causal_convolution_gb300 import build
        build.build()

    wl = Workload(device)
    stream = torch.cuda.Stream(device)
    # warm-up steps, the last ones with every launch bracketed: they pick the
    # dominant kernel, the only one bracketed inside the timed region
    wev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(KERNELS) + 1)] for _ in range(args.warmup)]
    for k in range(args.warmup):
        wl.step(stream, wev[k] if k >= args.warmup - 2 else None)
    torch.cuda.synchronize(device)
    wl.api.cc_check_device()
    warm_ms = {name: float(np.mean([wev[k][j].elapsed_time(wev[k][j + 1]) for k in range(args.warmup - 2, args.warmup)]))
               for j, name in enumerate(KERNELS)}
    dominant = max(KERNELS, key=lambda n: warm_ms[n])
    dj = KERNELS.index(dominant)

    # the timed region: steps back to back; events only around the dominant
    # kernel (its launch duration for the roofline, and the step period from
    # one of its starts to the next)
    ev_a = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev_b = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(device)
    clocks.start()
    time.sleep(0.25)
    t_start.record(stream)
    for k in range(args.steps):
        wl.step(stream, around=(dj, ev_a[k], ev_b[k]))
    t_end.record(stream)
    torch.cuda.synchronize(device)
    clocks.stop()
    if ws > 1:
        torch.distributed.barrier()
    wl.api.cc_check_device()
    elapsed = t_start.elapsed_time(t_end)
    dom_times = [ev_a[k].elapsed_time(ev_b[k]) for k in range(args.steps)]
    step_times = [ev_a[k].elapsed_time(ev_a[k + 1]) for k in range(args.steps - 1)] or [elapsed]
    ms_step = max_over_ranks(elapsed / args.steps, device)

    # every launch of the step bracketed by events, outside the timed region:
    # the per-kernel table (each time includes the gap before the next launch)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(KERNELS) + 1)] for _ in range(args.steps)]
    for k in range(args.steps):
        wl.step(stream, evs[k])
    torch.cuda.synchronize(device)
    wl.api.cc_check_device()
    per_kernel = {name: float(np.mean([evs[k][j].elapsed_time(evs[k][j + 1]) for k in range(args.steps)]))
                  for j, name in enumerate(KERNELS)}
    per_kernel_stats = {name: (float(np.median([evs[k][j].elapsed_time(evs[k][j + 1]) for k in range(args.steps)])),
                               float(np.min([evs[k][j].elapsed_time(evs[k][j + 1]) for k in range(args.steps)])))
                        for j, name in enumerate(KERNELS)}
    bracketed_step_ms = float(np.mean([evs[k][0].elapsed_time(evs[k][-1]) for k in range(args.steps)]))
    per_kernel_bracketed_dominant = per_kernel[dominant]
    per_kernel[dominant] = float(np.mean(dom_times))  # the timed region's own measurement
    per_kernel_stats[dominant] = (float(np.median(dom_times)), float(np.min(dom_times)))

    # steady state: the same step on a later chunk of a streamed decode (two
    # carried history frames, so no zero-padding taps to skip), outside the
    # timed region of `value`
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(KERNELS) + 1)] for _ in range(args.steps)]
    for _ in range(args.warmup):
        wl.step(stream, hist=2)
    for k in range(args.steps):
        wl.step(stream, sev[k], hist=2)
    torch.cuda.synchronize(device)
    steady = {name: float(np.mean([sev[k][j].elapsed_time(sev[k][j + 1]) for k in range(args.steps)]))
              for j, name in enumerate(KERNELS)}
    steady_ms = float(np.mean([sev[k][0].elapsed_time(sev[k][-1]) for k in range(args.steps)]))
    wl.api.cc_check_device()

    # the resampler's two-pass form (rows a4, a5), outside the step
    rev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(ROW_KERNELS) + 1)] for _ in range(args.steps)]
    for _ in range(2):
        wl.rows(stream, rev[0])
    for k in range(args.steps):
        wl.rows(stream, rev[k])
    torch.cuda.synchronize(device)
    for j, name in enumerate(ROW_KERNELS):
        per_kernel[name] = float(np.mean([rev[k][j].elapsed_time(rev[k][j + 1]) for k in range(args.steps)]))
    wl.api.cc_check_device()

    # end to end: host buffers, copies inside the timed region
    h2d, d2h = wl.host_buffers()
    for _ in range(3):
        wl.step_e2e(stream)
    torch.cuda.synchronize(device)
    if ws > 1:
        torch.distributed.barrier()
    e0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        wl.step_e2e(stream)
    torch.cuda.synchronize(device)
    e2e_ms = max_over_ranks((time.perf_counter() - e0) * 1e3 / args.e2e_steps, device)
    wl.api.cc_check_device()

    peaks = load_peaks()
    work = algorithmic_work(wl.rescale_bytes(stream))
    roofs = {}
    for name in KERNELS + ROW_KERNELS:
        bound, amount, unit = work[name]
        sec = per_kernel[name] * 1e-3
        if bound == "tensor":
            ach = amount / sec / 1e12
            peak = peaks["bf16_tflops"]
            roofs[name] = {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
                           "ms": per_kernel[name], "work": amount, "in_step": name in KERNELS}
        else:
            ach = amount / sec / 1e9
            peak = peaks["hbm_gbs"]
            roofs[name] = {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
                           "ms": per_kernel[name], "work": amount, "in_step": name in KERNELS}
    traffic = measured_traffic()
    for name in roofs:
        roofs[name]["traffic"] = traffic.get(name)  # per-launch DRAM bytes from ncu, None if stale
        if traffic.get(name):  # the same launch's DRAM bytes over its time, GB/s
            roofs[name]["traffic_gbs"] = traffic[name] / (per_kernel[name] * 1e-3) / 1e9
        if name in per_kernel_stats:
            roofs[name]["ms_median"], roofs[name]["ms_min"] = per_kernel_stats[name]
    # the fused head against the tensor roof too: its useful multiply-adds
    # take nearly as long at the bf16 peak as its bytes at the copy peak
    hu, hx = head_tensor_work()
    hsec = per_kernel["head_out_fused"] * 1e-3
    roofs["head_out_fused"]["tensor"] = {
        "achieved": hu / hsec / 1e12, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
        "frac": hu / hsec / 1e12 / peaks["bf16_tflops"], "work": hu, "executed_work": hx,
        "executed_frac": hx / hsec / 1e12 / peaks["bf16_tflops"]}
    # the whole step against the tensor roof: the useful flops of its five
    # tensor-core stages over the step's time
    step_flops = sum(work[n][1] for n in ("conv3d_causal", "attn_scores_exp", "attn_pv_exp", "resample_up2_fused")) + hu
    step_roof = {"useful_tflop": round(step_flops / 1e12, 4),
                 "achieved": round(step_flops / (ms_step * 1e-3) / 1e12, 2), "peak": peaks["bf16_tflops"],
                 "unit": "TFLOP/s", "frac": round(step_flops / (ms_step * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
                 "what": "conv + attention scores and PV + fused resampler + fused head multiply-adds (real taps) "
                         "per step time, against the burst bf16 peak"}
    dr = roofs[dominant]
    roofline = {"bound": dr["bound"], "achieved": round(dr["achieved"], 2), "peak": dr["peak"], "unit": dr["unit"],
                "frac": round(dr["frac"], 4), "traffic": traffic.get(dominant), "kernel": dominant,
                "timing": f"CUDA events around each of its {args.steps} launches in the timed region",
                "peak_source": f"{peaks['source']} ({'burst bf16 GEMM' if dr['bound'] == 'tensor' else 'copy'})"}

    line = {
        "metric": METRIC, "value": round(ms_step / ws, 4), "unit": "ms", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded normal inputs, fan-in-scaled weights)",
        "step_ms_stats": {"mean": round(float(np.mean(step_times)), 4), "median": round(float(np.median(step_times)), 4),
                          "min": round(float(np.min(step_times)), 4),
                          "what": "period from one step's dominant launch to the next one's, in the timed region"},
        "per_kernel_timing": {"what": "kernels[*].ms: the step again, every launch bracketed by CUDA events, after "
                                      "the timed region (each includes the gap before the next launch; an event "
                                      "between two launches stops the later one's early start); the dominant "
                                      "kernel's from the timed region",
                              "bracketed_step_ms": round(bracketed_step_ms, 4),
                              "dominant_bracketed_ms": round(per_kernel_bracketed_dominant, 4)},
        "config": config_dict(ws),
        "conv_tflops": round(roofs["conv3d_causal"]["achieved"], 2),
        "conv_frac_of_bf16_peak": round(roofs["conv3d_causal"]["frac"], 4),
        "resampler_interleave_gbs": round(roofs["resample_interleave"]["achieved"], 1),
        "resampler_interleave_frac_of_hbm": round(roofs["resample_interleave"]["frac"], 4),
        "head_stencil_gbs": round(roofs["head_stencil"]["achieved"], 1),
        "stage_ms": {"conv": per_kernel["conv3d_causal"],
                     "attention": per_kernel["attn_scores_exp"] + per_kernel["attn_exp_rescale"]
                     + per_kernel["attn_pv_exp"],
                     "attention_three_pass": per_kernel["attn_scores"] + per_kernel["attn_softmax"]
                     + per_kernel["attn_pv"],
                     "resampler": per_kernel["resample_up2_fused"],
                     "resampler_two_pass": per_kernel["resample_phase_conv"] + per_kernel["resample_interleave"],
                     "attention_fused": per_kernel["attn_frame_fused"],
                     "head": per_kernel["head_out_fused"],
                     "head_two_pass": per_kernel["head_temporal"] + per_kernel["head_stencil"]},
        "kernels": {n: {k: (round(v, 4) if isinstance(v, float) else
                            {kk: (round(vv, 4) if isinstance(vv, float) else vv) for kk, vv in v.items()}
                            if isinstance(v, dict) else v)
                        for k, v in r.items()}
                    for n, r in roofs.items()},
        "traffic_source": "profiles/ncu_traffic.json (per-launch dram read+write of one ncu capture; null when the "
                          "kernel's sources changed since)",
        "roofline": roofline,
        "step_roofline": step_roof,
        "steady_state": {"ms_per_step": round(steady_ms, 4),
                         "what": "the same step on a later chunk of a streamed decode: conv, resampler and head get "
                                 "the previous chunk's last two input frames (hist=2) instead of the zero frames, so "
                                 "no tap can be skipped",
                         "kernels_ms": {n: round(v, 4) for n, v in steady.items()}},
        "e2e": {"value": round(e2e_ms / ws, 4), "unit": "ms", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": len(KERNELS) * args.steps,
        "clocks": clocks.summary(),
    }

    if rank == 0 and not args.no_cpu_baseline:
        cpu = host_inputs(device)
        per_config = {}
        v, spent, desc = oracle_sample_step(cpu, args.cpu_budget_s, np.random.default_rng(0), per_config)
        oracle_toy_resampler(per_config)
        line["cpu_baseline"] = {"value": round(v, 1), "unit": "ms", "cores": cpu_threads(), "kind": "oracle",
                                "sample": f"{desc}; {spent:.1f} s of fp64 numpy oracle work",
                                "per_config": per_config, **host_facts()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
