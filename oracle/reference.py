"""Plain fp64 CPU oracle for the Wan2.2 VAE-decoder causal-convolution stack.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this module:
only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it. It shares no code with the CUDA path.

Every function takes numpy arrays (any float dtype; they are widened to
float64), applies no intermediate rounding and returns float64. Activations
are channels-last: ``[N, D, H, W, C]``. Weights keep the PyTorch Conv3d
order ``[C_out, C_in, kt, kh, kw]``.

Sources (pages of the reference material, by title and item):

* "FastVideo wan22_vae_decode solution/attn.cu", header comment: one head of
  softmax(q k^T / 32) v per latent frame over H*W positions, C=1024, no mask;
  the host code computes the scale as 1/sqrt(C) and the GEMM problem is a
  cross-correlation (no kernel flip).
* "FastVideo wan22_vae_decode solution/resample.h", header comment: the
  resampler is nearest x2 in space followed by a 3x3x3 convolution; bias and
  the nearest-duplicated shortcut are added after the convolution. The
  comment on ``resample_upsample``: the input carries two causal history
  frames in time and one row of zero padding.
* "FastVideo wan22_vae_decode solution/head.cu", header comment and
  ``head_stencil_kernel``: conv_out to 12 channels, bias, clamp to [-1, 1],
  zero padding in the plane; the two-stage split (temporal 3x1x1 conv into
  9x12 channels, then a 3x3 spatial sum) is the same sum regrouped.
* The stack's definition: a causal 3x3x3 convolution with two history frames
  (zeros before frame 0 of a first chunk) and spatial zero padding of 1, the
  history frames and padding the ``resample_upsample`` comment also names.

Readings where the pages are silent (each one is listed with its reason in the
design notes of the repository):

* Temporal alignment: tap kt reads frame t + kt - 2 (causal front padding of
  two frames); kh, kw read h + kh - 1, w + kw - 1.
* The resampler's shortcut has the input's channel count and is duplicated
  x2 in space only (no temporal duplication, no channel-to-row rearrangement).
* Attention normalises over keys (rows of P sum to one).
* The clamp is applied after the bias, to the closed interval [-1, 1].
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "causal_conv3d",
    "causal_conv3d_at",
    "nearest_up2",
    "resample_up2",
    "resample_up2_at",
    "resample_phase_kernels",
    "resample_phase_conv",
    "resample_interleave",
    "resample_up2_four_phase",
    "resample_phase_kernels_temporal",
    "resample_up2_temporal_eight_phase",
    "attn_probs",
    "attn_frame",
    "attn_frame_rows",
    "head_out",
    "head_out_at",
    "head_stage_a",
    "head_stage_b",
    "head_two_stage",
]


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def _pad_causal(x: np.ndarray, history: np.ndarray | None) -> np.ndarray:
    """x [N,D,H,W,C] -> [N,D+2,H+2,W+2,C]: two frames in front (zeros, or the
    given history), one zero row/column on each side in the plane."""
    n, d, h, w, c = x.shape
    xp = np.zeros((n, d + 2, h + 2, w + 2, c), dtype=np.float64)
    xp[:, 2:, 1:-1, 1:-1, :] = x
    if history is not None:
        hist = _f64(history)
        assert hist.shape == (n, 2, h, w, c), hist.shape
        xp[:, :2, 1:-1, 1:-1, :] = hist
    return xp


def causal_conv3d(x, w, b=None, history=None) -> np.ndarray:
    """Causal 3x3x3 convolution, the plain definition.

    y[n,t,h,w,co] = b[co] + sum_{ci,kt,kh,kw} w[co,ci,kt,kh,kw]
                                  * x~[n, t+kt-2, h+kh-1, w+kw-1, ci]

    with x~ = 0 outside the plane and, before frame 0, either zeros
    (``history=None``) or the two given history frames ``[N,2,H,W,Cin]``.
    Cross-correlation (no flip), as the attention page's GEMM problem states
    for the same convolution machinery.
    """
    x = _f64(x)
    w = _f64(w)
    n, d, h, wd, cin = x.shape
    cout = w.shape[0]
    assert w.shape == (cout, cin, 3, 3, 3), w.shape
    xp = _pad_causal(x, history)
    y = np.zeros((n, d, h, wd, cout), dtype=np.float64)
    if b is not None:
        y += _f64(b)
    for kt in range(3):
        for kh in range(3):
            for kw in range(3):
                # the channel sum of one tap, as a matrix product
                y += xp[:, kt:kt + d, kh:kh + h, kw:kw + wd, :] @ w[:, :, kt, kh, kw].T
    return y


def causal_conv3d_at(x, w, b, points, history=None) -> np.ndarray:
    """The same convolution evaluated only at ``points`` (an int array [P,4]
    of (n, t, h, w)); returns [P, Cout]. Used where the full output is too
    large for the CPU."""
    x = np.asarray(x)  # gathered windows are widened to float64 below
    w = _f64(w)
    pts = np.asarray(points, dtype=np.int64).reshape(-1, 4)
    n, d, h, wd, cin = x.shape
    cout = w.shape[0]
    out = np.zeros((len(pts), cout), dtype=np.float64)
    if b is not None:
        out += _f64(b)
    hist = None if history is None else np.asarray(history)
    for kt in range(3):
        for kh in range(3):
            for kw in range(3):
                tt = pts[:, 1] + kt - 2
                hh = pts[:, 2] + kh - 1
                ww = pts[:, 3] + kw - 1
                inside = (hh >= 0) & (hh < h) & (ww >= 0) & (ww < wd)
                win = np.zeros((len(pts), cin), dtype=np.float64)
                cur = inside & (tt >= 0)
                win[cur] = x[pts[cur, 0], tt[cur], hh[cur], ww[cur], :]
                if hist is not None:
                    old = inside & (tt < 0)
                    win[old] = hist[pts[old, 0], tt[old] + 2, hh[old], ww[old], :]
                out += win @ w[:, :, kt, kh, kw].T
    return out


def nearest_up2(x, temporal=False) -> np.ndarray:
    """Nearest-neighbour x2 in space: u[n,t,y,x,c] = x[n,t,y//2,x//2,c]; with
    ``temporal`` also x2 in time: u[n,T,y,x,c] = x[n,T//2,y//2,x//2,c]."""
    x = _f64(x)
    u = np.repeat(np.repeat(x, 2, axis=2), 2, axis=3)
    return np.repeat(u, 2, axis=1) if temporal else u


def resample_up2(x, w, b, skip, history=None, temporal=False) -> np.ndarray:
    """Resampler, direct form: nearest x2 in space (and in time when
    ``temporal``, the resample.h variant of up_blocks 0 and 1), the causal
    3x3x3 convolution with bias, then the equally duplicated shortcut added.
    In the temporal variant the up-sampled history is the last history frame
    twice (nearest x2 of frames -2, -1 keeps only frame -1 next to frame 0)."""
    if history is None:
        hist_up = None
    elif temporal:
        hist_up = nearest_up2(np.asarray(history)[:, 1:2], temporal=True)
    else:
        hist_up = nearest_up2(history)
    return causal_conv3d(nearest_up2(x, temporal), w, b, hist_up) + nearest_up2(skip, temporal)


def resample_up2_at(x, w, b, skip, points, history=None, temporal=False) -> np.ndarray:
    """The direct resampler at high-resolution ``points`` [P,4] of
    (n, t, y, x); the up-sampled tensor is indexed, never materialised. With
    ``temporal`` the output frame T reads low-resolution frame T // 2."""
    x = np.asarray(x)  # gathered windows are widened to float64 below
    w = _f64(w)
    pts = np.asarray(points, dtype=np.int64).reshape(-1, 4)
    n, d, hl, wl, cin = x.shape
    hh_max, ww_max = 2 * hl, 2 * wl
    cout = w.shape[0]
    out = np.zeros((len(pts), cout), dtype=np.float64) + _f64(b)
    hist = None if history is None else np.asarray(history)
    for kt in range(3):
        for kh in range(3):
            for kw in range(3):
                tu = pts[:, 1] + kt - 2  # frame of the (time-)up-sampled input
                tt = np.floor_divide(tu, 2) if temporal else tu
                yy = pts[:, 2] + kh - 1
                xx = pts[:, 3] + kw - 1
                inside = (yy >= 0) & (yy < hh_max) & (xx >= 0) & (xx < ww_max)
                win = np.zeros((len(pts), cin), dtype=np.float64)
                cur = inside & (tt >= 0)
                win[cur] = x[pts[cur, 0], tt[cur], yy[cur] // 2, xx[cur] // 2, :]
                if hist is not None:
                    old = inside & (tt < 0)
                    win[old] = hist[pts[old, 0], tt[old] + 2, yy[old] // 2, xx[old] // 2, :]
                out += win @ w[:, :, kt, kh, kw].T
    s = np.asarray(skip)
    ts = pts[:, 1] // 2 if temporal else pts[:, 1]
    out += s[pts[:, 0], ts, pts[:, 2] // 2, pts[:, 3] // 2, :].astype(np.float64)
    return out


# Rows of the 3x3 kernel that land on low-resolution row i + p - 1 + a, for
# output parity p and phase tap a (nearest x2 maps rows 2i+p-1..2i+p+1 onto
# low-resolution rows i-1, i, i+1).
_PHASE_ROWS = {(0, 0): (0,), (0, 1): (1, 2), (1, 0): (0, 1), (1, 1): (2,)}


def resample_phase_kernels(w) -> np.ndarray:
    """The four per-phase 3x2x2 kernels with repeated taps summed.

    Returns pk[2p+q, co, ci, kt, a, b] (fp64). The decomposition the
    resample.h header describes: nearest x2 then 3x3x3 equals one low-resolution
    conv per output parity (p, q) whose taps are sums of the original taps.
    """
    w = _f64(w)
    cout, cin = w.shape[:2]
    pk = np.zeros((4, cout, cin, 3, 2, 2), dtype=np.float64)
    for p in range(2):
        for q in range(2):
            for a in range(2):
                for bb in range(2):
                    for kh in _PHASE_ROWS[(p, a)]:
                        for kw in _PHASE_ROWS[(q, bb)]:
                            pk[2 * p + q, :, :, :, a, bb] += w[:, :, :, kh, kw]
    return pk


def resample_phase_conv(x, pk, history=None) -> np.ndarray:
    """The four low-resolution phase convolutions (no bias): phase 2p+q at
    (t, i, j) is sum_{ci,kt,a,b} pk[2p+q, co, ci, kt, a, b]
    * x~[t+kt-2, i+p-1+a, j+q-1+b, ci]. Returns [4, N, D, HL, WL, Cout]."""
    x = _f64(x)
    pk = _f64(pk)
    n, d, hl, wl, cin = x.shape
    cout = pk.shape[1]
    xp = _pad_causal(x, history)  # index offset: frame +2, row +1, column +1
    ph = np.zeros((4, n, d, hl, wl, cout), dtype=np.float64)
    for p in range(2):
        for q in range(2):
            for kt in range(3):
                for a in range(2):
                    for bb in range(2):
                        r0 = p + a  # = (i + p - 1 + a) + 1 - i
                        c0 = q + bb
                        ph[2 * p + q] += xp[:, kt:kt + d, r0:r0 + hl, c0:c0 + wl, :] @ pk[2 * p + q, :, :, kt, a, bb].T
    return ph


def resample_interleave(phases, b, skip) -> np.ndarray:
    """out[n, t, 2i+p, 2j+q, c] = phases[2p+q][n, t, i, j, c] + b[c] + skip[n, t, i, j, c]."""
    ph = _f64(phases)
    _, n, d, hl, wl, c = ph.shape
    out = np.zeros((n, d, 2 * hl, 2 * wl, c), dtype=np.float64)
    for p in range(2):
        for q in range(2):
            out[:, :, p::2, q::2, :] = ph[2 * p + q] + _f64(b) + _f64(skip)
    return out


# Taps kt of up-sampled output frame 2t+s that land on low-resolution frame
# t-1+a (causal: tap kt reads up-sampled frame 2t+s+kt-2).
_PHASE_FRAMES = {(0, 0): (0, 1), (0, 1): (2,), (1, 0): (0,), (1, 1): (1, 2)}


def resample_phase_kernels_temporal(w) -> np.ndarray:
    """Eight per-phase 2x2x2 kernels of the temporal variant: output frame
    2t+s, row 2i+p, column 2j+q; phase tap (a, bb, cc) reads low-resolution
    frame t-1+a, row i+p-1+bb, column j+q-1+cc. Causal tap kt of up-sampled
    frame 2t+s reads up-sampled frame 2t+s+kt-2, i.e. low-resolution frames
    t-1, t-1, t (s=0) or t-1, t, t (s=1): the grouping of rows with the parity
    flipped. Returns pk[4s+2p+q, co, ci, a, bb, cc]."""
    w = _f64(w)
    cout, cin = w.shape[:2]
    pk = np.zeros((8, cout, cin, 2, 2, 2), dtype=np.float64)
    for s_ in range(2):
        for p in range(2):
            for q in range(2):
                for a in range(2):
                    for bb in range(2):
                        for cc in range(2):
                            for kt in _PHASE_FRAMES[(s_, a)]:
                                for kh in _PHASE_ROWS[(p, bb)]:
                                    for kw in _PHASE_ROWS[(q, cc)]:
                                        pk[4 * s_ + 2 * p + q, :, :, a, bb, cc] += w[:, :, kt, kh, kw]
    return pk


def resample_up2_temporal_eight_phase(x, w, b, skip, history=None) -> np.ndarray:
    """The temporal resampler through its eight-phase form, kept to check the
    decomposition against the direct form (nearest x2 in time and space, then
    the conv)."""
    x = _f64(x)
    n, d, hl, wl, cin = x.shape
    pk = resample_phase_kernels_temporal(w)
    cout = pk.shape[1]
    xp = _pad_causal(x, history)  # frame t of x at index t + 2
    out = np.zeros((n, 2 * d, 2 * hl, 2 * wl, cout), dtype=np.float64)
    sk = _f64(skip)
    for s_ in range(2):
        for p in range(2):
            for q in range(2):
                ph = np.zeros((n, d, hl, wl, cout), dtype=np.float64)
                for a in range(2):
                    for bb in range(2):
                        for cc in range(2):
                            t0, r0, c0 = 1 + a, p + bb, q + cc  # frame t-1+a sits at index t+1+a
                            ph += xp[:, t0:t0 + d, r0:r0 + hl, c0:c0 + wl, :] @ pk[4 * s_ + 2 * p + q, :, :, a, bb, cc].T
                out[:, s_::2, p::2, q::2, :] = ph + _f64(b) + sk
    return out


def resample_up2_four_phase(x, w, b, skip, history=None) -> np.ndarray:
    """The resampler through the four-phase form (pre-summed kernels, four
    low-resolution convolutions, interleave with bias and shortcut), kept to
    check the decomposition against the direct form."""
    return resample_interleave(resample_phase_conv(x, resample_phase_kernels(w), history), b, skip)


def attn_probs(q, k, scale=None) -> np.ndarray:
    """P = softmax over keys of (q k^T) * scale, per frame; q,k [T,HW,C].
    The maximum is subtracted before the exponential (attn.cu, stage 3)."""
    q = _f64(q)
    k = _f64(k)
    if scale is None:
        scale = 1.0 / np.sqrt(q.shape[-1])
    s = np.einsum("tic,tjc->tij", q, k) * scale
    s -= s.max(axis=-1, keepdims=True)
    e = np.exp(s)
    return e / e.sum(axis=-1, keepdims=True)


def attn_frame(q, k, v, scale=None) -> np.ndarray:
    """Single-head attention per latent frame, no mask: O = softmax(q k^T *
    scale) v with scale = 1/sqrt(C) by default. q, k, v [T, HW, C]."""
    p = attn_probs(q, k, scale)
    return np.einsum("tij,tjc->tic", p, _f64(v))


def attn_frame_rows(q, k, v, rows, scale=None) -> np.ndarray:
    """Attention output for the query rows ``rows`` [P,2] of (frame, i)."""
    q, k, v = np.asarray(q), np.asarray(k), np.asarray(v)  # widened per frame below
    rows = np.asarray(rows, dtype=np.int64).reshape(-1, 2)
    if scale is None:
        scale = 1.0 / np.sqrt(q.shape[-1])
    out = np.zeros((len(rows), v.shape[-1]), dtype=np.float64)
    for t in np.unique(rows[:, 0]):
        kt, vt = _f64(k[t]), _f64(v[t])
        sel = np.nonzero(rows[:, 0] == t)[0]
        s = (_f64(q[t, rows[sel, 1]]) @ kt.T) * scale
        e = np.exp(s - s.max(axis=1, keepdims=True))
        out[sel] = (e / e.sum(axis=1, keepdims=True)) @ vt
    return out


def head_out(x, w, b, history=None) -> np.ndarray:
    """Output head: causal conv_out (3x3x3, C_in -> 12), bias, clamp to [-1, 1]."""
    return np.clip(causal_conv3d(x, w, b, history), -1.0, 1.0)


def head_out_at(x, w, b, points, history=None) -> np.ndarray:
    """The head at ``points`` [P,4] of (n, t, h, w)."""
    return np.clip(causal_conv3d_at(x, w, b, points, history), -1.0, 1.0)


def head_stage_a(x, w, history=None) -> np.ndarray:
    """Stage A of the regrouped head: a temporal-only (3x1x1) conv whose output
    channel (i*3+j)*Cout + c holds spatial tap (i, j) of channel c:
    g[n,t,h,w,(i*3+j)*Cout+c] = sum_{ci,kt} w[c,ci,kt,i,j] x~[n, t+kt-2, h, w, ci]."""
    x = _f64(x)
    w = _f64(w)
    n, d, h, wd, cin = x.shape
    cout = w.shape[0]
    xp = np.zeros((n, d + 2, h, wd, cin), dtype=np.float64)
    xp[:, 2:] = x
    if history is not None:
        xp[:, :2] = _f64(history)
    g = np.zeros((n, d, h, wd, 9 * cout), dtype=np.float64)
    for i in range(3):
        for j in range(3):
            for kt in range(3):
                g[..., (i * 3 + j) * cout:(i * 3 + j + 1) * cout] += xp[:, kt:kt + d] @ w[:, :, kt, i, j].T
    return g


def head_stage_b(g, b) -> np.ndarray:
    """Stage B: out[n,t,h,w,c] = clamp(b[c] + sum_{i,j} g[n,t,h+i-1,w+j-1,(i*3+j)*Cout+c],
    -1, 1), zero outside the plane."""
    g = _f64(g)
    b = _f64(b)
    cout = b.shape[0]
    n, d, h, wd, _ = g.shape
    gp = np.zeros((n, d, h + 2, wd + 2, 9 * cout), dtype=np.float64)
    gp[:, :, 1:-1, 1:-1] = g[..., :9 * cout]
    y = np.zeros((n, d, h, wd, cout), dtype=np.float64) + b
    for i in range(3):
        for j in range(3):
            y += gp[:, :, i:i + h, j:j + wd, (i * 3 + j) * cout:(i * 3 + j + 1) * cout]
    return np.clip(y, -1.0, 1.0)


def head_two_stage(x, w, b, history=None) -> np.ndarray:
    """The head regrouped as on the head.cu page (stage A then stage B), kept
    to check that the regrouping is the same sum as the direct conv."""
    return head_stage_b(head_stage_a(x, w, history), b)
