"""Shared helpers of the GPU tests: building/loading the library, the parity
bar, and conversions between torch bf16 tensors and the oracle's numpy."""

import os

import numpy as np
import torch

# Parity bar per output tensor: relative L2 error and max |difference|
# relative to the reference's max |value|.
REL_L2 = 4e-3
MAX_ABS_FRAC = 2.0 ** -6


def ensure_built():
    from causal_convolution_gb300 import _lib, build
    if not os.path.exists(_lib.LIB_PATH):
        build.build()
    return _lib.load()


def to_np(t: torch.Tensor) -> np.ndarray:
    """bf16/fp32 torch tensor (any device) -> float32 numpy (exact for bf16)."""
    return t.detach().float().cpu().numpy()


def parity(got, ref) -> dict:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    d = got - ref
    nref = np.linalg.norm(ref)
    return {
        "rel_l2": float(np.linalg.norm(d) / nref) if nref > 0 else float(np.linalg.norm(d)),
        "max_abs": float(np.abs(d).max()) if d.size else 0.0,
        "max_ref": float(np.abs(ref).max()) if ref.size else 0.0,
    }


def assert_parity(got, ref, what: str, rel_l2: float = REL_L2, max_frac: float = MAX_ABS_FRAC) -> dict:
    p = parity(got, ref)
    assert np.all(np.isfinite(np.asarray(got, dtype=np.float64))), f"{what}: non-finite output"
    assert p["rel_l2"] <= rel_l2, f"{what}: rel-L2 {p['rel_l2']:.3e} > {rel_l2:.1e} ({p})"
    assert p["max_abs"] <= max_frac * p["max_ref"] + 1e-30, f"{what}: max|d| {p['max_abs']:.3e} > bar ({p})"
    return p


def edge_points(n, d, h, w, extra, rng, m_tile=128):
    """(n, t, h, w) points: every corner and edge midpoint of every frame, the
    positions on both sides of each 128-row tile boundary near the start and
    end of the flattened grid, and `extra` random positions."""
    pts = set()
    for nn in range(n):
        for t in range(d):
            for hh in (0, h // 2, h - 1):
                for ww in (0, w // 2, w - 1):
                    pts.add((nn, t, hh, ww))
    total = n * d * h * w
    for base in list(range(m_tile, min(total, 4 * m_tile), m_tile)) + [total - total % m_tile]:
        for m in (base - 1, base):
            if 0 <= m < total:
                ww = m % w
                hh = (m // w) % h
                t = (m // (w * h)) % d
                nn = m // (w * h * d)
                pts.add((nn, t, hh, ww))
    for _ in range(extra):
        pts.add((int(rng.integers(n)), int(rng.integers(d)), int(rng.integers(h)), int(rng.integers(w))))
    return np.array(sorted(pts), dtype=np.int64)
