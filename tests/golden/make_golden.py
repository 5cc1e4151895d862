"""Writes the regression fixtures in this folder from the fp64 oracle alone.

Run from the repository root:  python tests/golden/make_golden.py

Inputs are small integer multiples of 1/8 drawn from a fixed numpy seed, so
every value is exact in bf16 and the fixtures can be fed to any
implementation; the outputs are the oracle's float64 results. The pages print
no worked example, so these fixtures guard the oracle against silent changes
(its pins against brute force and library routines live in the tests).
"""

import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402


def eighths(rng, *shape, lo=-8, hi=8):
    return rng.integers(lo, hi + 1, size=shape).astype(np.float64) / 8.0


def main():
    rng = np.random.default_rng(2024)
    fx = {}
    x = eighths(rng, 1, 2, 3, 4, 2)
    w = eighths(rng, 3, 2, 3, 3, 3, lo=-4, hi=4)
    b = eighths(rng, 3)
    fx["conv"] = {"x": x.tolist(), "w": w.tolist(), "b": b.tolist(), "y": oracle.causal_conv3d(x, w, b).tolist()}
    x = eighths(rng, 1, 2, 2, 3, 2)
    s = eighths(rng, 1, 2, 2, 3, 2)
    w = eighths(rng, 2, 2, 3, 3, 3, lo=-4, hi=4)
    b = eighths(rng, 2)
    fx["resample"] = {"x": x.tolist(), "skip": s.tolist(), "w": w.tolist(), "b": b.tolist(),
                      "y": oracle.resample_up2(x, w, b, s).tolist()}
    q, k, v = eighths(rng, 1, 5, 4), eighths(rng, 1, 5, 4), eighths(rng, 1, 5, 4)
    fx["attn"] = {"q": q.tolist(), "k": k.tolist(), "v": v.tolist(), "o": oracle.attn_frame(q, k, v).tolist()}
    x = eighths(rng, 1, 2, 3, 3, 4)
    w = eighths(rng, 12, 4, 3, 3, 3, lo=-2, hi=2)
    b = eighths(rng, 12)
    fx["head"] = {"x": x.tolist(), "w": w.tolist(), "b": b.tolist(), "y": oracle.head_out(x, w, b).tolist()}
    with open(os.path.join(HERE, "tiny_cases.json"), "w") as f:
        json.dump(fx, f, indent=None, separators=(",", ":"))
        f.write("\n")


if __name__ == "__main__":
    main()
