"""The oracle against its stored regression fixtures (tests/golden/tiny_cases.json,
written by tests/golden/make_golden.py from the oracle alone)."""

import json
import os

import numpy as np

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def load():
    with open(os.path.join(HERE, "golden", "tiny_cases.json")) as f:
        return {k: {kk: np.array(vv) for kk, vv in v.items()} for k, v in json.load(f).items()}


def test_golden_tiny_cases():
    fx = load()
    c = fx["conv"]
    np.testing.assert_allclose(oracle.causal_conv3d(c["x"], c["w"], c["b"]), c["y"], rtol=0, atol=1e-12)
    r = fx["resample"]
    np.testing.assert_allclose(oracle.resample_up2(r["x"], r["w"], r["b"], r["skip"]), r["y"], rtol=0, atol=1e-12)
    a = fx["attn"]
    np.testing.assert_allclose(oracle.attn_frame(a["q"], a["k"], a["v"]), a["o"], rtol=0, atol=1e-12)
    h = fx["head"]
    np.testing.assert_allclose(oracle.head_out(h["x"], h["w"], h["b"]), h["y"], rtol=0, atol=1e-12)


def test_golden_inputs_are_exact_in_bf16():
    import torch
    fx = load()
    for case in fx.values():
        for name, arr in case.items():
            if name in ("y", "o"):
                continue
            t = torch.from_numpy(arr)
            assert torch.equal(t.to(torch.bfloat16).double(), t), name
