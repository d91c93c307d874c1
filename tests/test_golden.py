"""Stored values: the pages' constants and a frozen tiny oracle case."""
import math
import os
import sys

import numpy as np
import torch

import oracle

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
sys.path.insert(0, HERE)
import make_golden  # noqa: E402


def _constants():
    out = {}
    with open(os.path.join(HERE, "pages_constants.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                name, val = line.split()
                out[name] = float(val)
    return out


def test_pages_constants():
    c = _constants()
    assert c["g_min"] == -5.0 and c["chunk"] == 16
    assert c["tile_inverse_log_bound"] == -c["g_min"] * c["chunk"]
    # the largest bf16 is what torch says it is
    assert c["bf16_max"] == float(torch.finfo(torch.bfloat16).max)
    # e^{80} is finite in bf16 and below its maximum
    assert math.exp(c["tile_inverse_log_bound"]) < c["bf16_max"]
    # the oracle's gate stays inside [g_min, 0]
    g = oracle.gate(np.linspace(-50, 50, 1001), c["g_min"])
    assert g.min() >= c["g_min"] and g.max() <= 0.0


def test_tiny_case_frozen():
    rows = {}
    with open(os.path.join(HERE, "tiny_case.txt")) as f:
        for line in f:
            if line.startswith("#"):
                continue
            tag, idx, a, b = line.split()
            rows[(tag, int(idx))] = (float(a), float(b))
    q, k, v, th, be, S0 = make_golden.case()
    o, S = oracle.fwd(q, k, v, th, be, -5.0, S0, nthreads=1)
    for t in range(8):
        assert np.allclose(o[0, t, 0], rows[("o", t)], rtol=0, atol=1e-14)
    for i in range(2):
        assert np.allclose(S[0, 0, i], rows[("S", i)], rtol=0, atol=1e-14)
