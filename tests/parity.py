"""Helpers shared by the GPU parity tests: run the CUDA path and the fp64
oracle on the very same input values and compare them."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle

# Tolerances on max |o - o_ref| relative to RMS(o_ref): 1e-4 for fp32
# inputs, 2e-2 for bf16 inputs with fp32 state.  The same rule is applied
# to the final state.
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def f64(t: torch.Tensor | None):
    if t is None:
        return None
    return t.detach().to("cpu", torch.float64).numpy()


def rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    rms = math.sqrt(float(np.mean(ref * ref)))
    return float(np.max(np.abs(got - ref))) / max(rms, 1e-30)


def assert_close(got, ref, tol, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    e = rel_err(got, ref)
    assert e <= tol, f"{what}: max|err|/rms = {e:.3e} > {tol:.1e}"
    return e


def oracle_full(inp: dict, g_min=-5.0, nthreads=None):
    """Oracle over every chain of a (CPU or GPU) input dict."""
    return oracle.fwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["theta"]),
                      f64(inp["beta"]), g_min, f64(inp["init_state"]),
                      None if inp["cu_seqlens"] is None else
                      inp["cu_seqlens"].cpu().numpy(), nthreads=nthreads)


def oracle_chain(inp: dict, seq: int, head: int, g_min=-5.0):
    """Oracle for one (sequence, head) pair of an input dict, copying only that
    chain to the host.  Returns (o [L, dv], S [dk, dv]) and the token range."""
    if inp["cu_seqlens"] is None:
        b, t0, t1 = seq, 0, inp["T"]
    else:
        cu = inp["cu_seqlens"].cpu().tolist()
        b, t0, t1 = 0, cu[seq], cu[seq + 1]

    def pick(x):
        return f64(x[b:b + 1, t0:t1, head:head + 1])

    init = inp["init_state"]
    S0 = None if init is None else f64(init[seq:seq + 1, head:head + 1])
    o, S = oracle.fwd(pick(inp["q"]), pick(inp["k"]), pick(inp["v"]), pick(inp["theta"]),
                      pick(inp["beta"]), g_min, S0, nthreads=1)
    return o[0, :, 0], S[0, 0], (b, t0, t1)
