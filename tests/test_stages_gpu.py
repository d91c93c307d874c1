"""GPU stage tests: the intermediate tiles of the tcgen05 path (through the
``kda_debug_fwd_stages`` test hook) against the fp64 chunk-parallel
restatement ``oracle.chunked.chunk_stages`` over the same 32-token units.

The kernel steps the state once per 32 tokens (two of the pages' 16-token
chunks, with the decay factors anchored at the boundary between them), so the
reference for each unit is ``chunk_stages`` over those 32 tokens, started from
the oracle's state at the unit's start.  Checked per stage, each at a
tolerance derived from the arithmetic that produces it:

  A, P, T   tf32 Gram operands (rounded to nearest: 2^-11 relative each, so
            at most ~1e-3 relative per product term) and fp32 arithmetic; an
            entry sums 128 such terms whose absolute sum is a few times the
            RMS entry: max |err| <= 1e-2 x RMS of the reference tile
  W         Tb and Kt as bf16 operands (2^-9 relative each) with fp32
            accumulation: |err| <= 2^-8 x sum_s |Tb_ts| |Kt_sc| per entry
            from the roundings, plus T's own error; W is heavy-tailed (the
            first rows carry e^{G} ~ 1, the last ~ e^{-80}), so the bar is
            2^-7 x max over entries of (|Tb| |Kt|)
  U         max |err| <= 2e-2 x RMS
  e^{G}     fp32 gate and cumulative sum: |err| <= 1e-3 x e^{G} (relative)
  q.k       fp32 from the bf16 inputs: max |err| <= 1e-5 x RMS

The decay-stress regime (theta ~ U[6, 12], every g close to g_min = -5)
puts the factors of the unit's first and last tokens at about e^{+-80}, the
bound of "Kimi K3 Deep Dive", section "The Design"."""
import numpy as np
import pytest
import torch

from linear_attention_04_gb300 import kda as binding
from linear_attention_04_gb300.workloads import Workload, make_inputs
from oracle import chunked

from parity import f64, rel_err

pytestmark = pytest.mark.gpu

UNIT = 32
TOLS = {"A": 1e-2, "P": 1e-2, "T": 1e-2, "U": 2e-2, "qk": 1e-5}


def _reference_units(inp, nunits, g_min=-5.0):
    """chunk_stages of chain (0, 0) for its first `nunits` 32-token units."""
    q, k, v, th, be = (f64(inp[n][0, :, 0]) for n in ("q", "k", "v", "theta", "beta"))
    g = chunked.gate(th, g_min)
    S = np.zeros((128, 128)) if inp["init_state"] is None else f64(inp["init_state"][0, 0])
    L = q.shape[0]
    units = []
    for u in range(nunits):
        t0, t1 = u * UNIT, min(L, (u + 1) * UNIT)
        st = chunked.chunk_stages(q[t0:t1], k[t0:t1], v[t0:t1], g[t0:t1], be[t0:t1], S)
        st["n"] = t1 - t0
        st["b"] = be[t0:t1]
        st["qk"] = np.sum(q[t0:t1] * k[t0:t1], axis=1)
        units.append(st)
        S = st["S"]
    return units


def _compare(stages, units):
    worst = {}
    for u, st in enumerate(units):
        n = st["n"]
        got = {name: stages[name][u].double().numpy() for name in stages}
        refs = {"A": st["A"], "P": np.tril(st["P"], -1), "T": st["T"], "U": st["U"],
                "qk": st["qk"]}
        Tb = st["T"] * st["b"][None, :]
        bound = 2.0 ** -7 * float(np.max(np.abs(Tb) @ np.abs(st["Kt"])))
        ew = float(np.max(np.abs(got["W"][:n] - st["W"])))
        worst["W"] = max(worst.get("W", 0.0), ew / bound)
        assert ew <= bound, f"unit {u} W: max|err| = {ew:.3e} > 2^-7 max(|Tb||Kt|) = {bound:.3e}"
        for name, ref in refs.items():
            g_ = got[name][:n, :n] if name in ("A", "P", "T") else got[name][:n]
            assert np.all(np.isfinite(g_)), f"unit {u} {name}: non-finite"
            e = rel_err(g_, ref)
            worst[name] = max(worst.get(name, 0.0), e)
            assert e <= TOLS[name], f"unit {u} {name}: max|err|/rms = {e:.3e} > {TOLS[name]:.0e}"
        eg_ref = np.exp(st["G"][-1])
        eg = got["eG"]
        erel = np.max(np.abs(eg - eg_ref) / np.maximum(eg_ref, 1e-30))
        worst["eG"] = max(worst.get("eG", 0.0), erel)
        assert erel <= 1e-3, f"unit {u} e^G: relative error {erel:.3e}"
        # rows and columns past the end of a ragged last unit are exactly zero
        if n < UNIT:
            for name in ("A", "P"):
                assert not np.any(got[name][n:, :]) and not np.any(got[name][:, n:]), name
            assert not np.any(got["W"][n:]) and not np.any(got["U"][n:])
    return worst


@pytest.mark.parametrize("regime,T,init_std", [
    ("normal", 96, 0.0),       # theta ~ N(0,1): the train/base/long recipe
    ("fast", 96, 0.02),        # theta ~ U[6,12]: factors at the e^{+-80} bound
    ("slow", 96, 0.02),        # theta ~ N(-3,1): slow decay, the state carries over
    ("normal", 80, 0.02),      # ragged last unit (16 valid tokens)
    ("fast", 45, 0.0),         # ragged inside the first chunk of the second unit
])
@pytest.mark.parametrize("path", ["tc", "tc_split"])
def test_stages_against_chunk_stages(regime, T, init_std, path):
    theta = "uniform6_12" if regime == "fast" else "normal"
    beta = "uniform09_1" if regime == "fast" else "sigmoid_normal"
    w = Workload("stages", B=1, H=2, T=T, dk=128, dv=128, dtype=torch.bfloat16, theta=theta,
                 beta=beta, init_std=init_std)
    inp = make_inputs(w, seed=31 + T)
    if regime == "slow":
        inp["theta"] = (inp["theta"].float() - 3.0).to(torch.bfloat16)
    nunits = (T + UNIT - 1) // UNIT
    g = {k_: (x.cuda() if isinstance(x, torch.Tensor) else x) for k_, x in inp.items()}
    _, _, stages = binding.kda_debug_fwd_stages(g["q"], g["k"], g["v"], g["theta"], g["beta"], -5.0,
                                                g["init_state"], nsc=nunits, path=path)
    torch.cuda.synchronize()
    assert binding.kda_device_status(clear=True) == 0
    _compare(stages, _reference_units(inp, nunits))
