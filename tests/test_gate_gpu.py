"""The log-decay gate mode (theta holds g itself) against the oracle, and the
unbounded -softplus control: with g = -softplus(theta) the in-chunk factor
e^{-G} overflows once the logits are large, so the dense tile products stop
being finite, while the bounded gate g_min * sigmoid(theta) on the very same
logits never leaves e^{80} ("Architecture Deep Dive", sec. 3.2; "Kimi K3 Deep
Dive", section "The Design").  The register-resident path detects such chunks
and forms their tiles position by position (per-pair e^{G_r - G_s}), so its
results stay finite and within the bar; the tcgen05 path has no such
fallback and is the control."""
import numpy as np
import pytest
import torch

from linear_attention_04_gb300 import kda_chunk_fwd, kda_device_status
from linear_attention_04_gb300.workloads import Workload, make_inputs

from parity import TOL, assert_close, f64
import oracle

pytestmark = pytest.mark.gpu


def _case(dtype, mu, seed, T=400, H=3):
    w = Workload("gate", B=2, H=H, T=T, dk=128, dv=128, dtype=dtype)
    inp = make_inputs(w, seed=seed)
    logits = inp["theta"].float() + mu
    g = -torch.nn.functional.softplus(logits)
    return inp, logits.to(dtype), g.to(dtype)


def _run(inp, theta, path, gate):
    c = {k_: (x.cuda() if isinstance(x, torch.Tensor) else x) for k_, x in inp.items()}
    o, S = kda_chunk_fwd(c["q"], c["k"], c["v"], theta.cuda(), c["beta"], -5.0, path=path,
                         gate=gate)
    torch.cuda.synchronize()
    assert kda_device_status(clear=True) == 0
    return o, S


@pytest.mark.parametrize("dtype,path", [(torch.float32, "simt"), (torch.bfloat16, "simt"),
                                        (torch.bfloat16, "mma"), (torch.bfloat16, "mma_tc"),
                                        (torch.bfloat16, "tc"), (torch.bfloat16, "tc_split")])
def test_log_decay_gate_vs_oracle(dtype, path):
    # logits ~ N(2, 1): |g| ~ 2.2 per token, the decay rate of the named
    # workloads (the bf16 operand plan's error grows past the 2e-2 bar once the
    # in-chunk decay is much slower, for either gate)
    inp, _, g = _case(dtype, mu=2.0, seed=31)
    ro, rS = oracle.fwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(g), f64(inp["beta"]),
                        -5.0, None, theta_is_g=True)
    o, S = _run(inp, g, path, "log_decay")
    tol = TOL[torch.float32] if path == "simt" else TOL[dtype]
    assert_close(f64(o), ro, tol, f"log-decay gate out ({path}, {dtype})")
    assert_close(f64(S), rS, tol, f"log-decay gate state ({path}, {dtype})")


@pytest.mark.parametrize("path", ["mma", "mma_tc", "tc"])
def test_unbounded_softplus_control(path):
    # logits ~ N(8, 1): every 16-token chunk reaches -G ~ 128 > 88.7 with the
    # -softplus gate; the bounded gate on the same logits stays below 80
    inp, logits, g = _case(torch.bfloat16, mu=8.0, seed=32)
    G = -g.double().reshape(2, -1, 16, 3, 128).sum(dim=2)          # -G_16 per chunk
    assert float(G.max()) > 88.72
    gs = -5.0 * torch.sigmoid(logits.double())
    assert float((-gs.reshape(2, -1, 16, 3, 128).sum(dim=2)).max()) <= 80.0
    # the fp64 oracle is finite either way
    ro, rS = oracle.fwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(g), f64(inp["beta"]),
                        -5.0, None, theta_is_g=True)
    assert np.all(np.isfinite(ro))
    o, S = _run(inp, g, path, "log_decay")
    if path == "tc":
        # the dense tile path with the unbounded gate: not finite
        assert not bool(torch.isfinite(o).all())
    else:
        # every chunk takes the position-wise fallback: finite and within the bar
        assert_close(f64(o), ro, TOL[torch.bfloat16], "position-wise fallback out")
        assert_close(f64(S), rS, TOL[torch.bfloat16], "position-wise fallback state")
    # the same logits through the bounded gate: finite and within the bar
    rb, rSb = oracle.fwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(logits),
                         f64(inp["beta"]), -5.0, None)
    ob, Sb = _run(inp, logits, path, "sigmoid")
    assert_close(f64(ob), rb, TOL[torch.bfloat16], "bounded gate, same logits")


@pytest.mark.parametrize("path", ["mma", "mma_tc"])
def test_fallback_on_some_chunks_only(path):
    """logits ~ N(4.75, 1): some 16-token chunks (about a fifth) pass the dense tile's limit
    (-G = 126 / log2 e = 87.3 on any channel) and some do not, so the
    register-resident path mixes dense and position-wise chunks in one chain."""
    inp, _, g = _case(torch.bfloat16, mu=4.75, seed=33, T=640)
    G = (-g.double()).reshape(2, -1, 16, 3, 128).sum(dim=2).amax(dim=-1)  # per chunk and head
    share = float((G > 126.0 / 1.4426950408889634).double().mean())
    assert 0.05 < share < 0.99
    ro, rS = oracle.fwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(g), f64(inp["beta"]),
                        -5.0, None, theta_is_g=True)
    o, S = _run(inp, g, path, "log_decay")
    assert_close(f64(o), ro, TOL[torch.bfloat16], "mixed fallback out")
    assert_close(f64(S), rS, TOL[torch.bfloat16], "mixed fallback state")
