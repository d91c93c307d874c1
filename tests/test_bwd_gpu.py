"""GPU parity of the backward pass (kda_chunk_bwd) against the fp64 backward
oracle (reverse-mode differentiation of the token recurrence, pinned by finite
differences): element-wise on every gradient."""
import numpy as np
import pytest
import torch

from linear_attention_04_gb300 import kda_chunk_bwd, kda_device_status
from linear_attention_04_gb300.workloads import Workload, make_inputs

from parity import assert_close, f64
from oracle import backward

pytestmark = pytest.mark.gpu

# fp32 arithmetic throughout (the inputs' own rounding is not part of the error)
TOL_BWD = 1e-4


def _case(dtype, T, H=2, B=1, seed=0, init=0.05):
    w = Workload("bwd", B=B, H=H, T=T, dk=128, dv=128, dtype=dtype, init_std=init)
    inp = make_inputs(w, seed=seed)
    g = torch.Generator().manual_seed(seed + 1)
    d_out = torch.randn(B, T, H, 128, generator=g)
    d_fin = torch.randn(B, H, 128, 128, generator=g)
    return inp, d_out, d_fin


# 1, 2, 3, 5 and 9 chunks: the recurrences hand two operand buffers between
# their warp groups, so the first chunks and the last two take the edge paths
@pytest.mark.parametrize("dtype,T", [(torch.float32, 16), (torch.bfloat16, 32), (torch.float32, 40),
                                     (torch.bfloat16, 70), (torch.bfloat16, 130)])
def test_bwd_vs_oracle(dtype, T):
    inp, d_out, d_fin = _case(dtype, T, seed=T)
    ref = backward.bwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["theta"]),
                       f64(inp["beta"]), -5.0, f64(inp["init_state"]), d_out.double().numpy(),
                       d_fin.double().numpy())
    c = lambda x: None if x is None else x.cuda()
    got = kda_chunk_bwd(c(inp["q"]), c(inp["k"]), c(inp["v"]), c(inp["theta"]), c(inp["beta"]),
                        c(d_out), -5.0, c(inp["init_state"]), c(d_fin))
    torch.cuda.synchronize()
    assert kda_device_status(clear=True) == 0
    for name, key in (("dq", "dq"), ("dk", "dk"), ("dv", "dv"), ("dtheta", "dtheta"),
                      ("dbeta", "dbeta"), ("d_init", "dS0")):
        assert_close(f64(got[name]), ref[key], TOL_BWD, f"{name} T={T} {dtype}")


def test_bwd_log_decay_gate_and_no_state_gradients():
    inp, d_out, _ = _case(torch.bfloat16, 50, seed=7, init=0.0)
    gl = -torch.nn.functional.softplus(inp["theta"].float() + 0.5).to(torch.bfloat16)
    ref = backward.bwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(gl), f64(inp["beta"]),
                       -5.0, None, d_out.double().numpy(), None, theta_is_g=True)
    got = kda_chunk_bwd(inp["q"].cuda(), inp["k"].cuda(), inp["v"].cuda(), gl.cuda(),
                        inp["beta"].cuda(), d_out.cuda(), -5.0, gate="log_decay")
    torch.cuda.synchronize()
    for name, key in (("dq", "dq"), ("dk", "dk"), ("dv", "dv"), ("dtheta", "dtheta"),
                      ("dbeta", "dbeta"), ("d_init", "dS0")):
        assert_close(f64(got[name]), ref[key], TOL_BWD, f"{name} (log-decay gate)")


def test_bwd_fast_decay_multi_chain():
    """theta ~ U[6, 12] (every log-decay near g_min, sigmoid(theta) near 1),
    beta ~ U[0.9, 1], B = 2, H = 3, T = 48 (three whole chunks): chain
    indexing of every launch and the gate derivative where 1 - sigmoid is
    small."""
    B, H, T = 2, 3, 48
    w = Workload("bwd_fast", B=B, H=H, T=T, dk=128, dv=128, dtype=torch.bfloat16,
                 theta="uniform6_12", beta="uniform09_1", init_std=0.05)
    inp = make_inputs(w, seed=5)
    g = torch.Generator().manual_seed(6)
    d_out = torch.randn(B, T, H, 128, generator=g)
    d_fin = torch.randn(B, H, 128, 128, generator=g)
    ref = backward.bwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["theta"]),
                       f64(inp["beta"]), -5.0, f64(inp["init_state"]), d_out.double().numpy(),
                       d_fin.double().numpy())
    c = lambda x: x.cuda()
    got = kda_chunk_bwd(c(inp["q"]), c(inp["k"]), c(inp["v"]), c(inp["theta"]), c(inp["beta"]),
                        c(d_out), -5.0, c(inp["init_state"]), c(d_fin))
    torch.cuda.synchronize()
    assert kda_device_status(clear=True) == 0
    for name, key in (("dq", "dq"), ("dk", "dk"), ("dv", "dv"), ("dtheta", "dtheta"),
                      ("dbeta", "dbeta"), ("d_init", "dS0")):
        assert_close(f64(got[name]), ref[key], TOL_BWD, f"{name} fast decay")


def test_bwd_long_sequence():
    """T = 1000 (62 whole chunks and a ragged 8-token tail), two heads, an
    initial state and a final-state gradient: the two recurrences over many
    chunks and the staged next-chunk inputs at every step."""
    inp, d_out, d_fin = _case(torch.bfloat16, 1000, H=2, seed=21, init=0.02)
    ref = backward.bwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["theta"]),
                       f64(inp["beta"]), -5.0, f64(inp["init_state"]), d_out.double().numpy(),
                       d_fin.double().numpy())
    c = lambda x: x.cuda()
    got = kda_chunk_bwd(c(inp["q"]), c(inp["k"]), c(inp["v"]), c(inp["theta"]), c(inp["beta"]),
                        c(d_out), -5.0, c(inp["init_state"]), c(d_fin))
    torch.cuda.synchronize()
    assert kda_device_status(clear=True) == 0
    for name, key in (("dq", "dq"), ("dk", "dk"), ("dv", "dv"), ("dtheta", "dtheta"),
                      ("dbeta", "dbeta"), ("d_init", "dS0")):
        assert_close(f64(got[name]), ref[key], TOL_BWD, f"{name} T=1000")


@pytest.mark.parametrize("with_final", [True, False])
def test_bwd_empty_and_single_token(with_final):
    """T = 0: no tokens, so the initial state's gradient is the final state's
    (zero without one) and nothing else is written.  T = 1: one ragged chunk
    of a single token against the oracle."""
    B, H = 2, 3
    g = torch.Generator().manual_seed(31)
    d_fin = torch.randn(B, H, 128, 128, generator=g) if with_final else None
    z = lambda *s: torch.zeros(*s, dtype=torch.bfloat16, device="cuda")
    got = kda_chunk_bwd(z(B, 0, H, 128), z(B, 0, H, 128), z(B, 0, H, 128), z(B, 0, H, 128),
                        z(B, 0, H), torch.zeros(B, 0, H, 128, device="cuda"), -5.0,
                        None, d_fin.cuda() if with_final else None)
    torch.cuda.synchronize()
    want = d_fin if with_final else torch.zeros(B, H, 128, 128)
    assert torch.equal(got["d_init"].cpu(), want)

    inp, d_out, d_fin1 = _case(torch.bfloat16, 1, H=H, B=B, seed=32)
    ref = backward.bwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["theta"]),
                       f64(inp["beta"]), -5.0, f64(inp["init_state"]), d_out.double().numpy(),
                       d_fin1.double().numpy() if with_final else None)
    c = lambda x: None if x is None else x.cuda()
    got = kda_chunk_bwd(c(inp["q"]), c(inp["k"]), c(inp["v"]), c(inp["theta"]), c(inp["beta"]),
                        c(d_out), -5.0, c(inp["init_state"]), c(d_fin1) if with_final else None)
    torch.cuda.synchronize()
    assert kda_device_status(clear=True) == 0
    for name, key in (("dq", "dq"), ("dk", "dk"), ("dv", "dv"), ("dtheta", "dtheta"),
                      ("dbeta", "dbeta"), ("d_init", "dS0")):
        assert_close(f64(got[name]), ref[key], TOL_BWD, f"{name} T=1")
