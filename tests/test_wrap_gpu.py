"""The wrapped schedule of the register-resident forward path.

A fixed-length batch with more (sequence, head) chains than CTAs that can be
resident at once (and not a multiple of that count) runs as equal windows of
chunk steps, one window per resident CTA, over the chains laid end to end.  A
chain cut by a window boundary runs its first chunks at the start of the later
window and the rest at the end of the earlier one; its state is handed over
through the chain's final-state slot.  The hand-over is an exact fp32 copy,
so the wrapped launch must equal, bit for bit in outputs and final states, the
same batch launched in slices of at most one chain per SM (each slice runs one
chain per CTA); and it must match the fp64 oracle on every chain.  The recurrence itself is the one of "Kimi K3 Deep Dive", section
"Core Innovation 1", with the gate of "Architecture Deep Dive", sec. 3.2."""
import numpy as np
import pytest
import torch

from linear_attention_04_gb300 import kda_chunk_fwd, kda_device_status
from linear_attention_04_gb300.workloads import Workload, make_inputs

from parity import TOL, assert_close, f64
import oracle

pytestmark = pytest.mark.gpu


def _sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _batch(extra_chains, H):
    """(B, H) with B * H = SM count + extra_chains rounded up to whole
    sequences, and not a multiple of the SM count."""
    n = _sms() + extra_chains
    B = -(-n // H)
    assert (B * H) % _sms() != 0
    return B, H


def _cuda(inp):
    return {k_: (x.cuda() if isinstance(x, torch.Tensor) else x) for k_, x in inp.items()}


def _fwd(c, theta, path, gate, out_dtype=torch.float32):
    o, S = kda_chunk_fwd(c["q"], c["k"], c["v"], theta, c["beta"], -5.0, c["init_state"],
                         path=path, gate=gate, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert kda_device_status(clear=True) == 0
    return o, S


def _sliced(c, theta, path, gate, out_dtype=torch.float32):
    """The same batch in slices of whole sequences with at most one chain per
    SM each: every slice runs one chain per CTA."""
    B, H = c["q"].shape[0], c["q"].shape[2]
    step = max(1, _sms() // H)
    outs, states = [], []
    for b0 in range(0, B, step):
        sl = slice(b0, min(B, b0 + step))
        o, S = kda_chunk_fwd(c["q"][sl], c["k"][sl], c["v"][sl], theta[sl], c["beta"][sl], -5.0,
                             None if c["init_state"] is None else c["init_state"][sl],
                             path=path, gate=gate, out_dtype=out_dtype)
        outs.append(o)
        states.append(S)
    torch.cuda.synchronize()
    assert kda_device_status(clear=True) == 0
    return torch.cat(outs), torch.cat(states)


def _oracle(inp, theta, gate, init):
    return oracle.fwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(theta), f64(inp["beta"]),
                      -5.0, None if init is None else f64(init), theta_is_g=gate == "log_decay")


@pytest.mark.parametrize("path", ["mma", "mma_tc"])
@pytest.mark.parametrize("T", [100, 96])  # a ragged last chunk, and whole chunks only
def test_wrapped_equals_plain_and_oracle(path, T):
    B, H = _batch(8, 16)
    w = Workload("wrap", B=B, H=H, T=T, dk=128, dv=128, dtype=torch.bfloat16, init_std=0.02)
    inp = make_inputs(w, seed=41 + T)
    c = _cuda(inp)
    o_w, S_w = _fwd(c, c["theta"], path, "sigmoid")
    o_p, S_p = _sliced(c, c["theta"], path, "sigmoid")
    assert torch.equal(o_w, o_p), "wrapped and one-chain-per-CTA outputs differ"
    assert torch.equal(S_w, S_p), "wrapped and one-chain-per-CTA final states differ"
    ro, rS = _oracle(inp, inp["theta"], "sigmoid", inp["init_state"])
    tol = TOL[torch.bfloat16]
    assert_close(f64(o_w), ro, tol, f"wrapped out ({path}, T={T})")
    assert_close(f64(S_w), rS, tol, f"wrapped state ({path}, T={T})")


def test_wrapped_short_windows():
    # one chain more than the SMs and 17 chunks per chain: every window is one
    # chunk-step longer than a chain, so nearly every chain is cut and a cut
    # chain's second part starts right after its first part ends (the
    # hand-over wait is exercised, not hidden behind other work)
    B, H = _batch(1, 1)
    w = Workload("wrap", B=B, H=H, T=257, dk=128, dv=128, dtype=torch.bfloat16)
    inp = make_inputs(w, seed=43)
    c = _cuda(inp)
    o_w, S_w = _fwd(c, c["theta"], "mma", "sigmoid")
    o_p, S_p = _sliced(c, c["theta"], "mma", "sigmoid")
    assert torch.equal(o_w, o_p) and torch.equal(S_w, S_p)
    ro, rS = _oracle(inp, inp["theta"], "sigmoid", None)
    tol = TOL[torch.bfloat16]
    assert_close(f64(o_w), ro, tol, "short windows out")
    assert_close(f64(S_w), rS, tol, "short windows state")


def test_wrapped_log_decay_gate_and_bf16_out():
    # the other instantiations: the log-decay gate (with the position-wise
    # fallback compiled in) and bf16 outputs.  Their precision against the
    # oracle is the gate tests' subject; here the final states only have to
    # equal the one-chain-per-CTA launch's, and the outputs stay within the
    # bf16-output bar
    B, H = _batch(8, 16)
    w = Workload("wrap", B=B, H=H, T=80, dk=128, dv=128, dtype=torch.bfloat16)
    inp = make_inputs(w, seed=44)
    g = (-torch.nn.functional.softplus(inp["theta"].float() + 2.0)).to(torch.bfloat16)
    c = _cuda(inp)
    gc = g.cuda()
    o_w, S_w = _fwd(c, gc, "mma", "log_decay", out_dtype=torch.bfloat16)
    o_p, S_p = _sliced(c, gc, "mma", "log_decay", out_dtype=torch.bfloat16)
    assert torch.equal(o_w, o_p) and torch.equal(S_w, S_p)
    ro, _ = _oracle(inp, g, "log_decay", None)
    # bf16 outputs: within the bar plus one bf16 rounding of each output
    got = f64(o_w)
    rms = float(np.sqrt(np.mean(ro ** 2)))
    assert np.all(np.abs(got - ro) <= TOL[torch.bfloat16] * rms + np.abs(ro) * 2.0 ** -8)


def test_wrapped_in_place_state():
    # init_state and final_state the same buffer: a cut chain's first part
    # reads its initial state before it writes the hand-over into that slot
    B, H = _batch(8, 16)
    w = Workload("wrap", B=B, H=H, T=64, dk=128, dv=128, dtype=torch.bfloat16, init_std=0.02)
    inp = make_inputs(w, seed=45)
    c = _cuda(inp)
    S = c["init_state"].clone()
    o, S2 = kda_chunk_fwd(c["q"], c["k"], c["v"], c["theta"], c["beta"], -5.0, S,
                          final_state=S, path="mma")
    torch.cuda.synchronize()
    assert kda_device_status(clear=True) == 0
    assert S2.data_ptr() == S.data_ptr()
    ro, rS = _oracle(inp, inp["theta"], "sigmoid", inp["init_state"])
    tol = TOL[torch.bfloat16]
    assert_close(f64(o), ro, tol, "in-place out")
    assert_close(f64(S), rS, tol, "in-place state")


def test_wrapped_flag_ring_reuse():
    # 140 wrapped launches in a row: each flag region of the 64-slot ring is
    # reused with the flags of an older launch still in it; a flag only passes
    # when it holds the current launch's epoch, so every launch must give the
    # same outputs and final states, bit for bit
    B, H = _batch(8, 16)
    w = Workload("wrap", B=B, H=H, T=48, dk=128, dv=128, dtype=torch.bfloat16, init_std=0.02)
    c = _cuda(make_inputs(w, seed=46))
    o0, S0 = _fwd(c, c["theta"], "mma", "sigmoid")
    out = torch.empty_like(o0)
    S = torch.empty_like(S0)
    for i in range(140):
        kda_chunk_fwd(c["q"], c["k"], c["v"], c["theta"], c["beta"], -5.0, c["init_state"], out, S,
                      path="mma")
        if i % 20 == 19:
            torch.cuda.synchronize()
            assert kda_device_status(clear=True) == 0
            assert torch.equal(out, o0) and torch.equal(S, S0), f"launch {i}"
    torch.cuda.synchronize()
    assert kda_device_status(clear=True) == 0
    assert torch.equal(out, o0) and torch.equal(S, S0)
