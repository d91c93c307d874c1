"""Pins for the fp64 oracle: facts the pages and the mathematics fix, checked
against the oracle without trusting it.  CPU only.

Each pin is a function taking a ``run`` callable with the signature of
``oracle.fwd`` and returning (passed, error).  ``test_planted_mistakes`` feeds
the oracle with each planted mistake and requires at least one pin to fail.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import chunked

RNG = np.random.default_rng(1234)


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _inputs(B=1, T=12, H=2, dk=4, dv=3, seed=0, init=True, theta_scale=1.0):
    r = np.random.default_rng(seed)
    q = _unit(r.standard_normal((B, T, H, dk)))
    k = _unit(r.standard_normal((B, T, H, dk)))
    v = r.standard_normal((B, T, H, dv))
    th = theta_scale * r.standard_normal((B, T, H, dk))
    be = 1.0 / (1.0 + np.exp(-r.standard_normal((B, T, H))))
    S0 = 0.5 * r.standard_normal((B, H, dk, dv)) if init else None
    return q, k, v, th, be, S0


def _close(a, b, tol):
    err = float(np.max(np.abs(a - b)) / max(1e-300, np.max(np.abs(b)), 1e-12))
    return err <= tol, err


# --------------------------------------------------------------------------
# pins on the recurrence
# --------------------------------------------------------------------------

def pin_bruteforce(run):
    """Brute-force unrolled form: S_t = (M_t..M_1) S_0 + sum_i (M_t..M_{i+1}) b_i k_i v_i^T
    with M_t = (I - b_t k_t k_t^T) Diag(e^{g_t}); o_t = S_t^T q_t.  Explicit
    dk x dk products, O(T^2 dk^3); log-decay passed directly (gate bypassed)."""
    B, T, H, dk, dv = 2, 10, 2, 4, 3
    q, k, v, th, be, S0 = _inputs(B, T, H, dk, dv, seed=11)
    g = -5.0 / (1.0 + np.exp(-th))  # any log-decay in [-5, 0]
    o, S = run(q, k, v, g, be, -5.0, S0, theta_is_g=True)
    ref_o = np.zeros_like(o)
    ref_S = np.zeros_like(S)
    I = np.eye(dk)
    for b in range(B):
        for h in range(H):
            M = [(I - be[b, t, h] * np.outer(k[b, t, h], k[b, t, h])) @ np.diag(np.exp(g[b, t, h]))
                 for t in range(T)]
            for t in range(T):
                prod = I.copy()
                for s in range(t + 1):
                    prod = M[s] @ prod
                St = prod @ S0[b, h]
                for i in range(t + 1):
                    P = I.copy()
                    for s in range(i + 1, t + 1):
                        P = M[s] @ P
                    St = St + P @ (be[b, i, h] * np.outer(k[b, i, h], v[b, i, h]))
                ref_o[b, t, h] = St.T @ q[b, t, h]
                if t == T - 1:
                    ref_S[b, h] = St
    ok1, e1 = _close(o, ref_o, 1e-12)
    ok2, e2 = _close(S, ref_S, 1e-12)
    return ok1 and ok2, max(e1, e2)


def pin_retrieval_beta1(run):
    """With unit keys and beta = 1 the delta rule overwrites the value stored
    under k_t: S_t^T k_t = v_t exactly, whatever the decay and the state.  So
    with q = k the output equals v."""
    q, k, v, th, be, S0 = _inputs(1, 20, 2, 6, 6, seed=12, theta_scale=3.0)
    be = np.ones_like(be)
    o, _ = run(k, k, v, th, be, -5.0, S0)
    return _close(o, v, 1e-12)


def pin_retrieval_general_beta(run):
    """General beta: S_t^T k_t = (1 - b_t) (Diag(e^{g_t}) S_{t-1})^T k_t + b_t v_t.
    S_{t-1} is taken from the oracle's own final state over the prefix, and
    Diag(e^{g_t}) applied here."""
    q, k, v, th, be, S0 = _inputs(1, 9, 1, 5, 4, seed=13)
    g = -5.0 / (1.0 + np.exp(-th))
    errs = []
    for t in (1, 4, 8):
        _, Sp = run(k[:, :t], k[:, :t], v[:, :t], g[:, :t], be[:, :t], -5.0, S0, theta_is_g=True)
        o, _ = run(k[:, :t + 1], k[:, :t + 1], v[:, :t + 1], g[:, :t + 1], be[:, :t + 1], -5.0, S0,
                   theta_is_g=True)
        D = np.exp(g[0, t, 0])[:, None] * Sp[0, 0]
        ref = (1 - be[0, t, 0]) * (D.T @ k[0, t, 0]) + be[0, t, 0] * v[0, t, 0]
        errs.append(_close(o[0, t, 0], ref, 1e-12))
    return all(e[0] for e in errs), max(e[1] for e in errs)


def pin_beta0_closed_form(run):
    """Literal beta = 0: nothing is written or erased, the state only decays,
    so o_t = S_0^T (e^{G_t} * q_t) with G_t the log-decay summed from the
    sequence start."""
    q, k, v, th, be, S0 = _inputs(2, 15, 2, 4, 3, seed=14)
    be = np.zeros_like(be)
    g = -5.0 / (1.0 + np.exp(-th)) * 0.1  # keep e^{G} away from underflow
    o, S = run(q, k, v, g, be, -5.0, S0, theta_is_g=True)
    G = np.cumsum(g, axis=1)
    ref = np.einsum("bhij,bthi->bthj", S0, np.exp(G) * q)
    refS = np.exp(G[:, -1])[..., None] * S0
    ok1, e1 = _close(o, ref, 1e-12)
    ok2, e2 = _close(S, refS, 1e-12)
    return ok1 and ok2, max(e1, e2)


def pin_gla(run):
    """Erase term dropped (gated linear attention, write weight b_i):
    o_t = S_0^T (e^{G_t} q_t) + sum_{i<=t} b_i ((q_t * e^{G_t - G_i}) . k_i) v_i,
    the O(T^2) form."""
    q, k, v, th, be, S0 = _inputs(1, 14, 2, 5, 4, seed=15)
    g = -5.0 / (1.0 + np.exp(-th))
    o, _ = run(q, k, v, g, be, -5.0, S0, theta_is_g=True, erase=False)
    G = np.cumsum(g, axis=1)
    ref = np.zeros_like(o)
    T = q.shape[1]
    for h in range(q.shape[2]):
        for t in range(T):
            acc = S0[0, h].T @ (np.exp(G[0, t, h]) * q[0, t, h])
            for i in range(t + 1):
                w = np.dot(q[0, t, h] * np.exp(G[0, t, h] - G[0, i, h]), k[0, i, h])
                acc = acc + be[0, i, h] * w * v[0, i, h]
            ref[0, t, h] = acc
    return _close(o, ref, 1e-12)


def pin_causal_linear_attention(run):
    """Erase dropped, g = 0, beta = 1, zero start: plain causal linear
    attention o_t = (sum_{i<=t} k_i v_i^T)^T q_t, via a cumulative sum."""
    q, k, v, th, be, _ = _inputs(1, 17, 3, 6, 4, seed=16, init=False)
    g = np.zeros_like(th)
    be = np.ones_like(be)
    o, _ = run(q, k, v, g, be, -5.0, None, theta_is_g=True, erase=False)
    KV = np.cumsum(np.einsum("bthi,bthj->bthij", k, v), axis=1)
    ref = np.einsum("bthij,bthi->bthj", KV, q)
    return _close(o, ref, 1e-12)


def pin_chunk_invariance(run):
    """The chunk-parallel (WY) restatement gives the same result for any chunk
    size; it must equal the token-by-token oracle."""
    q, k, v, th, be, S0 = _inputs(2, 37, 2, 8, 6, seed=17)
    o, S = run(q, k, v, th, be, -5.0, S0)
    worst, ok = 0.0, True
    for C in (1, 4, 16, 32):
        oc, Sc = chunked.fwd(q, k, v, th, be, -5.0, S0, chunk=C)
        a, e1 = _close(o, oc, 1e-11)
        b, e2 = _close(S, Sc, 1e-11)
        ok = ok and a and b
        worst = max(worst, e1, e2)
    return ok, worst


def pin_state_continuation(run):
    """Running [0, T1) and then [T1, T) from the returned state equals the
    whole run (the recurrent state is a complete checkpoint)."""
    q, k, v, th, be, S0 = _inputs(2, 30, 2, 6, 5, seed=18)
    o, S = run(q, k, v, th, be, -5.0, S0)
    T1 = 13
    o1, S1 = run(q[:, :T1], k[:, :T1], v[:, :T1], th[:, :T1], be[:, :T1], -5.0, S0)
    o2, S2 = run(q[:, T1:], k[:, T1:], v[:, T1:], th[:, T1:], be[:, T1:], -5.0, S1)
    ok1, e1 = _close(np.concatenate([o1, o2], axis=1), o, 1e-12)
    ok2, e2 = _close(S2, S, 1e-12)
    return ok1 and ok2, max(e1, e2)


def pin_linearity(run):
    """For fixed q, k, g, beta the map (V, S_0) -> (o, S_T) is linear."""
    q, k, v, th, be, S0 = _inputs(1, 16, 2, 5, 4, seed=19)
    r = np.random.default_rng(20)
    v2 = r.standard_normal(v.shape)
    S2 = r.standard_normal(S0.shape)
    a, b = 0.7, -1.3
    o1, F1 = run(q, k, v, th, be, -5.0, S0)
    o2, F2 = run(q, k, v2, th, be, -5.0, S2)
    o3, F3 = run(q, k, a * v + b * v2, th, be, -5.0, a * S0 + b * S2)
    ok1, e1 = _close(o3, a * o1 + b * o2, 1e-12)
    ok2, e2 = _close(F3, a * F1 + b * F2, 1e-12)
    return ok1 and ok2, max(e1, e2)


def pin_column_independence(run):
    """Column j of o and of S_T depends only on column j of V and of S_0."""
    q, k, v, th, be, S0 = _inputs(1, 16, 1, 5, 6, seed=21)
    o1, F1 = run(q, k, v, th, be, -5.0, S0)
    v2 = v.copy()
    S2 = S0.copy()
    v2[..., 2] += 1.0
    S2[..., 2] -= 0.5
    o2, F2 = run(q, k, v2, th, be, -5.0, S2)
    keep = [j for j in range(6) if j != 2]
    ok1, e1 = _close(o2[..., keep], o1[..., keep], 1e-13)
    ok2, e2 = _close(F2[..., keep], F1[..., keep], 1e-13)
    moved = np.max(np.abs(o2[..., 2] - o1[..., 2])) > 1e-3
    return ok1 and ok2 and moved, max(e1, e2)


def pin_varlen_independence(run):
    """A packed batch with cu_seqlens equals independent runs of each sequence,
    each starting from its own initial state."""
    lens = [5, 16, 1, 11]
    H, dk, dv = 2, 4, 3
    Tt = sum(lens)
    q, k, v, th, be, _ = _inputs(1, Tt, H, dk, dv, seed=22, init=False)
    S0 = np.random.default_rng(23).standard_normal((len(lens), H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    o, S = run(q, k, v, th, be, -5.0, S0, cu_seqlens=cu)
    ok, worst = True, 0.0
    for s in range(len(lens)):
        a, b = cu[s], cu[s + 1]
        os_, Ss = run(q[:, a:b], k[:, a:b], v[:, a:b], th[:, a:b], be[:, a:b], -5.0, S0[s:s + 1])
        x, e1 = _close(o[:, a:b], os_, 1e-13)
        y, e2 = _close(S[s:s + 1], Ss, 1e-13)
        ok = ok and x and y
        worst = max(worst, e1, e2)
    return ok, worst


PINS = [pin_bruteforce, pin_retrieval_beta1, pin_retrieval_general_beta, pin_beta0_closed_form,
        pin_gla, pin_causal_linear_attention, pin_chunk_invariance, pin_state_continuation,
        pin_linearity, pin_column_independence, pin_varlen_independence]


def _run_plain(*a, **kw):
    return oracle.fwd(*a, **kw)


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    ok, err = pin(_run_plain)
    assert ok, f"{pin.__name__}: error {err:.3e}"


# --------------------------------------------------------------------------
# pins on the gate (closed-form sigmoid values and the bound)
# --------------------------------------------------------------------------

def test_gate_closed_form():
    """g = g_min * sigmoid(theta) ("Kimi K3 Deep Dive", section "The Design"):
    sigmoid(0) = 1/2, sigmoid(ln 3) = 3/4, sigmoid(-ln 3) = 1/4, limits 1 and 0."""
    th = np.array([0.0, math.log(3.0), -math.log(3.0), 800.0, -800.0])
    g = oracle.gate(th, -5.0)
    ref = np.array([-2.5, -3.75, -1.25, -5.0, 0.0])
    assert np.max(np.abs(g - ref)) < 1e-15


def test_gate_used_by_recurrence():
    """fwd(theta) must equal fwd(g = gate(theta)) with the gate bypassed."""
    q, k, v, th, be, S0 = _inputs(1, 12, 2, 4, 3, seed=30, theta_scale=4.0)
    o1, S1 = oracle.fwd(q, k, v, th, be, -5.0, S0)
    o2, S2 = oracle.fwd(q, k, v, oracle.gate(th, -5.0), be, -5.0, S0, theta_is_g=True)
    assert np.array_equal(o1, o2) and np.array_equal(S1, S2)


@pytest.mark.parametrize("dist", ["normal", "uniform6_12", "extreme"])
def test_gmin_bound(dist):
    """The bound that removes the position-wise fallback: with g in [g_min, 0]
    the inverse decay inside any 16-token tile is at most e^{5*16} = e^{80}
    ("Architecture Deep Dive ...", sec. 3.2; "Kimi K3" explainer), finite in
    bf16 (max about 3.39e38), and its reciprocal is a normal bf16 number."""
    r = np.random.default_rng(31)
    n = 16 * 64
    if dist == "normal":
        th = r.standard_normal((n, 128))
    elif dist == "uniform6_12":
        th = r.uniform(6, 12, (n, 128))
    else:
        th = np.full((n, 128), 1e4)
    g = oracle.gate(th, -5.0)
    assert g.min() >= -5.0 and g.max() <= 0.0
    G = np.cumsum(g.reshape(-1, 16, 128), axis=1)  # inclusive, reset per chunk
    worst = float(np.max(-G))
    assert worst <= 80.0 * (1 + 1e-6)
    big = torch.tensor(math.exp(worst), dtype=torch.float64).to(torch.bfloat16)
    assert torch.isfinite(big).item()
    assert float(torch.tensor(math.exp(80.0)).to(torch.bfloat16)) < 3.39e38
    tiny = torch.tensor(math.exp(-80.0), dtype=torch.float64).to(torch.bfloat16)
    assert float(tiny) > 1.17549435e-38  # normal, not flushed
    if dist == "uniform6_12":
        assert worst > 79.0  # the stress workload really sits near the bound


def test_threads_deterministic():
    q, k, v, th, be, S0 = _inputs(3, 40, 3, 8, 8, seed=32)
    o1, S1 = oracle.fwd(q, k, v, th, be, -5.0, S0, nthreads=1)
    o2, S2 = oracle.fwd(q, k, v, th, be, -5.0, S0, nthreads=7)
    assert np.array_equal(o1, o2) and np.array_equal(S1, S2)


def test_rejects_bad_args():
    q, k, v, th, be, S0 = _inputs(1, 8, 1, 4, 4, seed=33)
    with pytest.raises(ValueError):
        oracle.fwd(q, k, v, th, be, -5.0, None, cu_seqlens=np.array([0, 3, 9]))  # 9 != T


# --------------------------------------------------------------------------
# planted mistakes: each must be caught by at least one pin
# --------------------------------------------------------------------------

@pytest.mark.parametrize("mutation", sorted(oracle.MUTATIONS))
def test_planted_mistakes(mutation):
    def run(*a, **kw):
        kw = dict(kw)
        kw["mutation"] = mutation
        return oracle.fwd(*a, **kw)

    failed = []
    for pin in PINS:
        try:
            res = pin(run)
        except ValueError:
            continue  # this mutation does not apply to the pin's shapes
        if not res[0]:
            failed.append(pin.__name__)
    if mutation == "gate_sign":
        # the recurrence pins bypass the gate; the gate itself is pinned by
        # closed-form values.  Run those against the mutated gate path.
        q, k, v, th, be, S0 = _inputs(1, 6, 1, 3, 3, seed=40)
        o1, _ = oracle.fwd(q, k, v, th, be, -5.0, S0, mutation=mutation)
        o2, _ = oracle.fwd(q, k, v, oracle.gate(th, -5.0), be, -5.0, S0, theta_is_g=True)
        if not np.allclose(o1, o2, rtol=1e-12, atol=1e-14):
            failed.append("gate_used_by_recurrence")
    assert failed, f"planted mistake '{mutation}' passed every pin"
