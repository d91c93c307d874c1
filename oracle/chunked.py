"""fp64 restatement of the chunk-parallel form of the KDA forward pass.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The recurrence S_t = (I - b_t k_t k_t^T) Diag(e^{g_t}) S_{t-1} + b_t k_t v_t^T,
o_t = S_t^T q_t is regrouped over chunks of C tokens.  Inside a chunk, with the
inclusive in-chunk cumulative log-decay G_r = g_1 + ... + g_r (the decay
product Gamma_ij of "Kimi K3 Deep Dive", section "The Problem", is
exp(G_j - G_i)), and

    Kt = K * e^{G},  Kh = K * e^{-G},  Qt = Q * e^{G},  KhC = K * e^{G_C - G}

the chunk is

    A  = strict_lower(Diag(b) Kt Kh^T)          P = lower_incl_diag(Qt Kh^T)
    Tm = (I + A)^{-1}                           (unit lower triangular)
    W  = Tm Diag(b) Kt                          U' = Tm Diag(b) V
    U  = U' - W S0                              O  = Qt S0 + P U
    S  = Diag(e^{G_C}) S0 + KhC^T U

Derivation: unrolling the recurrence inside the chunk gives
S_r = Gamma_r S0 + sum_{s<=r} Gamma_r Gamma_s^{-1} k_s u_s^T with
u_r = b_r (v_r - S_{r-1}^T Diag(e^{g_r}) k_r); collecting the u_r of a chunk
into U gives the triangular system (I + A) U = Diag(b)(V - Kt S0), and
substituting S_r into o_r = S_r^T q_r gives O.  The 16-token chunk is the size
"Kimi K3 Deep Dive" gives ("A typical chunk size is 16 tokens").

The inverse is taken with numpy's dense solver (a library routine serving as
one step); nothing else is fused or reordered.
"""
from __future__ import annotations

import numpy as np


def gate(theta, g_min):
    return g_min / (1.0 + np.exp(-np.asarray(theta, dtype=np.float64)))


def chunk_stages(Q, K, V, g, b, S0):
    """One chunk of one (sequence, head).  Q,K,g [n,dk]; V [n,dv]; b [n]; S0 [dk,dv].

    Returns a dict with every intermediate and the outputs O [n,dv], S [dk,dv].
    """
    n = Q.shape[0]
    G = np.cumsum(g, axis=0)
    eG = np.exp(G)
    Kt = K * eG
    Kh = K * np.exp(-G)
    Qt = Q * eG
    KhC = K * np.exp(G[-1][None, :] - G)
    A = np.tril(b[:, None] * (Kt @ Kh.T), -1)
    P = np.tril(Qt @ Kh.T, 0)
    Tm = np.linalg.solve(np.eye(n) + A, np.eye(n))
    W = Tm @ (b[:, None] * Kt)
    Up = Tm @ (b[:, None] * V)
    U = Up - W @ S0
    O = Qt @ S0 + P @ U
    S = np.exp(G[-1])[:, None] * S0 + KhC.T @ U
    return dict(G=G, Kt=Kt, Kh=Kh, Qt=Qt, KhC=KhC, A=A, P=P, T=Tm, W=W, Up=Up, U=U, O=O, S=S)


def fwd_chain(Q, K, V, g, b, S0, chunk):
    """A whole sequence of one head: Q,K,g [L,dk]; V [L,dv]; b [L]; S0 [dk,dv]."""
    L = Q.shape[0]
    out = np.zeros((L, V.shape[1]))
    S = np.array(S0, dtype=np.float64, copy=True)
    for c0 in range(0, L, chunk):
        c1 = min(L, c0 + chunk)
        st = chunk_stages(Q[c0:c1], K[c0:c1], V[c0:c1], g[c0:c1], b[c0:c1], S)
        out[c0:c1] = st["O"]
        S = st["S"]
    return out, S


def fwd(q, k, v, theta, beta, g_min=-5.0, init_state=None, cu_seqlens=None, *, chunk=16,
        theta_is_g=False):
    """Same contract as ``oracle.fwd`` (erase mode only), computed chunk by chunk."""
    q, k, v, theta, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, theta, beta))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    g = theta if theta_is_g else gate(theta, g_min)
    if cu_seqlens is None:
        spans = [(b, 0, T) for b in range(B)]
    else:
        cu = np.asarray(cu_seqlens)
        spans = [(0, int(cu[s]), int(cu[s + 1])) for s in range(len(cu) - 1)]
    out = np.zeros((B, T, H, dv))
    fin = np.zeros((len(spans), H, dk, dv))
    for si, (b, t0, t1) in enumerate(spans):
        for h in range(H):
            S0 = np.zeros((dk, dv)) if init_state is None else np.asarray(init_state)[si, h]
            o, S = fwd_chain(q[b, t0:t1, h], k[b, t0:t1, h], v[b, t0:t1, h], g[b, t0:t1, h],
                             beta[b, t0:t1, h], S0, chunk)
            out[b, t0:t1, h] = o
            fin[si, h] = S
    return out, fin
