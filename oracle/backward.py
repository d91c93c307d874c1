"""fp64 gradients of the KDA forward pass, by reverse-mode differentiation of
the token-by-token recurrence.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): only ``tests/`` may
import this module.

The forward pass differentiated here is the recurrence of "Kimi K3 Deep Dive",
section "Core Innovation 1", with the bounded gate of "Architecture Deep Dive",
sec. 3.2 (or a given log-decay):

    g_t = g_min * sigmoid(theta_t)
    S_t = (I - b_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + b_t k_t v_t^T,   o_t = S_t^T q_t

written out again with plain PyTorch CPU tensor operations in float64 (no code
shared with ``kda_oracle.c``); torch.autograd supplies the reverse pass.  For
a loss with upstream gradients d_out (w.r.t. o) and d_final (w.r.t. the final
state), ``bwd`` returns the gradients w.r.t. q, k, v, theta, beta and the
initial state.

Parity status: pinned -- by central finite differences of the C oracle's
forward (an independent implementation) and by the forward values of the C
oracle (tests/test_oracle_backward.py).
"""
from __future__ import annotations

import numpy as np
import torch


def forward_torch(q, k, v, theta, beta, g_min, init_state, theta_is_g=False):
    """The recurrence in float64 torch ops.  q, k, theta [B,T,H,dk]; v [B,T,H,dv];
    beta [B,T,H]; init_state [B,H,dk,dv] or None.  Returns (o, S_T)."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    S = (torch.zeros(B, H, dk, dv, dtype=torch.float64) if init_state is None
         else init_state)
    outs = []
    for t in range(T):
        g = theta[:, t] if theta_is_g else g_min * torch.sigmoid(theta[:, t])
        S = torch.exp(g)[..., None] * S                              # Diag(e^g) S
        kt = k[:, t]
        kS = torch.einsum("bhk,bhkv->bhv", kt, S)                    # k^T S
        S = S + beta[:, t][..., None, None] * kt[..., None] * (v[:, t] - kS)[..., None, :]
        outs.append(torch.einsum("bhk,bhkv->bhv", q[:, t], S))       # S^T q
    return torch.stack(outs, dim=1), S


def bwd(q, k, v, theta, beta, g_min, init_state, d_out, d_final=None, *, theta_is_g=False):
    """Gradients of sum(o * d_out) + sum(S_T * d_final).  Array arguments are
    numpy arrays (any float dtype, used as float64); d_final and init_state may
    be None.  Returns a dict of float64 numpy arrays: dq, dk, dv, dtheta,
    dbeta, dS0 (dS0 is present even without an initial state: the gradient
    w.r.t. a zero initial state)."""
    t64 = lambda x: torch.tensor(np.asarray(x, dtype=np.float64), requires_grad=True)
    q_, k_, v_, th_, b_ = (t64(x) for x in (q, k, v, theta, beta))
    B, T, H, dk = q_.shape
    dv = v_.shape[-1]
    S0 = t64(np.zeros((B, H, dk, dv)) if init_state is None else init_state)
    o, S = forward_torch(q_, k_, v_, th_, b_, g_min, S0, theta_is_g)
    loss = (o * torch.tensor(np.asarray(d_out, dtype=np.float64))).sum()
    if d_final is not None:
        loss = loss + (S * torch.tensor(np.asarray(d_final, dtype=np.float64))).sum()
    loss.backward()
    return {"dq": q_.grad.numpy(), "dk": k_.grad.numpy(), "dv": v_.grad.numpy(),
            "dtheta": th_.grad.numpy(), "dbeta": b_.grad.numpy(), "dS0": S0.grad.numpy()}
