"""Pins of the fp64 backward oracle (CPU): its forward equals the C oracle's,
and its gradients equal central finite differences of the C oracle's forward
(an independent implementation), on tiny inputs in every direction tested."""
import numpy as np
import pytest

import oracle
from oracle import backward


def _tiny(seed, B=1, T=6, H=2, dk=4, dv=3, init=True):
    r = np.random.default_rng(seed)
    q = r.standard_normal((B, T, H, dk))
    k = r.standard_normal((B, T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((B, T, H, dv))
    th = r.standard_normal((B, T, H, dk))
    be = 1 / (1 + np.exp(-r.standard_normal((B, T, H))))
    S0 = 0.3 * r.standard_normal((B, H, dk, dv)) if init else None
    dO = r.standard_normal((B, T, H, dv))
    dS = r.standard_normal((B, H, dk, dv))
    return q, k, v, th, be, S0, dO, dS


def test_forward_matches_the_c_oracle():
    import torch
    q, k, v, th, be, S0, _, _ = _tiny(1, T=9)
    o_c, S_c = oracle.fwd(q, k, v, th, be, -5.0, S0)
    t = lambda x: torch.tensor(x)
    o_t, S_t = backward.forward_torch(t(q), t(k), t(v), t(th), t(be), -5.0, t(S0))
    assert np.max(np.abs(o_t.numpy() - o_c)) < 1e-12
    assert np.max(np.abs(S_t.numpy() - S_c)) < 1e-12


@pytest.mark.parametrize("seed,init,theta_is_g", [(2, True, False), (3, False, False),
                                                  (4, True, True)])
def test_gradients_match_finite_differences(seed, init, theta_is_g):
    q, k, v, th, be, S0, dO, dS = _tiny(seed, init=init)
    if theta_is_g:
        th = -np.log1p(np.exp(th))          # a log-decay, -softplus of the logits
    grads = backward.bwd(q, k, v, th, be, -5.0, S0, dO, dS, theta_is_g=theta_is_g)
    base = dict(q=q, k=k, v=v, theta=th, beta=be, S0=S0 if init else np.zeros_like(dS))

    def loss(x):
        o, S = oracle.fwd(x["q"], x["k"], x["v"], x["theta"], x["beta"], -5.0, x["S0"],
                          theta_is_g=theta_is_g)
        return float(np.sum(o * dO) + np.sum(S * dS))

    r = np.random.default_rng(seed + 100)
    eps = 1e-6
    for name, gname in (("q", "dq"), ("k", "dk"), ("v", "dv"), ("theta", "dtheta"),
                        ("beta", "dbeta"), ("S0", "dS0")):
        for _ in range(3):
            d = r.standard_normal(base[name].shape)
            xp = dict(base)
            xm = dict(base)
            xp[name] = base[name] + eps * d
            xm[name] = base[name] - eps * d
            fd = (loss(xp) - loss(xm)) / (2 * eps)
            an = float(np.sum(grads[gname] * d))
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)
