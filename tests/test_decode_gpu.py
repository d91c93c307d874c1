"""GPU parity of the decode step (kda_decode_step): one token per (sequence,
head) against a resident fp32 state, checked against the fp64 oracle's
recurrence for T = 1 and, stepped T times, against the oracle over T tokens."""
import numpy as np
import pytest
import torch

from linear_attention_04_gb300 import kda_chunk_fwd, kda_decode_step, kda_device_status

from parity import assert_close, f64
import oracle

pytestmark = pytest.mark.gpu

# fp32 arithmetic on both input dtypes (no reduced-precision operands)
TOL_DECODE = 1e-4


def _inputs(N, H, T, dk, dv, dtype, seed, state_std=0.3):
    g = torch.Generator().manual_seed(seed)
    q = torch.nn.functional.normalize(torch.randn(N, T, H, dk, generator=g), dim=-1)
    k = torch.nn.functional.normalize(torch.randn(N, T, H, dk, generator=g), dim=-1)
    v = torch.randn(N, T, H, dv, generator=g)
    th = torch.randn(N, T, H, dk, generator=g)
    be = torch.sigmoid(torch.randn(N, T, H, generator=g))
    S0 = state_std * torch.randn(N, H, dk, dv, generator=g)
    cast = [x.to(dtype) for x in (q, k, v, th, be)]
    return cast, S0


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk,dv", [(16, 16), (64, 32), (128, 128), (32, 128)])
def test_decode_step_vs_oracle(dtype, dk, dv):
    (q, k, v, th, be), S0 = _inputs(3, 4, 1, dk, dv, dtype, seed=dk * 7 + dv)
    ro, rS = oracle.fwd(f64(q), f64(k), f64(v), f64(th), f64(be), -5.0, f64(S0))
    dev = [x[:, 0].contiguous().cuda() for x in (q, k, v, th, be)]
    state = S0.clone().cuda()
    out = kda_decode_step(*dev, state, g_min=-5.0)
    torch.cuda.synchronize()
    assert kda_device_status(clear=True) == 0
    assert_close(f64(out), ro[:, 0], TOL_DECODE, "decode out")
    assert_close(f64(state), rS, TOL_DECODE, "decode state")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_steps_equal_the_recurrence_over_a_sequence(dtype):
    N, H, T, d = 2, 3, 37, 128
    (q, k, v, th, be), S0 = _inputs(N, H, T, d, d, dtype, seed=99, state_std=0.05)
    ro, rS = oracle.fwd(f64(q), f64(k), f64(v), f64(th), f64(be), -5.0, f64(S0))
    state = S0.clone().cuda()
    outs = []
    for t in range(T):
        dev = [x[:, t].contiguous().cuda() for x in (q, k, v, th, be)]
        outs.append(kda_decode_step(*dev, state, g_min=-5.0))
    torch.cuda.synchronize()
    o = torch.stack(outs, 1)
    assert_close(f64(o), ro, TOL_DECODE, "decoded sequence")
    assert_close(f64(state), rS, TOL_DECODE, "decoded final state")
    # and the chunked forward over the same tokens continues from the same state
    if dtype == torch.bfloat16:
        co, cS = kda_chunk_fwd(*(x.cuda() for x in (q, k, v, th, be)), -5.0, S0.cuda())
        torch.cuda.synchronize()
        assert_close(f64(co), ro, 2e-2, "chunk path, same tokens")


def test_decode_large_batch_sampled():
    # a serving-sized batch: 128 sequences x 32 heads, checked on sampled heads
    N, H, d = 128, 32, 128
    (q, k, v, th, be), S0 = _inputs(N, H, 1, d, d, torch.bfloat16, seed=5)
    dev = [x[:, 0].contiguous().cuda() for x in (q, k, v, th, be)]
    state = S0.cuda()
    out = kda_decode_step(*dev, state, g_min=-5.0)
    torch.cuda.synchronize()
    for (n, h) in [(0, 0), (77, 13), (127, 31)]:
        ro, rS = oracle.fwd(f64(q[n:n + 1, :, h:h + 1]), f64(k[n:n + 1, :, h:h + 1]),
                            f64(v[n:n + 1, :, h:h + 1]), f64(th[n:n + 1, :, h:h + 1]),
                            f64(be[n:n + 1, :, h:h + 1]), -5.0, f64(S0[n:n + 1, h:h + 1]))
        assert_close(f64(out[n, h]), ro[0, 0, 0], TOL_DECODE, f"out n{n} h{h}")
        assert_close(f64(state[n, h]), rS[0, 0], TOL_DECODE, f"state n{n} h{h}")


def test_decode_empty_batch():
    z = torch.empty((0, 2, 16), device="cuda")
    state = torch.empty((0, 2, 16, 16), device="cuda")
    out = kda_decode_step(z, z, torch.empty((0, 2, 16), device="cuda"), z,
                          torch.empty((0, 2), device="cuda"), state)
    assert out.shape == (0, 2, 16)
