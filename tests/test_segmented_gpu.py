"""GPU parity of the segment-parallel forward (kda_chunk_fwd_segmented): the
same outputs and final state as the fp64 oracle, for several segment counts,
ragged lengths and a nonzero initial state; the long workload on sampled
chains."""
import pytest
import torch

from linear_attention_04_gb300 import (kda_chunk_fwd, kda_chunk_fwd_segmented, kda_device_status,
                                       kda_segmented_workspace_size)
from linear_attention_04_gb300.workloads import WORKLOADS, Workload, make_inputs

from parity import TOL, assert_close, f64, oracle_chain, oracle_full

pytestmark = pytest.mark.gpu
TOL_BF16 = TOL[torch.bfloat16]


def _cuda(inp):
    return {k_: (x.cuda() if isinstance(x, torch.Tensor) else x) for k_, x in inp.items()}


@pytest.mark.parametrize("T,segments", [(3000, 2), (3000, 3), (4096, 5), (1000, 8), (40, 4)])
def test_segmented_vs_oracle(T, segments):
    w = Workload("seg", B=2, H=3, T=T, dk=128, dv=128, dtype=torch.bfloat16, init_std=0.05)
    inp = make_inputs(w, seed=1000 + T + segments)
    g = _cuda(inp)
    ref_o, ref_S = oracle_full(inp)
    o, S = kda_chunk_fwd_segmented(g["q"], g["k"], g["v"], g["theta"], g["beta"], -5.0,
                                   g["init_state"], segments=segments)
    torch.cuda.synchronize()
    assert kda_device_status(clear=True) == 0
    assert_close(f64(o), ref_o, TOL_BF16, f"segmented out T={T} P={segments}")
    assert_close(f64(S), ref_S, TOL_BF16, f"segmented final state T={T} P={segments}")


@pytest.mark.parametrize("path", ["mma", "tc"])
def test_segmented_longer_first_segment(path):
    # 32 chains, P = 5 on 152 SMs: launch 1 holds 32 + 192 jobs, so the plan
    # makes segment 0 twice as long as the others (it runs beside the first
    # wave of the short jobs); every chain against the oracle
    w = Workload("seg", B=1, H=32, T=2048, dk=128, dv=128, dtype=torch.bfloat16, init_std=0.05)
    inp = make_inputs(w, seed=1077)
    g = _cuda(inp)
    ref_o, ref_S = oracle_full(inp)
    o, S = kda_chunk_fwd_segmented(g["q"], g["k"], g["v"], g["theta"], g["beta"], -5.0,
                                   g["init_state"], segments=5, path=path)
    torch.cuda.synchronize()
    assert kda_device_status(clear=True) == 0
    assert_close(f64(o), ref_o, TOL_BF16, f"segmented out, longer first segment ({path})")
    assert_close(f64(S), ref_S, TOL_BF16, f"segmented final state, longer first segment ({path})")


def test_segmented_slow_channels_carry_state_across_segments():
    # 16 key channels with theta shifted by -12 (g ~ -3e-5 per token) carry the
    # state across every segment boundary, so Phi and the chaining matter; the
    # other channels keep the recipe's decay
    w = Workload("seg", B=1, H=2, T=2048, dk=128, dv=128, dtype=torch.bfloat16)
    inp = make_inputs(w, seed=4242)
    th = inp["theta"].float()
    th[..., :16] -= 12.0
    inp["theta"] = th.to(torch.bfloat16)
    g = _cuda(inp)
    ref_o, ref_S = oracle_full(inp)
    o, S = kda_chunk_fwd_segmented(g["q"], g["k"], g["v"], g["theta"], g["beta"], -5.0,
                                   segments=4)
    torch.cuda.synchronize()
    assert_close(f64(o), ref_o, TOL_BF16, "segmented out, slow channels")
    assert_close(f64(S), ref_S, TOL_BF16, "segmented state, slow channels")


def test_segmented_matches_plain_path_and_reuses_workspace():
    w = Workload("seg", B=1, H=4, T=2000, dk=128, dv=128, dtype=torch.bfloat16, init_std=0.02)
    g = _cuda(make_inputs(w, seed=77))
    args = (g["q"], g["k"], g["v"], g["theta"], g["beta"], -5.0, g["init_state"])
    ws = torch.empty(kda_segmented_workspace_size(1, 4, 2000, 128, 128, 3), dtype=torch.uint8,
                     device="cuda")
    o1, S1 = kda_chunk_fwd_segmented(*args, segments=3, workspace=ws)
    o2, S2 = kda_chunk_fwd_segmented(*args, segments=3, workspace=ws)
    op, Sp = kda_chunk_fwd(*args, path="mma")
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(S1, S2)
    assert_close(f64(o1), f64(op), TOL_BF16, "segmented vs plain out")
    assert_close(f64(S1), f64(Sp), TOL_BF16, "segmented vs plain state")


def test_segmented_long_workload_sampled():
    w = WORKLOADS["long_bf16"]
    inp = make_inputs(w, device="cuda")
    o, S = kda_chunk_fwd_segmented(inp["q"], inp["k"], inp["v"], inp["theta"], inp["beta"],
                                   w.g_min, inp["init_state"], segments=4)
    torch.cuda.synchronize()
    assert kda_device_status(clear=True) == 0
    ro, rS, (b, t0, t1) = oracle_chain(inp, 0, 21)
    assert_close(f64(o[b, t0:t1, 21]), ro, TOL_BF16, "long segmented out h21")
    assert_close(f64(S[0, 21]), rS, TOL_BF16, "long segmented state h21")
