"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on the
same seeded inputs.  Element-wise on sizes the oracle finishes in seconds,
sampled chains at the full workload sizes."""
import concurrent.futures as cf

import numpy as np
import pytest
import torch

from linear_attention_04_gb300 import kda_chunk_fwd, kda_device_status, kda_select_path
from linear_attention_04_gb300.workloads import WORKLOADS, Workload, make_inputs

from parity import TOL, assert_close, f64, oracle_chain, oracle_full

pytestmark = pytest.mark.gpu


def _paths(dtype, dk, dv):
    if dtype == torch.float32:
        return ["simt"]
    ps = ["simt"]
    if dk == 128 and dv == 128:
        ps += ["tc", "tc_split", "mma", "mma_tc"]
    return ps


def _bf16_paths():
    return _paths(torch.bfloat16, 128, 128)


def _to(inp, device):
    out = dict(inp)
    for k_ in ("q", "k", "v", "theta", "beta", "init_state", "cu_seqlens"):
        if out[k_] is not None:
            out[k_] = out[k_].to(device)
    return out


def _run(inp, path, want_state=True):
    o, S = kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["theta"], inp["beta"], -5.0,
                         inp["init_state"], cu_seqlens=inp["cu_seqlens"],
                         want_final_state=want_state, path=path)
    torch.cuda.synchronize()
    assert kda_device_status(clear=True) == 0
    return o, S


def _check_full(w, inp_cpu, path, tol=None):
    tol = TOL[w.dtype] if tol is None else tol
    ref_o, ref_S = oracle_full(inp_cpu)
    inp = _to(inp_cpu, "cuda")
    o, S = _run(inp, path)
    eo = assert_close(f64(o), ref_o, tol, f"{w.name}/{path} out")
    es = assert_close(f64(S), ref_S, tol, f"{w.name}/{path} final_state")
    return eo, es


# ---------------------------------------------------------------- named configs

def test_tiny_f32_full():
    w = WORKLOADS["tiny_f32"]
    _check_full(w, make_inputs(w), "simt")


@pytest.mark.parametrize("path", _bf16_paths())
def test_base_bf16_full(path):
    w = WORKLOADS["base_bf16"]
    _check_full(w, make_inputs(w), path)


def _sampled(w, path, chains, seed=None):
    inp = make_inputs(w, seed=seed, device="cuda")
    o, S = _run(inp, path)
    with cf.ThreadPoolExecutor(max_workers=len(chains)) as ex:
        refs = list(ex.map(lambda c: oracle_chain(inp, *c), chains))
    tol = TOL[w.dtype]
    for (seq, head), (ro, rS, (b, t0, t1)) in zip(chains, refs):
        assert_close(f64(o[b, t0:t1, head]), ro, tol, f"{w.name}/{path} out seq{seq} h{head}")
        assert_close(f64(S[seq, head]), rS, tol, f"{w.name}/{path} state seq{seq} h{head}")
    return inp, o, S


# chains (index = sequence * H + head) spread over the 256: under the wrapped
# schedule (152 windows of 863 chunk-steps) chains 37, 75, 151, 170, 230 and
# 247 are cut by a window boundary and hand their state from one CTA to
# another, the others run whole; in a one-chain-per-CTA launch they fall in the
# first wave (0..151) and the second (152..255)
TRAIN_RANKS = [0, 37, 75, 118, 151, 152, 170, 199, 213, 230, 247, 255]


@pytest.mark.parametrize("path", _bf16_paths())
def test_train_bf16_sampled(path):
    w = WORKLOADS["train_bf16"]
    _sampled(w, path, [(r // w.H, r % w.H) for r in TRAIN_RANKS])


@pytest.mark.parametrize("path", _bf16_paths())
def test_long_bf16_sampled(path):
    w = WORKLOADS["long_bf16"]
    _sampled(w, path, [(0, 0), (0, 11), (0, 21), (0, 31)])


@pytest.mark.parametrize("path", _bf16_paths())
def test_varlen_bf16_sampled(path):
    w = WORKLOADS["varlen_bf16"]
    inp = make_inputs(w, device="cpu")
    lens = inp["lengths"]
    # sequences by rank in the longest-first launch order (ties by index), on
    # different heads: the longest, the shortest and ranks in between, so that
    # CTAs of the first, middle and last waves are checked
    order = sorted(range(len(lens)), key=lambda i: (-lens[i], i))
    ranks = [0, 3, 10, 21, 32, 44, 55, 63]
    chains = [(int(order[r]), (5 * j) % w.H) for j, r in enumerate(ranks)]
    _sampled(w, path, chains)


# ---------------------------------------------------------------- edge cases

def _custom(B=1, H=2, T=64, dk=128, dv=128, dtype=torch.bfloat16, init=0.0, theta="normal",
            beta="sigmoid_normal", seed=5):
    w = Workload("custom", B=B, H=H, T=T, dk=dk, dv=dv, dtype=dtype, init_std=init, theta=theta,
                 beta=beta)
    return w, make_inputs(w, seed=seed)


@pytest.mark.parametrize("T", [1, 15, 16, 17, 37, 100])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_ragged_lengths(T, dtype):
    w, inp = _custom(B=2, H=3, T=T, dtype=dtype, init=0.3, seed=T)
    for path in _paths(dtype, 128, 128):
        _check_full(w, inp, path)


@pytest.mark.parametrize("dk,dv", [(16, 16), (32, 64), (64, 32), (128, 64), (64, 128)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_head_dims(dk, dv, dtype):
    w, inp = _custom(B=1, H=2, T=50, dk=dk, dv=dv, dtype=dtype, init=0.2, seed=dk + dv)
    for path in _paths(dtype, dk, dv):
        _check_full(w, inp, path)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_varlen_edge_lengths(dtype):
    lens = [0, 1, 16, 17, 45, 3, 0, 64]
    w = Workload("custom_varlen", B=len(lens), H=2, T=0, dk=128, dv=128, dtype=dtype,
                 init_std=0.25, varlen=True)
    inp = make_inputs(w, seed=9, lengths=lens)
    for path in _paths(dtype, 128, 128):
        _check_full(w, inp, path)
        # zero-length sequences return their initial state untouched
        o, S = _run(_to(inp, "cuda"), path)
        assert torch.equal(S[0].cpu(), inp["init_state"][0])
        assert torch.equal(S[6].cpu(), inp["init_state"][6])


@pytest.mark.parametrize("path", _bf16_paths())
def test_decay_stress_small(path):
    """theta ~ U[6,12]: every log-decay within 0.01 of g_min, so the in-chunk
    inverse factor reaches about e^{80} (the bound the pages rely on)."""
    w, inp = _custom(B=1, H=4, T=160, theta="uniform6_12", beta="uniform09_1", seed=77)
    _check_full(w, inp, path)


@pytest.mark.parametrize("path", _bf16_paths())
def test_null_states_and_continuation(path):
    w, inp = _custom(B=2, H=2, T=96, init=0.0, seed=31)
    g = _to(inp, "cuda")
    o_full, S_full = _run(g, path)
    # no state requested
    o2, S2 = kda_chunk_fwd(g["q"], g["k"], g["v"], g["theta"], g["beta"], -5.0, None,
                           want_final_state=False, path=path)
    torch.cuda.synchronize()
    assert S2 is None and torch.equal(o2, o_full)
    # split at a chunk boundary and at a ragged point: continuation from the GPU state
    for T1 in (48, 41):
        a = {k_: (x[:, :T1].contiguous() if k_ in ("q", "k", "v", "theta", "beta") else x)
             for k_, x in g.items()}
        b = {k_: (x[:, T1:].contiguous() if k_ in ("q", "k", "v", "theta", "beta") else x)
             for k_, x in g.items()}
        a["T"], b["T"] = T1, 96 - T1
        oa, Sa = _run(a, path)
        b["init_state"] = Sa
        ob, Sb = _run(b, path)
        tol = TOL[torch.bfloat16]
        assert_close(f64(torch.cat([oa, ob], 1)), f64(o_full), tol, "continuation out")
        assert_close(f64(Sb), f64(S_full), tol, "continuation state")


@pytest.mark.parametrize("path", _bf16_paths())
def test_bf16_output_option(path):
    """bf16 out (opt-in): equal to the fp32-out result rounded to bf16 up to one
    bf16 ulp, and within 2e-2 RMS + one bf16 ulp of |o| of the oracle."""
    w, inp = _custom(B=1, H=3, T=70, init=0.2, seed=8)
    g = _to(inp, "cuda")
    o32, _ = _run(g, path)
    o16, _ = kda_chunk_fwd(g["q"], g["k"], g["v"], g["theta"], g["beta"], -5.0, g["init_state"],
                           out_dtype=torch.bfloat16, path=path)
    torch.cuda.synchronize()
    assert o16.dtype == torch.bfloat16
    ref_o, _ = oracle_full(inp)
    got = f64(o16)
    ulp = np.abs(ref_o) * 2.0 ** -8
    rms = float(np.sqrt(np.mean(ref_o ** 2)))
    assert np.all(np.abs(got - ref_o) <= 2e-2 * rms + ulp)
    assert np.all(np.abs(got - f64(o32)) <= np.abs(f64(o32)) * 2.0 ** -8 + 1e-30)


def test_empty_sequence_batch():
    w, inp = _custom(B=2, H=2, T=0, init=0.5, seed=3)
    g = _to(inp, "cuda")
    o, S = _run(g, "auto")
    assert o.numel() == 0
    assert torch.equal(S.cpu(), inp["init_state"])


def test_wrong_device_kind_rejected():
    w, inp = _custom(B=1, H=1, T=16, seed=4)
    with pytest.raises(ValueError):
        kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["theta"], inp["beta"])  # CPU tensors
