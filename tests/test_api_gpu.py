"""GPU tests through the bare entry points and of the argument contract:

* kda_chunk_fwd (bf16) and kda_chunk_fwd_f32 called directly through ctypes
  with raw device pointers, against the fp64 oracle at their tolerances;
* the slow-decay regime (theta ~ N(-3, 1) on every channel: the state carries
  over many chunks) on the tcgen05 paths, and the register-resident path's
  measured limit there;
* a malformed cu_seqlens table whose offsets stay inside [0, T]: the kernels
  store nothing for the bad sequences, report KDA_ERR_BAD_SEQLENS through the
  device status word, and the next call on the same context is correct."""
import ctypes

import pytest
import torch

from linear_attention_04_gb300 import kda as binding
from linear_attention_04_gb300 import kda_chunk_fwd, kda_device_status
from linear_attention_04_gb300.workloads import WORKLOADS, Workload, make_inputs

from parity import TOL, assert_close, f64, oracle_full

pytestmark = pytest.mark.gpu


def _cuda(inp):
    return {k_: (x.cuda() if isinstance(x, torch.Tensor) else x) for k_, x in inp.items()}


def _bare(fn, g, out, fin, B, H, T, dk, dv):
    lib = binding.load()
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = getattr(lib, fn)(p(g["q"]), p(g["k"]), p(g["v"]), p(g["theta"]), p(g["beta"]),
                          ctypes.c_float(-5.0), p(g["init_state"]), p(out), p(fin),
                          p(g["cu_seqlens"]), B, H, T, dk, dv,
                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return rc


@pytest.mark.parametrize("name,fn", [("base_bf16", "kda_chunk_fwd"),
                                     ("tiny_f32", "kda_chunk_fwd_f32")])
def test_bare_entry_points_against_the_oracle(name, fn):
    w = WORKLOADS[name]
    inp = make_inputs(w)
    g = _cuda(inp)
    out = torch.empty((w.B, w.T, w.H, w.dv), dtype=torch.float32, device="cuda")
    fin = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device="cuda")
    assert kda_device_status(clear=True) == 0
    assert _bare(fn, g, out, fin, w.B, w.H, w.T, w.dk, w.dv) == binding.KDA_OK
    assert kda_device_status(clear=True) == 0
    ro, rS = oracle_full(inp)
    assert_close(f64(out), ro, TOL[w.dtype], f"{fn} out")
    assert_close(f64(fin), rS, TOL[w.dtype], f"{fn} final_state")


@pytest.mark.parametrize("path", ["tc", "tc_split"])
def test_slow_decay_regime(path):
    """theta ~ N(-3, 1): g ~ -0.25 per token, so the state remembers hundreds
    of tokens and U = U' - W S, O = Qt S + P U become differences of larger
    terms; the 2e-2 x RMS bar holds on the tcgen05 path, whose tf32 Gram tile
    and high/low chunk factors were chosen for this regime."""
    w = Workload("slow", B=2, H=3, T=2048, dk=128, dv=128, dtype=torch.bfloat16)
    inp = make_inputs(w, seed=2048)
    inp["theta"] = (inp["theta"].float() - 3.0).to(torch.bfloat16)
    g = _cuda(inp)
    o, S = kda_chunk_fwd(g["q"], g["k"], g["v"], g["theta"], g["beta"], -5.0, path=path)
    torch.cuda.synchronize()
    assert kda_device_status(clear=True) == 0
    ro, rS = oracle_full(inp)
    assert_close(f64(o), ro, TOL[torch.bfloat16], f"slow decay out ({path})")
    assert_close(f64(S), rS, TOL[torch.bfloat16], f"slow decay state ({path})")


@pytest.mark.parametrize("path", ["simt", "mma", "mma_tc", "tc"])
def test_malformed_cu_seqlens_reported_and_the_context_survives(path):
    lens = [40, 24, 32]
    w = Workload("badcu", B=3, H=2, T=0, dk=128, dv=128, dtype=torch.bfloat16, varlen=True)
    inp = make_inputs(w, seed=5, lengths=lens)
    g = _cuda(inp)
    T = sum(lens)
    cases = {
        # a decreasing pair (sequence 1 runs backwards), every offset inside [0, T]
        "decreasing": torch.tensor([0, 40, 20, T], dtype=torch.int32, device="cuda"),
        # the last offset is not the token count
        "short": torch.tensor([0, 40, 64, 80], dtype=torch.int32, device="cuda"),
        # a negative start
        "negative": torch.tensor([-16, 40, 64, T], dtype=torch.int32, device="cuda"),
    }
    for what, cu in cases.items():
        assert kda_device_status(clear=True) == 0
        out = torch.full((1, T, 2, 128), 7.0, device="cuda")
        fin = torch.full((3, 2, 128, 128), 7.0, device="cuda")
        kda_chunk_fwd(g["q"], g["k"], g["v"], g["theta"], g["beta"], -5.0, None, out, fin, cu,
                      path=path)
        torch.cuda.synchronize()
        assert kda_device_status(clear=True) == binding.KDA_ERR_BAD_SEQLENS, what
        if what == "decreasing":
            # sequence 1's blocks stored nothing: its state is untouched
            assert bool((fin[1] == 7.0).all()), what
        else:
            # the table's end points are wrong: no block stored anything
            assert bool((out == 7.0).all()) and bool((fin == 7.0).all()), what
    # the next call with a valid table runs normally
    ro, rS = oracle_full(inp)
    o, S = kda_chunk_fwd(g["q"], g["k"], g["v"], g["theta"], g["beta"], -5.0, None,
                         cu_seqlens=g["cu_seqlens"], path=path)
    torch.cuda.synchronize()
    assert kda_device_status(clear=True) == 0
    assert_close(f64(o), ro, TOL[torch.bfloat16], f"valid table after the bad ones ({path})")
    assert_close(f64(S), rS, TOL[torch.bfloat16], f"valid table state ({path})")


def test_slow_decay_limit_of_the_register_resident_path():
    """The register-resident path (all-bf16 operands, the default for speed)
    in the same regime: a measured limit, not a pass.  Its error exceeds the
    2e-2 bar here (about 3.4e-2 on this case; the library header names the
    regime and the tcgen05 path for it); guard that it stays finite and below
    5e-2."""
    w = Workload("slow", B=2, H=3, T=2048, dk=128, dv=128, dtype=torch.bfloat16)
    inp = make_inputs(w, seed=2048)
    inp["theta"] = (inp["theta"].float() - 3.0).to(torch.bfloat16)
    g = _cuda(inp)
    o, S = kda_chunk_fwd(g["q"], g["k"], g["v"], g["theta"], g["beta"], -5.0, path="mma")
    torch.cuda.synchronize()
    assert kda_device_status(clear=True) == 0
    ro, rS = oracle_full(inp)
    assert_close(f64(o), ro, 5e-2, "slow decay out (register-resident path)")
