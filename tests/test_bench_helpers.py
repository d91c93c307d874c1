"""Host-side checks of bench.py's bookkeeping: workload overrides, the
backward's FLOP count and the per-kernel source hashes that tie a recorded
ncu capture to the code it was taken from."""
import argparse

import pytest
import torch

import bench


def _args(workload="train_bf16", batch=0, heads=0):
    return argparse.Namespace(workload=workload, batch=batch, heads=heads)


def test_workload_overrides_rename_the_workload():
    w = bench.selected_workload(_args())
    assert (w.name, w.B, w.H) == ("train_bf16", 8, 32)
    w = bench.selected_workload(_args(batch=19, heads=8))
    assert (w.B, w.H, w.T) == (19, 8, 8192)
    # a changed shape must not pick up the traffic recorded for the named workload
    assert w.name != "train_bf16"
    assert bench.traffic_from_profiles("kda_fwd_mma_kernel", w.name) == (None, None)
    with pytest.raises(SystemExit):
        bench.selected_workload(_args(workload="varlen_bf16", batch=2))


def test_backward_flop_count():
    # per token-head: 2 (9 d^2 + d^2 / 16 + 16 * 16 d + 2 * 16^2) at d = 128
    w = bench.selected_workload(_args(batch=1, heads=1))
    inp = {"lengths": [100]}
    assert bench.bwd_flops(w, inp) == 100 * 2 * (9 * 128 * 128 + 128 * 128 // 16
                                                + 16 * 16 * 128 + 2 * 16 * 16)
    assert bench.bwd_flops(w, inp) // 100 == 363520


def test_source_hash_is_per_kernel():
    # each known kernel hashes its own sources; an unknown name hashes every
    # CUDA source, so the two differ
    names = ["kda_fwd_mma_kernel", "kda_fwd_tc32_kernel", "kda_decode_kernel", "kda_bwd"]
    hashes = {n: bench.kernel_source_hash(n) for n in names}
    assert len(set(hashes.values())) == len(names)
    assert bench.kernel_source_hash("no_such_kernel") not in hashes.values()
    for n in names:
        assert len(hashes[n]) == 16 and hashes[n] == bench.kernel_source_hash(n)


def test_fp32_alu_peak_from_unit_counts():
    # 152 SMs x 128 fp32 lanes x 2 flop per FMA x 2070 MHz
    assert bench.FP32_ALU_TFLOPS == pytest.approx(80.54784)


def test_algorithmic_bytes_follow_the_scope_table():
    # 1282 B per token-head at d = 128 with out at the input's 2 B, plus the
    # fp32 final state; 1538 B with the fp32 output
    w = bench.selected_workload(_args())
    inp = {"lengths": [8192] * 8, "N": 8, "init_state": None}
    th = 8 * 8192 * 32
    state = 4 * 128 * 128 * 8 * 32
    assert bench.algorithmic_bytes(w, inp) == th * 1282 + state
    assert bench.algorithmic_bytes(w, inp, out_bytes=4) == th * 1538 + state
    assert bench.algorithmic_bytes(w, inp) == 2705326080
