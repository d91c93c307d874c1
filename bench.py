#!/usr/bin/env python
"""Benchmark of the KDA chunked forward pass (one JSON line on stdout).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one forward pass over the whole workload (every (sequence, head)
chain: gate, in-chunk cumulative sum, decayed Gram tiles, triangular inverse,
WY factors, state read-out and update, outputs and final state).  Default
workload: B=8, H=32, T=8192, dk=dv=128, bf16 inputs, fp32 state.

Multi-GPU (torchrun, one rank per GPU): weak scaling.  Every rank owns its
own shard of B sequences (the global batch is B * world), no data-path
collective; the only collectives are the barrier and the max-over-ranks of
the timed interval.

--impl reference times the fp64 CPU oracle on the host cores instead (rank 0
only), each step a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import glob
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from linear_attention_04_gb300.workloads import WORKLOADS, Workload, make_inputs  # noqa: E402

METRIC = "KDA fwd tokens/s at B8 H32 T8K d128; % of bf16 tensor peak and HBM GB/s"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
CHUNK = 16


# ----------------------------------------------------------------------------- accounting

def token_heads(w: Workload, inp: dict) -> int:
    return int(sum(inp["lengths"])) * w.H


def n_tokens(inp: dict) -> int:
    return int(sum(inp["lengths"]))


def algorithmic_bytes(w: Workload, inp: dict, out_bytes: int | None = None) -> int:
    """Minimum HBM bytes of one pass: q, k, theta, v, beta read and out written
    (e*(3dk+dv) + e + e_out*dv per token-head), plus the fp32 final state
    written and the fp32 initial state read when given (4*dk*dv per chain
    each).  e_out defaults to the input element size e (the counting rule of
    the scope table: 1282 B per token-head for bf16 at d = 128); pass 4 for
    the bytes of the fp32 output the library writes by default (1538 B)."""
    e = torch.tensor([], dtype=w.dtype).element_size()
    per = e * (3 * w.dk + w.dv) + e + (e if out_bytes is None else out_bytes) * w.dv
    chains = inp["N"] * w.H
    state = 4 * w.dk * w.dv * chains
    return token_heads(w, inp) * per + state * (2 if inp["init_state"] is not None else 1)


def chunk_gemm_flops(w: Workload, inp: dict) -> int:
    """6*dk*dv + 2C(3dk + 2dv) per token-head: A, P, W, U', P.U, W.S, Qt.S and
    KhC^T.U (the triangular inverse and padding not counted)."""
    return token_heads(w, inp) * (6 * w.dk * w.dv + 2 * CHUNK * (3 * w.dk + 2 * w.dv))


def measured_peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS,
            "bf16_tflops_sustained": 1700.0}, "fallback"


# The files each profiled kernel is compiled from (its translation unit and the
# headers it includes); other kernels' sources do not invalidate its capture.
KERNEL_SOURCES = {
    "kda_fwd_mma_kernel": ["csrc/kda_mma.cu", "csrc/kda_tmap.cu", "csrc/kda_sm100.cuh",
                           "csrc/kda_device.cuh", "csrc/kda_internal.cuh"],
    "kda_fwd_tc32_kernel": ["csrc/kda_tc32.cu", "csrc/kda_tmap.cu", "csrc/kda_sm100.cuh",
                            "csrc/kda_device.cuh", "csrc/kda_internal.cuh"],
    "kda_decode_kernel": ["csrc/kda_decode.cu", "csrc/kda_device.cuh", "csrc/kda_internal.cuh"],
    "kda_bwd": ["csrc/kda_bwd.cu", "csrc/kda_device.cuh", "csrc/kda_internal.cuh"],
}


def kernel_source_hash(kernel: str = "") -> str:
    """Hash of the sources of `kernel` (every CUDA source for an unknown name)."""
    pkg = os.path.join(ROOT, "linear_attention_04_gb300")
    files = KERNEL_SOURCES.get(kernel)
    paths = ([os.path.join(pkg, f) for f in files] if files else
             glob.glob(os.path.join(pkg, "csrc", "*")))
    h = hashlib.sha256()
    for f in sorted(paths):
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_from_profiles(kernel: str, workload: str) -> tuple[int | None, str | None]:
    """DRAM bytes per launch recorded from an ncu capture under profiles/, if
    the kernel sources still hash to the value recorded with it."""
    want = kernel_source_hash(kernel)
    for f in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.txt")) +
                    glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        kv = {}
        with open(f) as fh:
            for line in fh:
                line = line.strip().lstrip("-* ")
                if ":" in line:
                    a, b = line.split(":", 1)
                    kv[a.strip()] = b.strip()
        if kv.get("traffic_kernel") == kernel and kv.get("traffic_workload") == workload:
            if kv.get("source_hash") == want and kv.get("dram_bytes_per_launch"):
                return int(float(kv["dram_bytes_per_launch"])), os.path.basename(f)
    return None, None


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampled every 50 ms in the background; keeps timestamps."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        self.gpu_id = gpu_id
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", self.gpu_id],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        if not inside and self.samples:
            # the timed region was shorter than the sampling period: nearest samples
            mid = 0.5 * (t0 + t1)
            inside = [min(self.samples, key=lambda s: abs(s[0] - mid))[1]]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for p in inside if num(p[1]) is not None]
        smax = [num(p[2]) for p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for p in inside for i in range(4)
                          if p[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(inside),
                "power_w_max": max((num(p[3]) or 0.0) for p in inside)}


# ----------------------------------------------------------------------------- distributed

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def shard_sequences(n_per_rank: int, world: int, rank: int) -> range:
    """Global sequence indices owned by `rank` under weak scaling."""
    return range(rank * n_per_rank, (rank + 1) * n_per_rank)


def rank_seed(base: int, rank: int) -> int:
    return base + 1000 * rank


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- CPU oracle

def oracle_sample_inputs(w: Workload, n_chains: int, n_tok: int, seed: int) -> dict:
    """A bounded sample of the workload for the CPU oracle: n_chains chains of
    n_tok tokens each, drawn with the same recipe (on the host)."""
    n_chains = max(1, n_chains)
    sw = Workload(w.name + "_sample", B=n_chains, H=1, T=n_tok, dk=w.dk, dv=w.dv, dtype=w.dtype,
                  theta=w.theta, beta=w.beta, init_std=w.init_std)
    return make_inputs(sw, seed=seed)


def time_oracle(inp: dict, threads: int) -> float:
    import oracle  # CPU-baseline leg only

    def f64(t):
        return None if t is None else t.to(torch.float64).numpy()

    t0 = time.perf_counter()
    oracle.fwd(f64(inp["q"]), f64(inp["k"]), f64(inp["v"]), f64(inp["theta"]), f64(inp["beta"]),
               -5.0, f64(inp["init_state"]), nthreads=threads)
    return time.perf_counter() - t0


def cpu_baseline(w: Workload, target_s: float, seed: int) -> dict:
    """The oracle as it stands on the host cores, on a bounded sample sized to
    about target_s seconds; value converted to tokens/s of the workload's H."""
    import oracle
    oracle.build()
    threads = oracle.host_threads()
    n_tok = 1024
    probe = oracle_sample_inputs(w, threads, n_tok, seed)
    dt = time_oracle(probe, threads)
    rate = threads * n_tok / max(dt, 1e-6)  # token-heads/s
    n_chains = max(threads, int(round(rate * target_s / (2 * n_tok) / threads)) * threads)
    inp = oracle_sample_inputs(w, n_chains, 2 * n_tok, seed + 1)
    dt = time_oracle(inp, threads)
    th = n_chains * 2 * n_tok
    return {"value": th / dt / w.H, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{n_chains} (sequence, head) chains x {2 * n_tok} tokens of the "
                      f"{w.name} recipe (dk={w.dk}, dv={w.dv}), fp64, {threads} threads; "
                      f"{th} token-heads in {dt:.2f} s, converted at H={w.H} heads per token"}


# ----------------------------------------------------------------------------- our arm

def selected_workload(args):
    """The named workload, with B and H replaced when --batch / --heads are
    given (profiling cases of the same shape per sequence)."""
    w = WORKLOADS[args.workload]
    if args.batch or args.heads:
        if w.varlen:
            raise SystemExit("--batch and --heads apply to fixed-length workloads only")
        B, H = args.batch or w.B, args.heads or w.H
        # a new name: captures recorded for the named workload do not apply
        w = dataclasses.replace(w, B=B, H=H, name=f"{w.name}-B{B}-H{H}")
    return w


def run_ours(args, rank, world, local):
    from linear_attention_04_gb300 import kda_chunk_fwd, kda_device_status, kda_select_path

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = selected_workload(args)
    inp = make_inputs(w, seed=rank_seed(args.seed, rank), device=dev)
    q, k, v, th, be = inp["q"], inp["k"], inp["v"], inp["theta"], inp["beta"]
    init, cu = inp["init_state"], inp["cu_seqlens"]
    path = args.path if args.path != "auto" else kda_select_path(w.dtype, w.dk, w.dv)
    gate = getattr(args, "gate", "sigmoid")
    if gate == "log_decay":
        # the unbounded log-decay g = -softplus(logit), drawn before timing
        th = (-torch.nn.functional.softplus(th.float() + args.logit_mu)).to(th.dtype)
    out = torch.empty((q.shape[0], q.shape[1], w.H, w.dv), dtype=torch.float32, device=dev)
    fin = torch.empty((inp["N"], w.H, w.dk, w.dv), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    ws = None
    if args.segments > 1:
        from linear_attention_04_gb300 import kda_chunk_fwd_segmented, kda_segmented_workspace_size
        ws = torch.empty(kda_segmented_workspace_size(w.B, w.H, w.T, w.dk, w.dv, args.segments),
                         dtype=torch.uint8, device=dev)
        seg_kernel = "mma" if path == "mma" else path
        path = f"segmented x{args.segments} ({seg_kernel})"

    def step():
        if ws is not None:
            kda_chunk_fwd_segmented(q, k, v, th, be, w.g_min, init, out, fin,
                                    segments=args.segments, workspace=ws, path=seg_kernel,
                                    stream=stream)
        else:
            kda_chunk_fwd(q, k, v, th, be, w.g_min, init, out, fin, cu, path=path, gate=gate,
                          stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    status = kda_device_status(clear=True)
    if status != 0:
        raise RuntimeError(f"device status {status} after warm-up")

    gpu_id = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    gpu_id = str(gpu_id) if gpu_id is not None else str(local)
    if gpu_id and not gpu_id.startswith("GPU-") and len(gpu_id) == 36:
        gpu_id = "GPU-" + gpu_id
    clocks = ClockSampler(gpu_id).start()
    time.sleep(0.3)

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t_wall1 = time.time()
    time.sleep(0.25)
    clocks.stop()
    total_ms = start.elapsed_time(end)
    launch_ms = [a.elapsed_time(b) for a, b in evs]
    total_ms = max_over_ranks(total_ms, world)
    status = kda_device_status(clear=True)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed steps")

    tokens = n_tokens(inp)
    value = tokens * world * args.steps / (total_ms / 1e3)
    ms_per_step = total_ms / args.steps
    avg_launch_s = statistics.mean(launch_ms) / 1e3
    peaks, peak_src = measured_peaks()
    alg = algorithmic_bytes(w, inp)                  # out counted at the input's element size
    alg32 = algorithmic_bytes(w, inp, out_bytes=4)   # out counted as the fp32 the kernel writes
    flops = chunk_gemm_flops(w, inp)
    achieved = alg / avg_launch_s / 1e9
    achieved32 = alg32 / avg_launch_s / 1e9
    kernels = {"tc": "kda_fwd_tc32_kernel", "tc_split": "kda_fwd_tc32_kernel",
               "mma": "kda_fwd_mma_kernel", "mma_tc": "kda_fwd_mma_kernel"}
    kname = kernels.get(path, "kda_fwd_simt_kernel")
    if ws is not None:
        kname = kernels.get(seg_kernel, "kda_fwd_tc32_kernel")
    traffic, traffic_src = traffic_from_profiles(kname, w.name)
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
            "traffic": traffic, "peak_source": f"hbm_gbs of {peak_src}",
            "kernel": kname, "algorithmic_bytes_per_launch": alg,
            "bytes_counted": "q, k, theta, v, beta read and out written at the input element "
                             "size (2 B for bf16) plus the fp32 final state",
            "fp32_out": {"achieved": round(achieved32, 1),
                         "frac": round(achieved32 / peaks["hbm_gbs"], 4),
                         "algorithmic_bytes_per_launch": alg32,
                         "bytes_counted": "as above with out at 4 B (the fp32 output the "
                                          "kernel writes)"},
            "tensor": {"achieved_tflops": round(flops / avg_launch_s / 1e12, 2),
                       "peak_tflops": peaks["bf16_tflops"],
                       "frac": round(flops / avg_launch_s / 1e12 / peaks["bf16_tflops"], 4),
                       "flops_per_launch": flops}}
    if traffic_src:
        roof["traffic_source"] = traffic_src

    # ---- end to end: pinned host buffers in, result back out, every step.
    # Steps are pipelined the way a caller streaming batches would run them:
    # the host-to-device copy of step n+1, the kernel of step n and the
    # device-to-host copy of step n-1 run on three streams at once, over two
    # sets of device buffers.  Every step's copies lie inside the timed region.
    # (Splitting the upload over two streams measured the same: 11.95 ms per
    # step on train_bf16, bound by the host link.)
    e2e = None
    if not args.no_e2e:
        hq, hk, hv, hth, hbe = (x.cpu().pin_memory() for x in (q, k, v, th, be))
        hinit = init.cpu().pin_memory() if init is not None else None
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        hfin = torch.empty(fin.shape, dtype=fin.dtype).pin_memory()
        h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv, hth, hbe)) + \
            (hinit.numel() * 4 if hinit is not None else 0)
        d2h = hout.numel() * hout.element_size() + hfin.numel() * 4
        sets = []
        for _ in range(2):
            dev_in = [torch.empty_like(x) for x in (q, k, v, th, be)]
            dev_init = torch.empty_like(init) if init is not None else None
            sets.append({"in": dev_in, "init": dev_init, "out": torch.empty_like(out),
                         "fin": torch.empty_like(fin),
                         "h2d": torch.cuda.Event(), "cmp": torch.cuda.Event(),
                         "d2h": torch.cuda.Event(), "used": False})
        s_h2d, s_d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def e2e_step(i):
            b = sets[i % 2]
            with torch.cuda.stream(s_h2d):
                if b["used"]:
                    s_h2d.wait_event(b["cmp"])  # the kernel of step i-2 has read these inputs
                for d, h in zip(b["in"], (hq, hk, hv, hth, hbe)):
                    d.copy_(h, non_blocking=True)
                if b["init"] is not None:
                    b["init"].copy_(hinit, non_blocking=True)
                b["h2d"].record(s_h2d)
            stream.wait_event(b["h2d"])
            if b["used"]:
                stream.wait_event(b["d2h"])  # step i-2's outputs have left these buffers
            dq, dk_, dv_, dth, dbe = b["in"]
            if ws is not None:
                kda_chunk_fwd_segmented(dq, dk_, dv_, dth, dbe, w.g_min, b["init"], b["out"],
                                        b["fin"], segments=args.segments, workspace=ws,
                                        path=seg_kernel, stream=stream)
            else:
                kda_chunk_fwd(dq, dk_, dv_, dth, dbe, w.g_min, b["init"], b["out"], b["fin"], cu,
                              path=path, gate=gate, stream=stream)
            b["cmp"].record(stream)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(b["cmp"])
                hout.copy_(b["out"], non_blocking=True)
                hfin.copy_(b["fin"], non_blocking=True)
                b["d2h"].record(s_d2h)
            b["used"] = True

        for i in range(max(1, args.warmup)):
            e2e_step(i)
        torch.cuda.synchronize()
        n_e2e = max(3, min(args.steps, 10))
        barrier(world)
        torch.cuda.synchronize()
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s2.record(s_h2d)
        for i in range(n_e2e):
            e2e_step(i)
        for st in (stream, s_h2d):
            s_d2h.wait_stream(st)
        e2.record(s_d2h)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(s2.elapsed_time(e2), world)
        barrier(world)
        e2e = {"value": tokens * world * n_e2e / (e2e_ms / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "ms_per_step": round(e2e_ms / n_e2e, 3),
               "pipelining": "host-to-device copy, kernel and device-to-host copy of "
                             "consecutive steps overlap on three streams (two buffer sets)"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_seconds, args.seed + 17)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16"
            if w.dtype == torch.bfloat16 else "f32", "data": "synthetic",
            "out_dtype": "f32", "state_dtype": "f32",
            "config": {"workload": f"{w.name}: B={w.B} H={w.H} T={w.T} dk={w.dk} dv={w.dv}, "
                                   f"chunk 16, g_min={w.g_min}, fp32 state" +
                                   ("" if gate == "sigmoid" else
                                    f", log-decay gate g = -softplus(theta + {args.logit_mu})"),
                       "B_per_gpu": w.B, "H": w.H, "T": w.T, "dk": w.dk, "dv": w.dv,
                       "global_batch": w.B * world, "parallelism": f"sequence-shard x{world}",
                       "path": path, "seed": args.seed,
                       "l2": "inputs larger than L2 (no flush): "
                             f"{alg32 / 1e9:.2f} GB per step vs 126 MB L2"},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": args.steps,
            "clocks": clocks.summary(t_wall0, t_wall1),
            "kernel_ms": {"mean": round(statistics.mean(launch_ms), 4),
                          "min": round(min(launch_ms), 4), "max": round(max(launch_ms), 4)}}
    return line


# ----------------------------------------------------------------------------- reference arm

def run_reference(args, rank, world):
    import oracle
    w = selected_workload(args)
    oracle.build()
    threads = oracle.host_threads()
    # size one step's sample to about args.ref_step_seconds of oracle work
    n_tok = 1024
    probe = oracle_sample_inputs(w, threads, n_tok, args.seed)
    dt = time_oracle(probe, threads)
    rate = threads * n_tok / max(dt, 1e-6)
    n_chains = max(threads, int(round(rate * args.ref_step_seconds / n_tok / threads)) * threads)
    inp = oracle_sample_inputs(w, n_chains, n_tok, args.seed + 1)
    for _ in range(args.warmup):
        time_oracle(inp, threads)
    times = [time_oracle(inp, threads) for _ in range(args.steps)]
    th = n_chains * n_tok
    total = sum(times)
    value = th * args.steps / total / w.H
    sample = (f"{n_chains} (sequence, head) chains x {n_tok} tokens of the {w.name} recipe per "
              f"step, fp64 oracle, {threads} threads, converted at H={w.H} heads per token")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * total / args.steps, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{w.name}: B={w.B} H={w.H} T={w.T} dk={w.dk} dv={w.dv}, "
                                   f"chunk 16, g_min={w.g_min} (bounded sample per step)",
                       "sample": sample},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


# ----------------------------------------------------------------------------- main

# ----------------------------------------------------------------------------- decode step

DECODE = dict(N=128, H=32, d=128)  # serving-sized batch: 128 sequences x 32 heads, d = 128


def decode_bytes(N, H, dk, dv, e=2) -> int:
    """HBM bytes of one decode step: the fp32 state read and written, the
    token's q, k, theta, v, beta and the fp32 output."""
    return N * H * (2 * 4 * dk * dv + e * (3 * dk + dv) + e + 4 * dv)


def run_decode(args, rank, world, local):
    from linear_attention_04_gb300 import kda_decode_step, kda_device_status

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    N, H, d = DECODE["N"], DECODE["H"], DECODE["d"]
    g = torch.Generator(device="cpu").manual_seed(rank_seed(args.seed, rank))
    q = torch.nn.functional.normalize(torch.randn(N, H, d, generator=g), dim=-1)
    k = torch.nn.functional.normalize(torch.randn(N, H, d, generator=g), dim=-1)
    v = torch.randn(N, H, d, generator=g)
    th = torch.randn(N, H, d, generator=g)
    be = torch.sigmoid(torch.randn(N, H, generator=g))
    q, k, v, th, be = (x.to(dev, torch.bfloat16) for x in (q, k, v, th, be))
    state = (0.02 * torch.randn(N, H, d, d, generator=g)).to(dev)
    out = torch.empty((N, H, d), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kda_decode_step(q, k, v, th, be, state, -5.0, out, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if kda_device_status(clear=True) != 0:
        raise RuntimeError("device status after warm-up")
    gpu_id = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    gpu_id = str(gpu_id) if gpu_id is not None else str(local)
    if gpu_id and not gpu_id.startswith("GPU-") and len(gpu_id) == 36:
        gpu_id = "GPU-" + gpu_id
    clocks = ClockSampler(gpu_id).start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(args.steps):
        step()
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t_wall1 = time.time()
    time.sleep(0.25)
    clocks.stop()
    total_ms = max_over_ranks(start.elapsed_time(end), world)
    step_s = total_ms / args.steps / 1e3
    peaks, peak_src = measured_peaks()
    nbytes = decode_bytes(N, H, d, d)
    achieved = nbytes / step_s / 1e9
    return {"metric": "KDA decode tokens/s: one token per sequence against a resident fp32 "
                      "state, N=128 sequences x H=32 heads, d=128",
            "value": N * world / step_s, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "op": "decode",
            "config": {"workload": f"decode: N={N} H={H} d={d}, bf16 token inputs, fp32 state",
                       "l2": f"state {N * H * d * d * 4 / 1e6:.0f} MB per step vs 126 MB L2"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                         "traffic": None, "peak_source": f"hbm_gbs of {peak_src}",
                         "kernel": "kda_decode_kernel", "algorithmic_bytes_per_launch": nbytes},
            "cpu_baseline": None, "e2e": None, "gpu_launches": args.steps,
            "clocks": clocks.summary(t_wall0, t_wall1)}


# ----------------------------------------------------------------------------- backward

# fp32 CUDA-core peak of one GB300: 152 SMs x 128 fp32 FMA lanes x 2 flop x 2070 MHz
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12


def bwd_flops(w, inp, C=16) -> int:
    """Algorithmic FLOPs of one chunked backward pass: per token-head
    2 (9 d^2 + d^2 / C + 16 C d + 2 C^2) at d = dk = dv -- the chunk products of
    the forward recurrence (Kt S, KhC^T U and the 16 x 16 products), the reverse
    recurrence (KhC dS', [Qt; -Kt]^T [dO; dR] and the 16 x 16 products) and the
    per-chunk gradient kernel (Kt S, [dO; -dR] S^T, U dS'^T, dS' * S and the
    16 x 16 products)."""
    d = w.dk
    n = n_tokens(inp) * w.H
    return n * 2 * (9 * d * d + d * d // C + 16 * C * d + 2 * C * C)


def bwd_bytes(w, inp, e=2) -> int:
    """HBM bytes of one backward pass (token-heads x per-token-head bytes): the
    bf16 inputs, the fp32 d_out, the fp32 gradients dq, dk, dtheta, dv, dbeta."""
    n = n_tokens(inp) * w.H
    return n * (e * (3 * w.dk + w.dv) + e + 4 * w.dv + 4 * (3 * w.dk + w.dv) + 4)


# kda_chunk_bwd clears its work queue and launches one persistent kernel
BWD_LAUNCHES_PER_PASS = 1


def run_bwd(args, rank, world, local):
    from linear_attention_04_gb300 import kda_chunk_bwd, kda_device_status
    from linear_attention_04_gb300 import kda as binding

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = selected_workload(args)
    if w.varlen:
        raise SystemExit("the backward takes fixed-length batches")
    inp = make_inputs(w, seed=rank_seed(args.seed, rank), device=dev)
    g = torch.Generator(device="cpu").manual_seed(args.seed + 3)
    d_out = torch.randn(w.B, w.T, w.H, w.dv, generator=g).to(dev)
    ws = torch.empty(binding.load().kda_chunk_bwd_workspace_size(w.B, w.H, w.T, w.dk, w.dv),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        kda_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["theta"], inp["beta"], d_out, w.g_min,
                      inp["init_state"], None, workspace=ws, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if kda_device_status(clear=True) != 0:
        raise RuntimeError("device status after warm-up")
    barrier(world)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(args.steps):
        step()
    end.record(stream)
    torch.cuda.synchronize()
    total_ms = max_over_ranks(start.elapsed_time(end), world)
    step_s = total_ms / args.steps / 1e3
    peaks, peak_src = measured_peaks()
    nbytes = bwd_bytes(w, inp)
    flops = bwd_flops(w, inp)
    achieved = flops / step_s / 1e12
    traffic, traffic_src = traffic_from_profiles("kda_bwd", w.name)
    tokens = n_tokens(inp)
    return {"metric": "KDA backward tokens/s (all gradients of the forward pass)",
            "value": tokens * world / step_s, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "op": "bwd",
            "config": {"workload": f"{w.name}: B={w.B} H={w.H} T={w.T} dk={w.dk} dv={w.dv}, "
                                   "fp32 arithmetic on CUDA cores"},
            "roofline": {"bound": "alu", "achieved": round(achieved, 2),
                         "peak": round(FP32_ALU_TFLOPS, 1), "unit": "TFLOP/s",
                         "frac": round(achieved / FP32_ALU_TFLOPS, 4), "traffic": traffic,
                         "traffic_source": traffic_src,
                         "peak_source": "derived: 152 SMs x 128 fp32 FMA lanes x 2 x 2070 MHz",
                         "kernel": "kda_bwd_kernel (one persistent launch per pass)",
                         "algorithmic_flops_per_pass": flops,
                         "hbm": {"achieved_gbs": round(nbytes / step_s / 1e9, 1),
                                 "peak_gbs": peaks["hbm_gbs"],
                                 "algorithmic_bytes_per_pass": nbytes}},
            "cpu_baseline": None, "e2e": None,
            "gpu_launches": BWD_LAUNCHES_PER_PASS * args.steps}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="train_bf16")
    ap.add_argument("--path", choices=["auto", "simt", "tc", "tc_split", "mma", "mma_tc"],
                    default="auto")
    ap.add_argument("--batch", type=int, default=0,
                    help="replace the workload's B (fixed-length workloads; profiling cases)")
    ap.add_argument("--heads", type=int, default=0,
                    help="replace the workload's H (fixed-length workloads; profiling cases)")
    ap.add_argument("--seed", type=int, default=20261204)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-step-seconds", type=float, default=3.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--gate", choices=["sigmoid", "log_decay"], default="sigmoid",
                    help="fwd: log_decay feeds g = -softplus(theta + logit_mu) (the unbounded "
                         "parameterisation; chunks past -G = 88 take the position-wise fallback)")
    ap.add_argument("--logit-mu", type=float, default=2.0)
    ap.add_argument("--segments", type=int, default=1,
                    help="fwd: cut each sequence into this many segments (segment-parallel path)")
    ap.add_argument("--op", choices=["fwd", "decode", "bwd"], default="fwd",
                    help="fwd: the chunked forward (the headline); decode: one recurrent step; "
                         "bwd: the backward pass")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        print("note: at least 3 warm-up steps are required; using 3", file=sys.stderr)
        args.warmup = 3
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            if rank != 0:
                return 0
            line = run_reference(args, rank, world)
        else:
            line = {"decode": run_decode, "bwd": run_bwd}.get(args.op, run_ours)(args, rank, world,
                                                                            local)
        if rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            import torch.distributed as dist
            if dist.is_initialized():
                dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
