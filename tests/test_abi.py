"""The C ABI: the library builds and loads, exports every symbol include/kda.h
declares, and rejects bad arguments on the host (no compute, no GPU needed)."""
import ctypes
import os
import re

import pytest

from linear_attention_04_gb300 import kda as binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            with open(os.path.join(ROOT, "include", fn)) as f:
                txt = f.read()
            names += re.findall(r"KDA_API\s+[\w\s\*]+?\b(kda_\w+)\s*\(", txt)
    return sorted(set(names))


def test_header_declares_entry_points():
    names = _declared_symbols()
    for n in ("kda_chunk_fwd", "kda_chunk_fwd_f32", "kda_chunk_fwd_ex", "kda_device_status",
              "kda_strerror", "kda_select_path", "kda_version"):
        assert n in names


def test_fused_forward_needs_no_workspace():
    lib = binding.load()
    lib.kda_chunk_fwd_workspace_size.restype = ctypes.c_size_t
    for shape in ((8, 32, 8192, 128, 128), (1, 2, 64, 16, 16), (3, 1, 0, 64, 128)):
        assert lib.kda_chunk_fwd_workspace_size(*shape) == 0


def test_library_exports_every_declared_symbol():
    lib = binding.load()
    missing = [n for n in _declared_symbols() if not hasattr(lib, n)]
    assert not missing, missing


def test_strerror_and_version():
    lib = binding.load()
    for code in range(-9, 1):
        assert lib.kda_strerror(code)
    assert lib.kda_strerror(-999) == b"unknown status code"
    assert lib.kda_version() >= 100


def _args(**over):
    a = dict(q=0x1000, k=0x2000, v=0x3000, theta=0x4000, beta=0x5000, g_min=-5.0,
             init_state=None, out=0x6000, final_state=None, cu_seqlens=None, B=1, H=1, T=16,
             dk=128, dv=128, dtype=0, out_dtype=1, path=0)
    a.update(over)
    return binding._Args(**a)


@pytest.mark.parametrize("over,code", [
    (dict(q=None), binding.KDA_ERR_INVALID_ARG),
    (dict(beta=None), binding.KDA_ERR_INVALID_ARG),
    (dict(out=None), binding.KDA_ERR_INVALID_ARG),
    (dict(B=0), binding.KDA_ERR_INVALID_ARG),
    (dict(H=-1), binding.KDA_ERR_INVALID_ARG),
    (dict(T=-5), binding.KDA_ERR_INVALID_ARG),
    (dict(g_min=0.0), binding.KDA_ERR_INVALID_ARG),
    (dict(g_min=1.0), binding.KDA_ERR_INVALID_ARG),
    (dict(g_min=float("nan")), binding.KDA_ERR_INVALID_ARG),
    (dict(dtype=7), binding.KDA_ERR_INVALID_ARG),
    (dict(out_dtype=3), binding.KDA_ERR_INVALID_ARG),
    (dict(dtype=1, out_dtype=0), binding.KDA_ERR_INVALID_ARG),
    (dict(path=9), binding.KDA_ERR_INVALID_ARG),
    (dict(path=6), binding.KDA_ERR_INVALID_ARG),
    (dict(dk=24), binding.KDA_ERR_UNSUPPORTED_SHAPE),
    (dict(dv=256), binding.KDA_ERR_UNSUPPORTED_SHAPE),
    (dict(q=0x1001), binding.KDA_ERR_MISALIGNED),
    (dict(final_state=0x7004), binding.KDA_ERR_MISALIGNED),
    (dict(cu_seqlens=0x8002), binding.KDA_ERR_MISALIGNED),
])
def test_host_side_rejection(over, code):
    lib = binding.load()
    a = _args(**over)
    assert lib.kda_chunk_fwd_ex(ctypes.byref(a), None) == code
    assert lib.kda_chunk_fwd_ex(None, None) == binding.KDA_ERR_INVALID_ARG


def test_select_path_host_logic():
    lib = binding.load()
    assert lib.kda_select_path(1, 16, 16) == 1          # fp32 -> SIMT
    assert lib.kda_select_path(0, 24, 128) == binding.KDA_ERR_UNSUPPORTED_SHAPE
    assert lib.kda_select_path(5, 128, 128) == binding.KDA_ERR_INVALID_ARG
    assert lib.kda_select_path(0, 64, 64) == 1          # bf16 off the 128 x 128 shape -> SIMT
    assert lib.kda_select_path(0, 128, 128) == 3        # bf16, dk = dv = 128 -> register-resident path


def _decode(lib, **over):
    a = dict(q=0x1000, k=0x2000, v=0x3000, theta=0x4000, beta=0x5000, g_min=-5.0, state=0x6000,
             out=0x7000, N=2, H=4, dk=128, dv=128, dtype=0)
    a.update(over)
    return lib.kda_decode_step(a["q"], a["k"], a["v"], a["theta"], a["beta"], a["g_min"],
                               a["state"], a["out"], a["N"], a["H"], a["dk"], a["dv"], a["dtype"],
                               None)


@pytest.mark.parametrize("over,code", [
    (dict(q=None), binding.KDA_ERR_INVALID_ARG),
    (dict(state=None), binding.KDA_ERR_INVALID_ARG),
    (dict(out=None), binding.KDA_ERR_INVALID_ARG),
    (dict(N=-1), binding.KDA_ERR_INVALID_ARG),
    (dict(H=0), binding.KDA_ERR_INVALID_ARG),
    (dict(g_min=0.0), binding.KDA_ERR_INVALID_ARG),
    (dict(dtype=4), binding.KDA_ERR_INVALID_ARG),
    (dict(dk=48), binding.KDA_ERR_UNSUPPORTED_SHAPE),
    (dict(dv=8), binding.KDA_ERR_UNSUPPORTED_SHAPE),
    (dict(theta=0x4008), binding.KDA_ERR_MISALIGNED),
    (dict(state=0x6004), binding.KDA_ERR_MISALIGNED),
])
def test_decode_host_side_rejection(over, code):
    assert _decode(binding.load(), **over) == code


def test_decode_empty_batch_is_a_noop():
    # N = 0 returns before any device work (null pointers allowed)
    assert _decode(binding.load(), N=0, q=None, k=None, v=None, theta=None, beta=None, state=None,
                   out=None) == binding.KDA_OK


def test_segmented_workspace_size_host_logic():
    lib = binding.load()
    n1 = lib.kda_segmented_workspace_size(1, 32, 262144, 128, 128, 4)
    n2 = lib.kda_segmented_workspace_size(1, 32, 262144, 128, 128, 8)
    assert 0 < n1 < n2 and n1 % 256 == 0
    # one segment needs no scratch beyond alignment; bad shapes give 0
    assert lib.kda_segmented_workspace_size(1, 32, 262144, 128, 128, 1) < 1024
    assert lib.kda_segmented_workspace_size(1, 32, 4096, 64, 128, 4) == 0
    assert lib.kda_segmented_workspace_size(0, 32, 4096, 128, 128, 4) == 0


@pytest.mark.parametrize("over,extra,code", [
    (dict(dtype=1), {}, binding.KDA_ERR_UNSUPPORTED_SHAPE),
    (dict(dk=64), {}, binding.KDA_ERR_UNSUPPORTED_SHAPE),
    (dict(cu_seqlens=0x9000), {}, binding.KDA_ERR_INVALID_ARG),
    (dict(), dict(segments=0), binding.KDA_ERR_INVALID_ARG),
    (dict(T=4096), dict(ws=0x10000, nbytes=64), binding.KDA_ERR_INVALID_ARG),
    (dict(T=4096), dict(ws=None), binding.KDA_ERR_INVALID_ARG),
    (dict(T=4096), dict(ws=0x10010), binding.KDA_ERR_MISALIGNED),
    (dict(q=None, T=4096), {}, binding.KDA_ERR_INVALID_ARG),
    (dict(B=1024, T=1 << 21), {}, binding.KDA_ERR_INVALID_ARG),   # B * T >= 2^31
])
def test_segmented_host_side_rejection(over, extra, code):
    lib = binding.load()
    a = _args(**over)
    seg = extra.get("segments", 4)
    ws = extra.get("ws", 0x10000)
    nbytes = extra.get("nbytes", 1 << 40)
    assert lib.kda_chunk_fwd_segmented(ctypes.byref(a), seg, ws, nbytes, None) == code


@pytest.mark.parametrize("over,seg,code", [
    (dict(B=1, H=32, T=262144), 16, binding.KDA_ERR_SCRATCH_TOO_SMALL),   # needs > 24 MiB
    (dict(B=8, H=32, T=8192), 4, binding.KDA_ERR_SCRATCH_TOO_SMALL),
    (dict(dtype=1), 4, binding.KDA_ERR_UNSUPPORTED_SHAPE),
    (dict(cu_seqlens=0x9000), 4, binding.KDA_ERR_INVALID_ARG),
    (dict(), 0, binding.KDA_ERR_INVALID_ARG),
    (dict(g_min=0.5), 4, binding.KDA_ERR_INVALID_ARG),
    (dict(B=1024, T=1 << 21), 2, binding.KDA_ERR_INVALID_ARG),   # B * T >= 2^31
])
def test_noalloc_host_side_rejection(over, seg, code):
    lib = binding.load()
    a = _args(**over)
    assert lib.kda_chunk_fwd_segmented_noalloc(ctypes.byref(a), seg, None) == code


def test_noalloc_capacity_covers_the_long_workload():
    lib = binding.load()
    cap = 24 << 20
    assert lib.kda_segmented_workspace_size(1, 32, 262144, 128, 128, 5) <= cap
    assert lib.kda_segmented_workspace_size(1, 32, 262144, 128, 128, 6) > cap


def test_gate_mode_host_checks():
    lib = binding.load()
    a = _args(gate=7)
    assert lib.kda_chunk_fwd_ex(ctypes.byref(a), None) == binding.KDA_ERR_INVALID_ARG
    # the log-decay gate ignores g_min, so g_min = 0 passes the argument check
    # (and stops only at the device check on a machine without a GB300)
    a = _args(gate=1, g_min=0.0)
    assert lib.kda_chunk_fwd_ex(ctypes.byref(a), None) != binding.KDA_ERR_INVALID_ARG
    # every tensor-core path takes both gates; they need bf16 inputs at 128 x 128
    for path in (2, 3, 4, 5):
        a = _args(gate=1, path=path)
        assert lib.kda_chunk_fwd_ex(ctypes.byref(a), None) not in (
            binding.KDA_ERR_INVALID_ARG, binding.KDA_ERR_UNSUPPORTED_SHAPE)
        a = _args(path=path, dk=64, dv=64)
        assert lib.kda_chunk_fwd_ex(ctypes.byref(a), None) == binding.KDA_ERR_UNSUPPORTED_SHAPE


def _bwd_args(**over):
    a = dict(q=0x1000, k=0x2000, v=0x3000, theta=0x4000, beta=0x5000, g_min=-5.0,
             init_state=None, d_out=0x6000, d_final=None, dq=0x7000, dk=0x8000, dv=0x9000,
             dtheta=0xa000, dbeta=0xb000, d_init=None, B=1, H=2, T=64, dk_dim=128, dv_dim=128,
             dtype=0, gate=0)
    a.update(over)
    return binding._BwdArgs(**a)


@pytest.mark.parametrize("over,code", [
    (dict(dq=None), binding.KDA_ERR_INVALID_ARG),
    (dict(d_out=None), binding.KDA_ERR_INVALID_ARG),
    (dict(B=0), binding.KDA_ERR_INVALID_ARG),
    (dict(g_min=1.0), binding.KDA_ERR_INVALID_ARG),
    (dict(gate=5), binding.KDA_ERR_INVALID_ARG),
    (dict(dk_dim=64), binding.KDA_ERR_UNSUPPORTED_SHAPE),
    (dict(dtheta=0xa004), binding.KDA_ERR_MISALIGNED),
])
def test_bwd_host_side_rejection(over, code):
    lib = binding.load()
    a = _bwd_args(**over)
    assert lib.kda_chunk_bwd(ctypes.byref(a), 0x100000, 1 << 40, None) == code


def test_bwd_workspace_rules():
    lib = binding.load()
    # per chain and 16-token chunk: the chunk-start state, the end-of-chunk
    # state gradient (128 x 128 fp32 each), dU, R and U (16 x 128 fp32 each)
    # per chunk: two fp32 128 x 128 states and three 16 x 128 tiles; then the
    # work queue: its position (256 bytes) and one int per chain, in 256-byte units
    queue = 256 + 256
    n = lib.kda_chunk_bwd_workspace_size(1, 2, 64, 128, 128)
    assert n == 2 * 4 * (2 * 128 * 128 + 3 * 16 * 128) * 4 + queue
    assert lib.kda_chunk_bwd_workspace_size(1, 2, 65, 128, 128) == \
        2 * 5 * (2 * 128 * 128 + 3 * 16 * 128) * 4 + queue
    assert lib.kda_chunk_bwd_workspace_size(8, 32, 16, 128, 128) == \
        256 * (2 * 128 * 128 + 3 * 16 * 128) * 4 + 256 + 1024
    assert lib.kda_chunk_bwd_workspace_size(1, 2, 64, 64, 128) == 0
    a = _bwd_args()
    assert lib.kda_chunk_bwd(ctypes.byref(a), 0x100000, n - 1, None) == binding.KDA_ERR_INVALID_ARG
    assert lib.kda_chunk_bwd(ctypes.byref(a), None, n, None) == binding.KDA_ERR_INVALID_ARG


@pytest.mark.parametrize("over,limit,ws,code", [
    (dict(), 0, 0x10000, binding.KDA_ERR_INVALID_ARG),
    (dict(T=8), 1000000, 0x10000, binding.KDA_ERR_INVALID_ARG),
    (dict(), 1000000, None, binding.KDA_ERR_INVALID_ARG),
    (dict(dtype=1), 1000000, 0x10000, binding.KDA_ERR_UNSUPPORTED_SHAPE),
    (dict(), 1000000, 0x10008, binding.KDA_ERR_MISALIGNED),
])
def test_selftest_hook_host_side_rejection(over, limit, ws, code):
    lib = binding.load()
    a = _args(**over)
    assert lib.kda_selftest_withheld_handoff(ctypes.byref(a), limit, ws, 256, None) == code


@pytest.mark.parametrize("over,nsc,dump,code", [
    (dict(), 0, 0x20000, binding.KDA_ERR_INVALID_ARG),
    (dict(), 2, None, binding.KDA_ERR_INVALID_ARG),
    (dict(), 2, 0x20004, binding.KDA_ERR_MISALIGNED),
    (dict(dtype=1), 2, 0x20000, binding.KDA_ERR_UNSUPPORTED_SHAPE),
    (dict(dk=64, dv=64), 2, 0x20000, binding.KDA_ERR_UNSUPPORTED_SHAPE),
    (dict(T=0), 2, 0x20000, binding.KDA_ERR_INVALID_ARG),
])
def test_stage_dump_hook_host_side_rejection(over, nsc, dump, code):
    lib = binding.load()
    a = _args(**over)
    assert lib.kda_debug_fwd_stages(ctypes.byref(a), dump, nsc, None) == code
    assert lib.kda_debug_stage_floats() == 3 * 32 * 32 + 2 * 32 * 128 + 128 + 32


def _cpu_inputs(B=1, T=32, H=2, d=128):
    import torch
    mk = lambda *s: torch.zeros(*s, dtype=torch.bfloat16)
    return mk(B, T, H, d), mk(B, T, H, d), mk(B, T, H, d), mk(B, T, H, d), mk(B, T, H)


def test_binding_rejects_a_mismatched_out_before_the_c_call():
    import torch
    q, k, v, th, be = _cpu_inputs()
    # an out whose element type disagrees with the requested one: caught in
    # Python, before any pointer reaches the library
    with pytest.raises(ValueError, match="out_dtype"):
        binding.kda_chunk_fwd_segmented_noalloc(q, k, v, th, be, -5.0, None,
                                                torch.zeros(1, 32, 2, 128, dtype=torch.bfloat16),
                                                None, out_dtype=torch.float32)
    with pytest.raises(ValueError, match="out"):
        binding.kda_chunk_fwd_segmented(q, k, v, th, be, -5.0,
                                        out=torch.zeros(1, 16, 2, 128))
    with pytest.raises(ValueError, match="final_state"):
        binding.kda_chunk_fwd_segmented_noalloc(q, k, v, th, be, -5.0, None,
                                                torch.zeros(1, 32, 2, 128), torch.zeros(1, 2, 64, 128))
    with pytest.raises(ValueError, match="theta"):
        binding.kda_chunk_fwd(q, k, v, th[:, :16].contiguous(), be)


def _list_schedule(jobs, sms):
    import heapq
    free = [0] * sms
    end = 0
    for j in jobs:
        t = heapq.heappop(free) + j
        heapq.heappush(free, t)
        end = max(end, t)
    return end


def _model(chains, P, n, u0, u, sms):
    # launch 1: segment 0 of every chain, then two jobs per segment 1 .. P-2;
    # launch 2: one job per segment 1 .. P-1 (the last what is left)
    j1 = [u0] * chains + [u] * (chains * 2 * (P - 2))
    j2 = []
    for s in range(1, P):
        j2 += [u if s < P - 1 else n - u0 - (P - 2) * u] * chains
    return _list_schedule(j1, sms) + _list_schedule(j2, sms)


@pytest.mark.parametrize("B,H,T,P,sms", [(1, 32, 262144, 5, 152), (1, 32, 262144, 4, 152),
                                         (1, 32, 262144, 6, 152), (2, 3, 3000, 3, 152),
                                         (1, 32, 2048, 5, 152), (1, 32, 262144, 5, 0)])
def test_segment_plan_host_logic(B, H, T, P, sms):
    # the planner keeps equal segments unless a first segment of twice the
    # others' length finishes first under a list-scheduling model of the two
    # launches (restated here on its own)
    lib = binding.load()
    lib.kda_debug_segment_plan.argtypes = [ctypes.c_int] * 5 + [ctypes.POINTER(ctypes.c_int64)]
    out = (ctypes.c_int64 * 3)()
    assert lib.kda_debug_segment_plan(B, H, T, P, sms, out) == 0
    nseg, l0, l = out[0], out[1], out[2]
    n = -(-T // 32)                      # 32-token units
    per = -(-n // P)
    assert nseg == -(-n // per)
    equal = (per * 32, per * 32)
    u = (n + P) // (P + 1)
    doubled = (2 * u * 32, u * 32)
    chains = B * H
    pick = equal
    if sms > 0 and nseg >= 3 and 2 * u + (nseg - 2) * u < n and \
            _model(chains, nseg, n, 2 * u, u, sms) < _model(chains, nseg, n, per, per, sms):
        pick = doubled
    assert (l0, l) == pick
    # the segments cover the sequence
    assert l0 + (nseg - 1) * l >= T > l0 + (nseg - 2) * l
    if (B, H, T, P, sms) == (1, 32, 262144, 5, 152):
        assert (l0, l) == doubled      # the long workload's plan
    if sms == 0 or chains < 8:
        assert (l0, l) == equal
