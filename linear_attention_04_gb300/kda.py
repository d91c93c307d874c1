"""Thin Python binding of libkda.so (argument marshalling only).

Every step of the forward pass runs in the library's CUDA kernels; this module
only checks tensor metadata, allocates outputs with torch when the caller did
not pass them, and forwards raw device pointers and sizes through ctypes.
There is no fallback: if the library cannot be loaded the call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

KDA_OK = 0
KDA_ERR_INVALID_ARG = -1
KDA_ERR_MISALIGNED = -2
KDA_ERR_UNSUPPORTED_DEVICE = -3
KDA_ERR_LAUNCH = -4
KDA_ERR_DEVICE_TIMEOUT = -5
KDA_ERR_CUDA = -6
KDA_ERR_UNSUPPORTED_SHAPE = -7
KDA_ERR_SCRATCH_TOO_SMALL = -8
KDA_ERR_BAD_SEQLENS = -9

PATHS = {"auto": 0, "simt": 1, "tc": 2, "mma": 3, "tc_split": 4, "mma_tc": 5}
GATES = {"sigmoid": 0, "log_decay": 1}
DTYPES = {torch.bfloat16: 0, torch.float32: 1}

_lock = threading.Lock()
_lib = None


class KdaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} (code {code})")


class _BwdArgs(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k", "v", "theta", "beta")] + \
        [("g_min", ctypes.c_float)] + \
        [(n, ctypes.c_void_p) for n in ("init_state", "d_out", "d_final", "dq", "dk", "dv",
                                        "dtheta", "dbeta", "d_init")] + \
        [(n, ctypes.c_int) for n in ("B", "H", "T", "dk_dim", "dv_dim", "dtype", "gate")]


class _Args(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("theta", ctypes.c_void_p), ("beta", ctypes.c_void_p), ("g_min", ctypes.c_float),
                ("init_state", ctypes.c_void_p), ("out", ctypes.c_void_p),
                ("final_state", ctypes.c_void_p), ("cu_seqlens", ctypes.c_void_p),
                ("B", ctypes.c_int), ("H", ctypes.c_int), ("T", ctypes.c_int),
                ("dk", ctypes.c_int), ("dv", ctypes.c_int), ("dtype", ctypes.c_int),
                ("out_dtype", ctypes.c_int), ("path", ctypes.c_int), ("gate", ctypes.c_int)]


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libkda.so (building it first if needed).  Raises if impossible."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if build_if_missing:
                path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"libkda.so not found at {path}; run __graft_entry__.build()")
            lib = ctypes.CDLL(path)
            vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
            sig = [vp, vp, vp, vp, vp, f, vp, vp, vp, vp, i, i, i, i, i, vp]
            for name in ("kda_chunk_fwd", "kda_chunk_fwd_f32"):
                fn = getattr(lib, name)
                fn.restype = i
                fn.argtypes = sig
            lib.kda_segmented_workspace_size.restype = ctypes.c_size_t
            lib.kda_segmented_workspace_size.argtypes = [i, i, i, i, i, i]
            lib.kda_chunk_fwd_segmented.restype = i
            lib.kda_chunk_fwd_segmented.argtypes = [ctypes.POINTER(_Args), i, vp, ctypes.c_size_t,
                                                    vp]
            lib.kda_chunk_fwd_segmented_noalloc.restype = i
            lib.kda_chunk_fwd_segmented_noalloc.argtypes = [ctypes.POINTER(_Args), i, vp]
            lib.kda_chunk_bwd_workspace_size.restype = ctypes.c_size_t
            lib.kda_chunk_bwd_workspace_size.argtypes = [i, i, i, i, i]
            lib.kda_chunk_bwd.restype = i
            lib.kda_chunk_bwd.argtypes = [ctypes.POINTER(_BwdArgs), vp, ctypes.c_size_t, vp]
            lib.kda_selftest_withheld_handoff.restype = i
            lib.kda_selftest_withheld_handoff.argtypes = [ctypes.POINTER(_Args), ctypes.c_longlong,
                                                          vp, ctypes.c_size_t, vp]
            lib.kda_decode_step.restype = i
            lib.kda_decode_step.argtypes = [vp, vp, vp, vp, vp, f, vp, vp, i, i, i, i, i, vp]
            lib.kda_chunk_fwd_ex.restype = i
            lib.kda_chunk_fwd_ex.argtypes = [ctypes.POINTER(_Args), vp]
            lib.kda_debug_fwd_stages.restype = i
            lib.kda_debug_fwd_stages.argtypes = [ctypes.POINTER(_Args), vp, i, vp]
            lib.kda_debug_stage_floats.restype = i
            lib.kda_debug_stage_floats.argtypes = []
            lib.kda_device_status.restype = i
            lib.kda_device_status.argtypes = [i]
            lib.kda_select_path.restype = i
            lib.kda_select_path.argtypes = [i, i, i]
            lib.kda_strerror.restype = ctypes.c_char_p
            lib.kda_strerror.argtypes = [i]
            lib.kda_version.restype = i
            lib.kda_version.argtypes = []
            _lib = lib
    return _lib


def strerror(code: int) -> str:
    try:
        return load(build_if_missing=False).kda_strerror(int(code)).decode()
    except Exception:  # pragma: no cover - used while reporting another error
        return f"status {code}"


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _check_fwd(q, k, v, theta, beta, init_state, out, final_state, out_dtype, nseq=None):
    """Metadata checks shared by the forward bindings (before any C call)."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dtype = q.dtype
    if dtype not in DTYPES:
        raise TypeError(f"unsupported dtype {dtype}")
    for name, t, shape in (("k", k, (B, T, H, dk)), ("theta", theta, (B, T, H, dk)),
                           ("v", v, (B, T, H, dv)), ("beta", beta, (B, T, H))):
        if t.dtype != dtype or tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"{name}: expected contiguous {dtype} {shape}, got {t.dtype} "
                             f"{tuple(t.shape)}")
        if t.device != q.device:
            raise ValueError(f"{name} on {t.device}, q on {q.device}")
    if out_dtype not in DTYPES:
        raise TypeError(f"unsupported out dtype {out_dtype}")
    sshape = (B if nseq is None else nseq, H, dk, dv)
    for name, t in (("init_state", init_state), ("final_state", final_state)):
        if t is not None and (t.dtype != torch.float32 or tuple(t.shape) != sshape or
                              not t.is_contiguous() or t.device != q.device):
            raise ValueError(f"{name}: expected contiguous fp32 {sshape} on {q.device}")
    if out is not None and (out.dtype != out_dtype or tuple(out.shape) != (B, T, H, dv) or
                            not out.is_contiguous() or out.device != q.device):
        raise ValueError(f"out: expected contiguous {out_dtype} {(B, T, H, dv)} on {q.device}, "
                         f"got {out.dtype} {tuple(out.shape)}")
    if not q.is_cuda or not q.is_contiguous():
        raise ValueError("q must be a contiguous CUDA tensor")
    return sshape


def kda_chunk_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, theta: torch.Tensor,
                  beta: torch.Tensor, g_min: float = -5.0,
                  init_state: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                  final_state: Optional[torch.Tensor] = None,
                  cu_seqlens: Optional[torch.Tensor] = None, *, want_final_state: bool = True,
                  out_dtype: torch.dtype = torch.float32, path: str = "auto", gate: str = "sigmoid",
                  stream=None):
    """KDA chunked forward through the C ABI (``kda_chunk_fwd_ex``).

    q, k, theta [B,T,H,dk]; v [B,T,H,dv]; beta [B,T,H], all bf16 or all fp32,
    contiguous, on one CUDA device.  out [B,T,H,dv] is fp32 by default
    (``out_dtype=torch.bfloat16`` is accepted for bf16 inputs).  init_state/final_state fp32 [N,H,dk,dv]
    (N = B, or the number of sequences when cu_seqlens [N+1] int32 is given
    and B == 1).  Returns (out, final_state or None).  Asynchronous on
    ``stream`` (default: torch's current stream).
    ``path``: "auto" (the register-resident kernel for bf16 at dk = dv = 128,
    else the fp32 SIMT kernel), "mma", "mma_tc" (the same with the intra-chunk
    A and P on tcgen05), "tc" / "tc_split" (the tcgen05 kernel with 32-token
    state steps, more accurate under slow decay), or "simt".  ``gate``:
    "sigmoid" (g = g_min sigmoid(theta)) or "log_decay" (theta is g).
    """
    lib = load()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dtype = q.dtype
    nseq = B
    if cu_seqlens is not None:
        if B != 1:
            raise ValueError("packed varlen input must have B == 1")
        if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda:
            raise ValueError("cu_seqlens must be an int32 CUDA tensor")
        nseq = cu_seqlens.numel() - 1
    sshape = _check_fwd(q, k, v, theta, beta, init_state, out, final_state, out_dtype, nseq)
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=out_dtype, device=q.device)
    if final_state is None and want_final_state:
        final_state = torch.empty(sshape, dtype=torch.float32, device=q.device)
    a = _Args(_ptr(q), _ptr(k), _ptr(v), _ptr(theta), _ptr(beta), float(g_min),
              _ptr(init_state), _ptr(out), _ptr(final_state), _ptr(cu_seqlens),
              nseq, H, T, dk, dv, DTYPES[dtype], DTYPES[out_dtype], PATHS[path], GATES[gate])
    with torch.cuda.device(q.device):
        rc = lib.kda_chunk_fwd_ex(ctypes.byref(a), _stream_ptr(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_chunk_fwd_ex")
    return out, final_state


def kda_segmented_workspace_size(B: int, H: int, T: int, dk: int, dv: int, segments: int) -> int:
    return int(load().kda_segmented_workspace_size(B, H, T, dk, dv, segments))


def kda_chunk_fwd_segmented(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                            theta: torch.Tensor, beta: torch.Tensor, g_min: float = -5.0,
                            init_state: Optional[torch.Tensor] = None,
                            out: Optional[torch.Tensor] = None,
                            final_state: Optional[torch.Tensor] = None, *, segments: int = 4,
                            workspace: Optional[torch.Tensor] = None,
                            want_final_state: bool = True, out_dtype: torch.dtype = torch.float32,
                            path: str = "auto", stream=None):
    """Segment-parallel forward through the C ABI (``kda_chunk_fwd_segmented``):
    same arguments and results as ``kda_chunk_fwd`` for a fixed-length bf16
    batch with dk = dv = 128.  ``workspace`` is a uint8 CUDA tensor of at least
    ``kda_segmented_workspace_size`` bytes (allocated here when not given).
    ``path`` picks the kernel that runs the pieces ("mma", "tc_split", else tcgen05)."""
    lib = load()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    sshape = _check_fwd(q, k, v, theta, beta, init_state, out, final_state, out_dtype)
    if workspace is not None and (not workspace.is_cuda or not workspace.is_contiguous() or
                                  workspace.device != q.device):
        raise ValueError("workspace must be a contiguous CUDA tensor on q's device")
    if out is None:
        out = torch.empty((B, T, H, dv), dtype=out_dtype, device=q.device)
    if final_state is None and want_final_state:
        final_state = torch.empty(sshape, dtype=torch.float32, device=q.device)
    need = kda_segmented_workspace_size(B, H, T, dk, dv, segments)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    a = _Args(_ptr(q), _ptr(k), _ptr(v), _ptr(theta), _ptr(beta), float(g_min),
              _ptr(init_state), _ptr(out), _ptr(final_state), None, B, H, T, dk, dv,
              DTYPES[q.dtype], DTYPES[out_dtype], PATHS[path])
    with torch.cuda.device(q.device):
        rc = lib.kda_chunk_fwd_segmented(ctypes.byref(a), int(segments), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_chunk_fwd_segmented")
    return out, final_state


def kda_chunk_fwd_segmented_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                                    theta: torch.Tensor, beta: torch.Tensor, g_min: float,
                                    init_state: Optional[torch.Tensor], out: torch.Tensor,
                                    final_state: Optional[torch.Tensor], *, segments: int = 4,
                                    out_dtype: Optional[torch.dtype] = None, path: str = "auto",
                                    stream=None):
    """``kda_chunk_fwd_segmented_noalloc`` through the C ABI: the segment-parallel
    forward over the library's own scratch area.  ``out`` (and ``final_state``
    when wanted) are caller tensors; nothing is allocated here.  The output
    element type is ``out.dtype`` (``out_dtype``, if given, must agree)."""
    lib = load()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if out is None:
        raise ValueError("out must be given")
    if out_dtype is not None and out_dtype != out.dtype:
        raise ValueError(f"out_dtype {out_dtype} does not match out.dtype {out.dtype}")
    out_dtype = out.dtype
    _check_fwd(q, k, v, theta, beta, init_state, out, final_state, out_dtype)
    a = _Args(_ptr(q), _ptr(k), _ptr(v), _ptr(theta), _ptr(beta), float(g_min),
              _ptr(init_state), _ptr(out), _ptr(final_state), None, B, H, T, dk, dv,
              DTYPES[q.dtype], DTYPES[out_dtype], PATHS[path])
    with torch.cuda.device(q.device):
        rc = lib.kda_chunk_fwd_segmented_noalloc(ctypes.byref(a), int(segments),
                                                 _stream_ptr(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_chunk_fwd_segmented_noalloc")
    return out, final_state


def kda_chunk_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, theta: torch.Tensor,
                  beta: torch.Tensor, d_out: torch.Tensor, g_min: float = -5.0,
                  init_state: Optional[torch.Tensor] = None,
                  d_final: Optional[torch.Tensor] = None, *, gate: str = "sigmoid",
                  workspace: Optional[torch.Tensor] = None, stream=None) -> dict:
    """Backward pass through the C ABI (``kda_chunk_bwd``): gradients of
    sum(out * d_out) + sum(final_state * d_final) w.r.t. q, k, v, theta, beta
    and init_state, as fp32 tensors in a dict (dq, dk, dv, dtheta, dbeta,
    d_init).  Fixed-length batch, dk = dv = 128."""
    lib = load()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    dev = q.device
    for name, t, shape in (("k", k, (B, T, H, dk)), ("theta", theta, (B, T, H, dk)),
                           ("v", v, (B, T, H, dv)), ("beta", beta, (B, T, H))):
        if t.dtype != q.dtype or tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"{name}: expected contiguous {q.dtype} {shape}")
    if d_out.dtype != torch.float32 or tuple(d_out.shape) != (B, T, H, dv) or \
            not d_out.is_contiguous():
        raise ValueError(f"d_out: expected contiguous fp32 {(B, T, H, dv)}")
    g = {"dq": torch.empty((B, T, H, dk), device=dev), "dk": torch.empty((B, T, H, dk), device=dev),
         "dv": torch.empty((B, T, H, dv), device=dev),
         "dtheta": torch.empty((B, T, H, dk), device=dev),
         "dbeta": torch.empty((B, T, H), device=dev),
         "d_init": torch.empty((B, H, dk, dv), device=dev)}
    need = int(lib.kda_chunk_bwd_workspace_size(B, H, T, dk, dv))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    a = _BwdArgs(_ptr(q), _ptr(k), _ptr(v), _ptr(theta), _ptr(beta), float(g_min),
                 _ptr(init_state), _ptr(d_out), _ptr(d_final), _ptr(g["dq"]), _ptr(g["dk"]),
                 _ptr(g["dv"]), _ptr(g["dtheta"]), _ptr(g["dbeta"]), _ptr(g["d_init"]),
                 B, H, T, dk, dv, DTYPES[q.dtype], GATES[gate])
    with torch.cuda.device(dev):
        rc = lib.kda_chunk_bwd(ctypes.byref(a), _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream_ptr(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_chunk_bwd")
    return g


def kda_decode_step(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, theta: torch.Tensor,
                    beta: torch.Tensor, state: torch.Tensor, g_min: float = -5.0,
                    out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """One recurrent step through the C ABI (``kda_decode_step``): q, k, theta
    [N,H,dk]; v [N,H,dv]; beta [N,H] (all bf16 or all fp32, contiguous, on one
    CUDA device); state fp32 [N,H,dk,dv] is updated in place.  Returns out fp32
    [N,H,dv].  Asynchronous on ``stream``."""
    lib = load()
    N, H, dk = q.shape
    dv = v.shape[-1]
    dtype = q.dtype
    if dtype not in DTYPES:
        raise TypeError(f"unsupported dtype {dtype}")
    for name, t, shape in (("k", k, (N, H, dk)), ("theta", theta, (N, H, dk)),
                           ("v", v, (N, H, dv)), ("beta", beta, (N, H))):
        if t.dtype != dtype or tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"{name}: expected contiguous {dtype} {shape}, got {t.dtype} "
                             f"{tuple(t.shape)}")
        if t.device != q.device:
            raise ValueError(f"{name} on {t.device}, q on {q.device}")
    if not q.is_cuda or not q.is_contiguous():
        raise ValueError("q must be a contiguous CUDA tensor")
    if state.dtype != torch.float32 or tuple(state.shape) != (N, H, dk, dv) or \
            not state.is_contiguous() or state.device != q.device:
        raise ValueError(f"state: expected contiguous fp32 {(N, H, dk, dv)} on {q.device}")
    if out is None:
        out = torch.empty((N, H, dv), dtype=torch.float32, device=q.device)
    elif out.dtype != torch.float32 or tuple(out.shape) != (N, H, dv) or not out.is_contiguous():
        raise ValueError(f"out: expected contiguous fp32 {(N, H, dv)}")
    with torch.cuda.device(q.device):
        rc = lib.kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(theta), _ptr(beta), float(g_min),
                                 _ptr(state), _ptr(out), N, H, dk, dv, DTYPES[dtype],
                                 _stream_ptr(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_decode_step")
    return out


def kda_debug_fwd_stages(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, theta: torch.Tensor,
                         beta: torch.Tensor, g_min: float = -5.0,
                         init_state: Optional[torch.Tensor] = None, *, nsc: int = 2,
                         gate: str = "sigmoid", path: str = "tc", stream=None):
    """Test hook ``kda_debug_fwd_stages``: runs the tcgen05 forward and returns
    (out, final_state, stages) where stages holds the intermediate tiles of
    the first (sequence, head) chain for its first ``nsc`` 32-token units as
    fp32 CPU tensors: A, P, T [nsc,32,32]; W, U [nsc,32,128]; eG [nsc,128];
    qk [nsc,32]."""
    lib = load()
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    sshape = _check_fwd(q, k, v, theta, beta, init_state, None, None, torch.float32)
    out = torch.empty((B, T, H, dv), dtype=torch.float32, device=q.device)
    fin = torch.empty(sshape, dtype=torch.float32, device=q.device)
    per = int(lib.kda_debug_stage_floats())
    dump = torch.zeros(nsc * per, dtype=torch.float32, device=q.device)
    a = _Args(_ptr(q), _ptr(k), _ptr(v), _ptr(theta), _ptr(beta), float(g_min),
              _ptr(init_state), _ptr(out), _ptr(fin), None, B, H, T, dk, dv,
              DTYPES[q.dtype], DTYPES[torch.float32], PATHS[path], GATES[gate])
    with torch.cuda.device(q.device):
        rc = lib.kda_debug_fwd_stages(ctypes.byref(a), _ptr(dump), int(nsc), _stream_ptr(stream))
    if rc != KDA_OK:
        raise KdaError(rc, "kda_debug_fwd_stages")
    d = dump.view(nsc, per).cpu()
    o = 0
    stages = {}
    for name, shape in (("A", (32, 32)), ("P", (32, 32)), ("T", (32, 32)), ("W", (32, 128)),
                        ("U", (32, 128)), ("eG", (128,)), ("qk", (32,))):
        n = 1
        for x in shape:
            n *= x
        stages[name] = d[:, o:o + n].reshape((nsc,) + shape)
        o += n
    return out, fin, stages


def kda_device_status(clear: bool = False) -> int:
    return int(load().kda_device_status(1 if clear else 0))


def kda_select_path(dtype: torch.dtype, dk: int, dv: int) -> str:
    r = load().kda_select_path(DTYPES[dtype], dk, dv)
    if r < 0:
        raise KdaError(r, "kda_select_path")
    return {v: k for k, v in PATHS.items()}[r]
