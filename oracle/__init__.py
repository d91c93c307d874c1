"""fp64 CPU oracle for the Kimi Delta Attention (KDA) forward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The CUDA library
never links, loads or calls it, and it imports nothing from the CUDA side.

``kda_oracle.c`` holds the token-by-token recurrence (see its header for the
equations and the passages they come from); ``chunked.py`` holds an fp64
restatement of the chunk-parallel (WY) form, used to check the oracle's
chunk invariance and to give reference values for the individual stages.

Parity status of each function (what pins it is listed in the tests):
  fwd        pinned (brute-force unrolled products, beta=1 retrieval identity,
             GLA / causal-linear-attention reductions, state continuation,
             linearity, column independence, varlen independence)
  gate       pinned (closed form values of the sigmoid, range [g_min, 0])
  chunked    pinned against ``fwd`` (chunk-size invariance)
  backward   (oracle/backward.py) pinned: its forward equals ``fwd``; its
             gradients equal central finite differences of ``fwd``
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None

# planted mistakes, mirrored from kda_oracle.c (test use only)
MUTATIONS = {
    "no_decay": 1,
    "decay_after": 2,
    "erase_sign": 3,
    "read_before": 4,
    "read_transposed": 5,
    "erase_no_beta": 6,
    "gate_sign": 7,
    "decay_channel": 8,
    "no_reset": 9,
    "beta_shift": 10,
    "write_key": 11,
}


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (portable flags only)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int32)
            lib.kda_oracle_fwd_f64.restype = ctypes.c_int
            lib.kda_oracle_fwd_f64.argtypes = [dp, dp, dp, dp, dp, ctypes.c_double, dp, dp, dp,
                                               ip] + [ctypes.c_int] * 9
            lib.kda_oracle_gate_f64.restype = None
            lib.kda_oracle_gate_f64.argtypes = [dp, ctypes.c_double, ctypes.c_int64, dp]
            _lib = lib
    return _lib


def host_threads() -> int:
    """Cores this process may run on (the oracle's default thread count)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _f64(a):
    if a is None:
        return None
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    return a


def _ptr(a, ty=ctypes.c_double):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ty))


def fwd(q, k, v, theta, beta, g_min=-5.0, init_state=None, cu_seqlens=None, *,
        theta_is_g=False, erase=True, mutation=0, nthreads=None, want_state=True):
    """Run the fp64 recurrence.

    Shapes: q,k,theta [B,T,H,dk]; v [B,T,H,dv]; beta [B,T,H]; init_state
    [N,H,dk,dv] with N = B (fixed length) or the number of sequences (varlen,
    where B must be 1 and cu_seqlens has N+1 entries).
    Returns (o [B,T,H,dv], final_state [N,H,dk,dv] or None).
    """
    q, k, v, theta, beta = (_f64(x) for x in (q, k, v, theta, beta))
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    assert k.shape == q.shape and theta.shape == q.shape
    assert v.shape == (B, T, H, dv) and beta.shape == (B, T, H)
    cu = None
    nseq = B
    if cu_seqlens is not None:
        assert B == 1
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
        nseq = cu.shape[0] - 1
    init = _f64(init_state)
    if init is not None:
        assert init.shape == (nseq, H, dk, dv)
    out = np.zeros((B, T, H, dv), dtype=np.float64)
    fin = np.zeros((nseq, H, dk, dv), dtype=np.float64) if want_state else None
    if isinstance(mutation, str):
        mutation = MUTATIONS[mutation]
    nthreads = host_threads() if nthreads is None else int(nthreads)
    lib = _load()
    rc = lib.kda_oracle_fwd_f64(
        _ptr(q), _ptr(k), _ptr(v), _ptr(theta), _ptr(beta), float(g_min), _ptr(init),
        _ptr(out), _ptr(fin), _ptr(cu, ctypes.c_int32), nseq, H, T if cu is not None else T,
        dk, dv, int(bool(theta_is_g)), int(bool(erase)), int(mutation), nthreads)
    if rc != 0:
        raise ValueError(f"kda_oracle_fwd_f64 rejected its arguments (rc={rc})")
    return out, fin


def gate(theta, g_min=-5.0):
    """g = g_min * sigmoid(theta), fp64, same shape as theta."""
    th = _f64(theta)
    g = np.empty_like(th)
    _load().kda_oracle_gate_f64(_ptr(th), float(g_min), th.size, _ptr(g))
    return g
