"""Seeded synthetic inputs for the KDA forward pass.

This module only draws random numbers and shapes them; it holds none of the
method's arithmetic, so both the CUDA path and the fp64 oracle may use it.

The five named workloads follow the shapes and value distributions of the
pages' training setting (pre-training contexts of 8K-1M tokens, "Kimi K3",
section "Training the whole system"; 16-token chunks and g_min = -5 from
"Kimi K3 Deep Dive", section "Core Innovation 1").  No dataset is involved:
everything is synthetic.

Recipe (all values drawn in fp32 with ``torch.Generator.manual_seed(seed)``,
in this order, then cast to the workload dtype):
  q, k   N(0,1), then L2-normalised over the channel axis per (token, head)
  v      N(0,1)
  theta  N(0,1) per (token, head, channel)   [tiny/base/train/long]
         U[6,12]                             [varlen stress: every g ~ g_min]
  beta   sigmoid(N(0,1)) per (token, head)   [tiny/base/train/long]
         U[0.9,1.0]                          [varlen stress]
  init   zero, except "long": fp32 N(0, 0.02^2) per state entry
Varlen lengths come from a second generator seeded with ``seed + 7919``:
L = 16 * randint(8, 1024 inclusive), i.e. uniform over the multiples of 16 in
[128, 16384].
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

DEFAULT_SEED = 20261202


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int                      # batch (fixed length) or number of sequences (varlen)
    H: int
    T: int                      # tokens per sequence (fixed) -- ignored for varlen
    dk: int
    dv: int
    dtype: torch.dtype
    theta: str = "normal"       # "normal" | "uniform6_12"
    beta: str = "sigmoid_normal"  # "sigmoid_normal" | "uniform09_1"
    init_std: float = 0.0       # 0 => zero initial state
    varlen: bool = False
    min_len: int = 128          # varlen only (multiples of 16)
    max_len: int = 16384
    g_min: float = -5.0
    index: int = -1             # position in the named list (seed offset)

    @property
    def dtype_name(self) -> str:
        return {torch.float32: "f32", torch.bfloat16: "bf16"}[self.dtype]


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", B=1, H=2, T=64, dk=16, dv=16, dtype=torch.float32, index=0),
    "base_bf16": Workload("base_bf16", B=1, H=8, T=4096, dk=128, dv=128, dtype=torch.bfloat16,
                          index=1),
    "train_bf16": Workload("train_bf16", B=8, H=32, T=8192, dk=128, dv=128,
                           dtype=torch.bfloat16, index=2),
    "long_bf16": Workload("long_bf16", B=1, H=32, T=262144, dk=128, dv=128,
                          dtype=torch.bfloat16, init_std=0.02, index=3),
    "varlen_bf16": Workload("varlen_bf16", B=64, H=16, T=0, dk=128, dv=128, dtype=torch.bfloat16,
                            theta="uniform6_12", beta="uniform09_1", varlen=True, index=4),
}
ORDER = ["tiny_f32", "base_bf16", "train_bf16", "long_bf16", "varlen_bf16"]


def default_seed(w: Workload) -> int:
    return DEFAULT_SEED + max(w.index, 0)


def varlen_lengths(w: Workload, seed: int) -> list[int]:
    g = torch.Generator().manual_seed(seed + 7919)
    lo, hi = w.min_len // 16, w.max_len // 16
    n = torch.randint(lo, hi + 1, (w.B,), generator=g)
    return [int(16 * x) for x in n.tolist()]


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)


def make_inputs(w: Workload, seed: Optional[int] = None, device="cpu",
                lengths: Optional[list[int]] = None) -> dict:
    """Draw one input set.  Returns a dict of tensors on ``device``:

    q,k,theta [Bt,T,H,dk]; v [Bt,T,H,dv]; beta [Bt,T,H] (workload dtype);
    init_state [N,H,dk,dv] fp32 or None; cu_seqlens int32 [N+1] or None;
    plus 'N' (sequences), 'T' (tokens per row of the batch) and 'lengths'.
    For varlen, Bt = 1 and T = sum of the lengths.
    """
    seed = default_seed(w) if seed is None else int(seed)
    device = torch.device(device)
    if w.varlen:
        lens = list(lengths) if lengths is not None else varlen_lengths(w, seed)
        Bt, T, N = 1, int(sum(lens)), len(lens)
        cu = torch.zeros(N + 1, dtype=torch.int32)
        cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    else:
        lens = [w.T] * w.B
        Bt, T, N = w.B, w.T, w.B
        cu = None
    gen = torch.Generator(device=device).manual_seed(seed)
    H, dk, dv = w.H, w.dk, w.dv

    def randn(*shape):
        return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)

    def rand(*shape):
        return torch.rand(*shape, generator=gen, device=device, dtype=torch.float32)

    q = _unit_rows(randn(Bt, T, H, dk)).to(w.dtype)
    k = _unit_rows(randn(Bt, T, H, dk)).to(w.dtype)
    v = randn(Bt, T, H, dv).to(w.dtype)
    if w.theta == "normal":
        theta = randn(Bt, T, H, dk).to(w.dtype)
    elif w.theta == "uniform6_12":
        theta = (6.0 + 6.0 * rand(Bt, T, H, dk)).to(w.dtype)
    else:
        raise ValueError(w.theta)
    if w.beta == "sigmoid_normal":
        beta = torch.sigmoid(randn(Bt, T, H)).to(w.dtype)
    elif w.beta == "uniform09_1":
        beta = (0.9 + 0.1 * rand(Bt, T, H)).to(w.dtype)
    else:
        raise ValueError(w.beta)
    init = None
    if w.init_std > 0:
        init = (w.init_std * randn(N, H, dk, dv)).contiguous()
    return dict(q=q, k=k, v=v, theta=theta, beta=beta, init_state=init,
                cu_seqlens=None if cu is None else cu.to(device), N=N, T=T, lengths=lens)
