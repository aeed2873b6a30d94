"""Seeded synthetic inputs for the log-linear Mamba-2 forward and decode.

This module only draws random numbers and casts them; it holds none of the
method's arithmetic.  Both the CUDA path (tests, bench) and the CPU oracle
consume exactly the tensors it returns.

Workloads (shapes follow the kernel benchmark of the log-linear attention
write-up: 48 heads, head dim 64, state 128, chunk 64, two heads per Q/K group,
page 1 section 对Mamba-2和门控的对数线性推广):

* ``tiny``   B=1, H=2 (ungrouped), T=256, d_k=d_v=16, chunk 16, fp32.
* ``small``  B=2, H=8 (4 Q/K groups of 2), T=2048, d_k=128, d_v=64, chunk 64, bf16.
* ``pages``  B=4, H=48 (24 groups), T=8192, d_k=128, d_v=64, chunk 64, bf16.
* ``long``   B=1, H=48, T=131072, otherwise as ``pages``.
* ``decode`` B=64, H=48, prefix T=32768 then 1024 single-token steps.

Distributions:

* q, k, v ~ N(0, 1) * d_k^-1/2.
* ``iid`` decay (tiny, small): a = exp(-softplus(z) * 0.5), z ~ N(0, 1) per (b, t, h).
* ``mamba2`` decay (pages, long, decode): dt = softplus(z - 2), z ~ N(0, 1) per
  (b, t, h); A_log ~ U(0, log 16) per head; a = exp(-min(dt * exp(A_log), 60)).
  The clamp keeps a > 0 in fp32 (a = 0 has no logarithm); it only touches the
  far tail (dt * exp(A_log) > 60 needs z > 5.7).
* ``iid`` lambda (tiny, small): softplus(N(0, 1)) per (b, t, h, level).
* ``linear`` lambda (pages, long, decode): softplus(x W), x ~ N(0, 1) of width
  1536 per (b, t), W ~ N(0, 1/1536) of shape (1536, H * levels), no bias.

Draw order is fixed: q, k, v, decay draws, lambda draws, from one
``torch.Generator`` seeded with ``seed`` on the target device.  Values are drawn
in fp32 and q, k, v are then cast to the workload dtype.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch
import torch.nn.functional as F


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    heads: int
    heads_per_group: int
    T: int
    d_k: int
    d_v: int
    chunk: int
    levels: int
    dtype: torch.dtype
    decay: str  # "iid" | "mamba2" | "ones" | "slow"
    lam: str  # "iid" | "linear" | "ones"
    decode_steps: int = 0

    @property
    def groups(self) -> int:
        return self.heads // self.heads_per_group

    @property
    def T_total(self) -> int:
        return self.T + self.decode_steps


def levels_for(T: int) -> int:
    """ceil(log2 T) + 1: the number of distinct bucket levels a query < T sees."""
    return max(T - 1, 0).bit_length() + 1


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 1, 256, 16, 16, 16, 9, torch.float32, "iid", "iid"),
    "small": Workload("small", 2, 8, 2, 2048, 128, 64, 64, 12, torch.bfloat16, "iid", "iid"),
    "pages": Workload("pages", 4, 48, 2, 8192, 128, 64, 64, 14, torch.bfloat16, "mamba2", "linear"),
    "long": Workload("long", 1, 48, 2, 131072, 128, 64, 64, 18, torch.bfloat16, "mamba2", "linear"),
    "decode": Workload("decode", 64, 48, 2, 32768, 128, 64, 64, 17, torch.bfloat16, "mamba2",
                       "linear", decode_steps=1024),
}


def workload(name: str, **overrides) -> Workload:
    w = WORKLOADS[name]
    return replace(w, **overrides) if overrides else w


@dataclass
class Inputs:
    q: torch.Tensor  # (B, T, G, d_k)
    k: torch.Tensor  # (B, T, G, d_k)
    v: torch.Tensor  # (B, T, H, d_v)
    a: torch.Tensor  # (B, T, H) fp32
    lam: torch.Tensor  # (B, T, H, levels) fp32


def _normal(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)


def make_inputs(w: Workload, device="cpu", seed: int = 0, T: int | None = None) -> Inputs:
    """Draw the inputs of workload ``w`` for T tokens (default: prefix plus decode steps)."""
    T = w.T_total if T is None else T
    B, H, G = w.batch, w.heads, w.groups
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    sc = w.d_k ** -0.5
    q = (_normal((B, T, G, w.d_k), gen, device) * sc).to(w.dtype)
    k = (_normal((B, T, G, w.d_k), gen, device) * sc).to(w.dtype)
    v = (_normal((B, T, H, w.d_v), gen, device) * sc).to(w.dtype)
    if w.decay == "iid":
        a = torch.exp(-F.softplus(_normal((B, T, H), gen, device)) * 0.5)
    elif w.decay == "mamba2":
        dt = F.softplus(_normal((B, T, H), gen, device) - 2.0)
        a_log = torch.rand((H,), generator=gen, device=device) * math.log(16.0)
        a = torch.exp(-torch.clamp(dt * torch.exp(a_log), max=60.0))
    elif w.decay == "slow":
        a = torch.exp(-F.softplus(_normal((B, T, H), gen, device)) * 1e-3)
    elif w.decay == "ones":
        a = torch.ones((B, T, H), device=device)
    else:
        raise ValueError(w.decay)
    L = w.levels
    if w.lam == "iid":
        lam = F.softplus(_normal((B, T, H, L), gen, device))
    elif w.lam == "linear":
        W = _normal((1536, H * L), gen, device) / math.sqrt(1536.0)
        lam = torch.empty((B, T, H, L), device=device, dtype=torch.float32)
        step = max(1, (1 << 22) // 1536)
        for b in range(B):
            for t0 in range(0, T, step):
                t1 = min(T, t0 + step)
                x = _normal((t1 - t0, 1536), gen, device)
                lam[b, t0:t1] = F.softplus(x @ W).view(t1 - t0, H, L)
    elif w.lam == "ones":
        lam = torch.ones((B, T, H, L), device=device)
    else:
        raise ValueError(w.lam)
    return Inputs(q.contiguous(), k.contiguous(), v.contiguous(), a.contiguous().float(),
                  lam.contiguous().float())


def to_numpy64(x: torch.Tensor):
    """Exact fp64 copy of a (possibly bf16) tensor, for the oracle."""
    return x.detach().to("cpu", torch.float64).numpy()
