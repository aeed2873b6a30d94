"""Sequence-sharded log-linear Mamba-2 forward: rank r of a group holds the tokens
[r*T, (r+1)*T) of every sequence (T a power of two, the same on every rank).

Every bucket of a position in rank r's segment lies either inside the segment or before
r*T, where it is one of the buckets of r*T, and each of those is made of whole earlier
segments (log-linear attention write-up, https://www.yoousoft.com/industry/3746.html,
section 特殊结构：树划分, Fig. 2; memories of pieces combined level by level, section
高效训练算法, Algorithm 1).  So the forward needs a single exchange:

1. each rank computes its segment's memory and summed log-decay (loglinear_segment_total);
2. one all-gather of those (B*H*d_k*d_v + B*H floats per rank);
3. each rank builds the bucket memories at its start from the segments before it
   (loglinear_prefix_states) and runs the forward that continues from them
   (loglinear_fwd_continue).

This module only moves data between ranks and calls the library; every arithmetic step
runs in the library's kernels.  Over a gloo group the gathered tensors travel through
host memory; over NCCL they stay on the device.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


class LibraryBackend:
    """The library's entry points (the default backend)."""

    def segment_total(self, k, v, a, chunk):
        from . import loglinear_segment_total

        return loglinear_segment_total(k, v, a, chunk=chunk)

    def prefix_states(self, seg_states, seg_logdecay, seg_len, levels):
        from . import loglinear_prefix_states

        return loglinear_prefix_states(seg_states, seg_logdecay, seg_len, levels)

    def fwd_continue(self, q, k, v, a, lam, T0, prefix_states, prefix_logscale, chunk):
        from . import loglinear_fwd_continue

        return loglinear_fwd_continue(q, k, v, a, lam, T0, prefix_states, prefix_logscale, chunk=chunk)


def _all_gather(t: torch.Tensor, world: int, group) -> list[torch.Tensor]:
    """All-gather of one tensor per rank; through host memory when the group's backend
    cannot take device tensors (gloo)."""
    host = t.is_cuda and dist.get_backend(group) == "gloo"
    src = t.cpu() if host else t.contiguous()
    out = [torch.empty_like(src) for _ in range(world)]
    dist.all_gather(out, src, group=group)
    return [x.to(t.device) for x in out] if host else out


def sharded_forward(q, k, v, a, lam, chunk: int = 64, group=None, backend=None):
    """The output of this rank's segment.  q, k: (B, T, G, d_k); v: (B, T, H, d_v);
    a: (B, T, H); lam: (B, T, H, L) with absolute levels (L >= bit_length(world*T - 1) + 1)."""
    be = backend or LibraryBackend()
    rank = dist.get_rank(group)
    world = dist.get_world_size(group)
    T = q.shape[1]
    if T < 1 or T & (T - 1):
        raise ValueError(f"the segment length must be a power of two, got {T}")
    if world > 64:
        raise ValueError("at most 64 segments")
    total, logdecay = be.segment_total(k, v, a, chunk)
    states = _all_gather(total, world, group)
    decays = _all_gather(logdecay, world, group)
    T0 = rank * T
    if rank == 0:
        return be.fwd_continue(q, k, v, a, lam, 0, None, None, chunk)
    levels = T0.bit_length() + 1
    pst, plsc = be.prefix_states(torch.stack(states[:rank]), torch.stack(decays[:rank]), T, levels)
    return be.fwd_continue(q, k, v, a, lam, T0, pst, plsc, chunk)
