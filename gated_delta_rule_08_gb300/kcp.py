"""Context parallelism across devices for one long sequence (KCP).

Kimi K3: Open Frontier Intelligence (kimi-k3-paper.pages.dev), section 13.3.2, and the open-day
article (mlqm.cn), section 5.2: the sequence is cut into consecutive token ranges, one per rank.
Over its range each rank's state pass is affine in the range's initial state, S_out = P S_in + b
(P: the range's accumulated transition; b: its final state from a zero state).  The ranks
all-gather these fixed-size maps (one message of H * dk * (dk + dv) fp32 values per rank), each
rank folds the maps of the ranges before its own into its initial state, and then runs the
ordinary prefill on its range from that state.

All arithmetic runs in libkda on the rank's GPU (kda_chunk_fwd_segment_map, kda_state_compose,
kda_chunk_fwd); this module only moves the maps between ranks with torch.distributed (NCCL between
GPUs).  Ranks hold the ranges in rank order of the process group.
"""
from __future__ import annotations

from typing import Optional

import torch
import torch.distributed as dist

from . import binding


def exchange_segment_maps(P: torch.Tensor, b: torch.Tensor, group=None):
    """All-gather every rank's map.  P: [H, dk, dk], b: [H, dk, dv] (same shapes on every rank).
    Returns (Ps [world, H, dk, dk], bs [world, H, dk, dv]) in rank order.  The two tensors travel
    as one fixed-size message per rank."""
    world = dist.get_world_size(group)
    H, dk, _ = P.shape
    dv = b.shape[2]
    msg = torch.cat([P.reshape(H, dk, dk), b.reshape(H, dk, dv)], dim=2).contiguous()
    parts = [torch.empty_like(msg) for _ in range(world)]
    dist.all_gather(parts, msg, group=group)
    allm = torch.stack(parts)
    return allm[..., :dk].contiguous(), allm[..., dk:].contiguous()


def kcp_chunk_fwd(q, k, v, g, beta, h0: Optional[torch.Tensor] = None, group=None, **fwd_kw):
    """Prefill of this rank's range of one sequence split across the ranks of `group`.
    q, k: [T_r, H, dk]; v: [T_r, H, dv]; g: [T_r, H, dk] fp32; beta: [T_r, H] fp32 (this rank's
    tokens); h0: [1, H, dk, dv] fp32 initial state of the whole sequence, or None (zero), the same
    on every rank.  Other keywords go to kda_chunk_fwd (gate, norm_weight, eps, out, out_dtype).
    Returns (out [T_r, H, dv], the state after this rank's range [1, H, dk, dv]); on the last rank
    that is the sequence's final state."""
    rank = dist.get_rank(group)
    P, b = binding.kda_chunk_fwd_segment_map(k, v, g, beta)
    Ps, bs = exchange_segment_maps(P, b, group)
    S0 = None if h0 is None else h0.reshape(h0.shape[-3:]).contiguous()
    S_in = binding.kda_state_compose(Ps[:rank].contiguous(), bs[:rank].contiguous(), S0=S0)
    out, hT = binding.kda_chunk_fwd(q, k, v, g, beta, h0=S_in.unsqueeze(0), **fwd_kw)
    return out, hT
