"""Gradient oracle for the KDA recurrence — TEST INFRASTRUCTURE.

Only tests/, __graft_entry__.smoke() and bench.py's CPU baseline may use anything under oracle/;
the CUDA path never does.

A plain fp64 PyTorch restatement of the per-token recurrence, differentiated by
torch.autograd.  It follows the same steps as oracle/kda_oracle.c, in the same order:
  Kimi K3: Open Frontier Intelligence (kimi-k3-paper.pages.dev), section 2.2 Eq. 1
    S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T   (decay, erase, write)
  section 2.4 Eq. 3
    o_t = S_t^T q_t
and gives the gradients of  L = sum_t <dout_t, o_t> + <dhT, hT>.  Pinned by the CPU tests against
the C oracle's forward (same outputs to 1e-12) and against finite differences
(torch.autograd.gradcheck).  Token loops in Python: small problems only.
"""
from __future__ import annotations

import numpy as np
import torch


def _f64(x):
    if x is None:
        return None
    if isinstance(x, np.ndarray):
        return torch.from_numpy(x).double()
    return x.detach().to("cpu").double()


def recurrence_torch(q, k, v, g, beta, h0=None, cu_seqlens=None):
    """fp64 forward with autograd.  q, k, g: [T_tot, H, dk]; v: [T_tot, H, dv]; beta: [T_tot, H];
    h0: [B, H, dk, dv] or None; cu_seqlens: [B+1] or None (one sequence).
    Returns (out [T_tot, H, dv], hT [B, H, dk, dv])."""
    T_tot, H, dk = q.shape
    dv = v.shape[2]
    cu = [0, T_tot] if cu_seqlens is None else [int(x) for x in cu_seqlens]
    B = len(cu) - 1
    outs, finals = [], []
    for b in range(B):
        S = h0[b] if h0 is not None else torch.zeros(H, dk, dv, dtype=q.dtype)
        for t in range(cu[b], cu[b + 1]):
            S = torch.exp(g[t]).unsqueeze(-1) * S                                 # decay rows
            S = S - beta[t].view(H, 1, 1) * k[t].unsqueeze(-1) * torch.einsum("hi,hij->hj", k[t], S).unsqueeze(1)  # erase
            S = S + beta[t].view(H, 1, 1) * k[t].unsqueeze(-1) * v[t].unsqueeze(1)  # write
            outs.append(torch.einsum("hij,hi->hj", S, q[t]))                       # read
        finals.append(S)
    out = torch.stack(outs) if outs else torch.zeros(0, H, dv, dtype=q.dtype)
    return out, torch.stack(finals)


def oracle_kda_backward(q, k, v, g, beta, dout, h0=None, cu_seqlens=None, dhT=None):
    """Gradients (dq, dk, dv, dg, dbeta, dh0) of sum <dout, out> + <dhT, hT>, as fp64 numpy arrays
    (dh0 is None when h0 is None)."""
    args = [_f64(x) for x in (q, k, v, g, beta)]
    for a in args:
        a.requires_grad_(True)
    h = _f64(h0)
    if h is not None:
        h.requires_grad_(True)
    cu = None if cu_seqlens is None else [int(x) for x in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist")
                                                         else cu_seqlens)]
    out, hT = recurrence_torch(*args, h0=h, cu_seqlens=cu)
    loss = (out * _f64(dout)).sum()
    if dhT is not None:
        loss = loss + (hT * _f64(dhT)).sum()
    wrt = args + ([h] if h is not None else [])
    grads = torch.autograd.grad(loss, wrt, allow_unused=True)
    res = [gr.numpy() if gr is not None else np.zeros(a.shape) for gr, a in zip(grads, wrt)]
    if h is None:
        res.append(None)
    return tuple(res)
