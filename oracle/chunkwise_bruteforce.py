"""Brute-force fp64 chunkwise (Eq. 4) evaluation of KDA, for pinning only.

TEST INFRASTRUCTURE (see the package docstring).  This is a second, independent
route to the same numbers as the token-by-token recurrence: the sequence is cut
into chunks of C tokens (counted from the start of the sequence); inside a chunk
everything is dense linear algebra with explicit pairwise decays
exp(G_r - G_s) and an explicit matrix inverse, and only the chunk-boundary
state is carried serially.  It is meant for tiny inputs (the pairwise decay
tensor is C x C x dk).

Derivation (Kimi K3 report walk-through, section 2.5, Eq. 4: an inter-chunk
term Gamma * Q * S[t] that is serial and an intra-chunk causal dense term
A[t] * V_hat[t]).  Within one chunk, positions r = 1..n, chunk-start state S0,
G_r = sum_{s<=r} g_s (per key channel), Gamma_r = exp(G_r):
    u_r  = beta_r (v_r - S_{r-1}^T Diag(alpha_r) k_r)     (the delta of token r)
    S_r  = Diag(Gamma_r) S0 + sum_{s<=r} Diag(Gamma_r / Gamma_s) k_s u_s^T
  =>  (I + A) U = Diag(beta) (V - K_hat S0),
      A_rs = beta_r sum_c k_rc k_sc exp(G_rc - G_sc)   for s < r (0 otherwise)
      K_hat_r = k_r * Gamma_r
  =>  U = T V - T K_hat S0 with T = (I + A)^{-1} Diag(beta)
      O = Q_hat S0 + M U,   Q_hat_r = q_r * Gamma_r,
      M_rs = sum_c q_rc k_sc exp(G_rc - G_sc)          for s <= r
      S_n = Diag(Gamma_n) S0 + K_bar^T U,   K_bar_s = k_s * Gamma_n / Gamma_s
"""
from __future__ import annotations

import numpy as np


def chunkwise_chain(q, k, v, g, beta, S0, C: int):
    """One (sequence, head) chain.  q, k, g: [T, dk]; v: [T, dv]; beta: [T];
    S0: [dk, dv].  Returns (out [T, dv], S_T [dk, dv]) in fp64."""
    q, k, v, g, beta, S = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta, S0))
    S = S.copy()
    T = q.shape[0]
    out = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, C):
        sl = slice(c0, min(c0 + C, T))
        Q, K, V, b = q[sl], k[sl], v[sl], beta[sl]
        n = Q.shape[0]
        G = np.cumsum(g[sl], axis=0)                       # [n, dk], inclusive
        D = np.exp(G[:, None, :] - G[None, :, :])          # [n, n, dk] pairwise decay
        A = np.tril(np.einsum("rc,sc,rsc->rs", K, K, D), -1) * b[:, None]
        M = np.tril(np.einsum("rc,sc,rsc->rs", Q, K, D))
        Tm = np.linalg.inv(np.eye(n) + A) @ np.diag(b)
        K_hat = K * np.exp(G)
        Q_hat = Q * np.exp(G)
        K_bar = K * np.exp(G[-1][None, :] - G)
        U = Tm @ V - (Tm @ K_hat) @ S
        out[sl] = Q_hat @ S + M @ U
        S = np.exp(G[-1])[:, None] * S + K_bar.T @ U
    return out, S


def chunkwise_prefill(q, k, v, g, beta, h0=None, cu_seqlens=None, C: int = 64):
    """Packed batch, same layouts as the recurrence oracle (no epilogue)."""
    q, k, v, g, beta = (np.asarray(x, dtype=np.float64) for x in (q, k, v, g, beta))
    T_tot, H, dk = q.shape
    dv = v.shape[2]
    cu = np.array([0, T_tot]) if cu_seqlens is None else np.asarray(cu_seqlens, dtype=np.int64)
    B = len(cu) - 1
    out = np.zeros((T_tot, H, dv))
    hT = np.zeros((B, H, dk, dv))
    for b in range(B):
        a, e = int(cu[b]), int(cu[b + 1])
        for h in range(H):
            S0 = np.zeros((dk, dv)) if h0 is None else np.asarray(h0, dtype=np.float64)[b, h]
            if e > a:
                o, S = chunkwise_chain(q[a:e, h], k[a:e, h], v[a:e, h], g[a:e, h], beta[a:e, h], S0, C)
                out[a:e, h] = o
            else:
                S = S0.copy()
            hT[b, h] = S
    return out, hT
