"""Checks that pin a KDA prefill implementation to facts other than itself.

Each ``check_*`` takes ``prefill(q, k, v, g, beta, h0, cu_seqlens) -> (out, hT)``
(fp64 numpy in and out, layouts as the oracle) and returns the worst error it
saw.  The tests apply them to the fp64 oracle (all must pass) and to planted
mutants of a small recurrence (each mutant must fail at least one), which shows
that the set of pins catches the plausible mistakes: a dropped term, a wrong
sign or order, a transposed operand.

What pins what (Kimi K3 report walk-through, kimi-k3-paper.pages.dev):
  - hand-derived 2x2 example (tests/golden/hand_2x2.json): Eq. 1 of section 2.2
    evaluated by hand in exact decimals: decay rows, then erase, then write.
  - beta = 0: S_t = Diag(prod_s alpha_s) S_0 exactly (decay only, section 2.3).
  - |k| = 1, beta = 1: the delta rule overwrites the value stored under k,
    S_t^T k_t = v_t (section 2.2, "subtract the overlap, then write").
  - the delta rule is one gradient step of size beta on 1/2 |S^T k - v|^2 taken
    from the decayed state (the textbook online-regression reading of the
    delta rule), checked with torch.autograd.
  - chunkwise form (section 2.5, Eq. 4) with any chunk size == recurrence.
  - linearity in (V, S_0) and independence of the value columns.
"""
from __future__ import annotations

import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rand_inputs(rng, T, H, dk, dv, *, beta=None, g_scale=5.0, unit_k=True, B=1):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit_k:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    g = -g_scale / (1.0 + np.exp(-rng.standard_normal((T, H, dk))))
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H)))) if beta is None else np.full((T, H), float(beta))
    h0 = rng.standard_normal((B, H, dk, dv)) * 0.5
    return q, k, v, g, b, h0


def _cu(T):
    return np.array([0, T], dtype=np.int64)


def check_hand_example(prefill):
    with open(os.path.join(GOLDEN, "hand_2x2.json")) as f:
        ex = json.load(f)
    arr = {key: np.asarray(ex[key], dtype=np.float64) for key in
           ("q", "k", "v", "g", "beta", "h0", "out", "hT")}
    out, hT = prefill(arr["q"], arr["k"], arr["v"], arr["g"], arr["beta"], arr["h0"], _cu(arr["q"].shape[0]))
    return max(np.abs(out - arr["out"]).max(), np.abs(hT - arr["hT"]).max())


def check_beta_zero(prefill, seed=1):
    rng = np.random.default_rng(seed)
    T, H, dk, dv = 40, 2, 6, 5
    q, k, v, g, _, h0 = rand_inputs(rng, T, H, dk, dv)
    beta = np.zeros((T, H))
    out, hT = prefill(q, k, v, g, beta, h0, _cu(T))
    err = 0.0
    for h in range(H):
        decay = np.cumprod(np.exp(g[:, h, :]), axis=0)           # [T, dk]
        S_t = decay[:, :, None] * h0[0, h][None, :, :]            # [T, dk, dv]
        o_ref = np.einsum("tij,ti->tj", S_t, q[:, h, :])
        err = max(err, np.abs(out[:, h] - o_ref).max() / np.abs(o_ref).max())
        err = max(err, np.abs(hT[0, h] - S_t[-1]).max() / np.abs(S_t[-1]).max())
    return err


def check_overwrite(prefill, seed=2):
    rng = np.random.default_rng(seed)
    T, H, dk, dv = 30, 2, 7, 4
    q, k, v, g, _, h0 = rand_inputs(rng, T, H, dk, dv)
    beta = np.ones((T, H))
    out, _ = prefill(k.copy(), k, v, g, beta, h0, _cu(T))     # read with q_t = k_t
    return np.abs(out - v).max()


def check_gradient_step(prefill, seed=3):
    """One token: S_1 = S' - beta * dL/dS' with L = 1/2 |S'^T k - v|^2, S' = Diag(alpha) S_0."""
    import torch
    rng = np.random.default_rng(seed)
    dk, dv = 5, 3
    q, k, v, g, b, h0 = rand_inputs(rng, 1, 1, dk, dv)
    _, hT = prefill(q, k, v, g, b, h0, _cu(1))
    Sp = torch.tensor(np.exp(g[0, 0])[:, None] * h0[0, 0], dtype=torch.float64, requires_grad=True)
    kt = torch.tensor(k[0, 0], dtype=torch.float64)
    vt = torch.tensor(v[0, 0], dtype=torch.float64)
    loss = 0.5 * ((Sp.T @ kt - vt) ** 2).sum()
    (grad,) = torch.autograd.grad(loss, Sp)
    S1 = (Sp - float(b[0, 0]) * grad).detach().numpy()
    return np.abs(hT[0, 0] - S1).max()


def check_chunkwise(prefill, chunkwise, seed=4, T=24, dk=5, dv=3):
    """Chunkwise brute force for every chunk size 1..T against ``prefill``."""
    rng = np.random.default_rng(seed)
    q, k, v, g, b, h0 = rand_inputs(rng, T, 1, dk, dv)
    out, hT = prefill(q, k, v, g, b, h0, _cu(T))
    err = 0.0
    for C in range(1, T + 1):
        o2, h2 = chunkwise(q, k, v, g, b, h0, _cu(T), C)
        err = max(err, np.abs(out - o2).max(), np.abs(hT - h2).max())
    return err


def check_linearity(prefill, seed=5):
    rng = np.random.default_rng(seed)
    T, H, dk, dv = 20, 1, 4, 3
    q, k, v1, g, b, h01 = rand_inputs(rng, T, H, dk, dv)
    v2 = rng.standard_normal(v1.shape)
    h02 = rng.standard_normal(h01.shape)
    o1, s1 = prefill(q, k, v1, g, b, h01, _cu(T))
    o2, s2 = prefill(q, k, v2, g, b, h02, _cu(T))
    o3, s3 = prefill(q, k, v1 + 2 * v2, g, b, h01 + 2 * h02, _cu(T))
    return max(np.abs(o3 - (o1 + 2 * o2)).max(), np.abs(s3 - (s1 + 2 * s2)).max())


def check_column_split(prefill, seed=6):
    """Running each value column alone and stacking == running all columns."""
    rng = np.random.default_rng(seed)
    T, H, dk, dv = 18, 1, 4, 3
    q, k, v, g, b, h0 = rand_inputs(rng, T, H, dk, dv)
    out, hT = prefill(q, k, v, g, b, h0, _cu(T))
    err = 0.0
    for j in range(dv):
        oj, sj = prefill(q, k, v[:, :, j:j + 1], g, b, h0[:, :, :, j:j + 1], _cu(T))
        err = max(err, np.abs(oj[..., 0] - out[..., j]).max(), np.abs(sj[..., 0] - hT[..., j]).max())
    return err


ALL_CHECKS = ("hand_example", "beta_zero", "overwrite", "gradient_step", "chunkwise", "linearity",
              "column_split")
