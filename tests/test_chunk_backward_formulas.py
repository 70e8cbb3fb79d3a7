"""The chunkwise reverse-mode formulas that the backward kernels evaluate, written out plainly in
fp64 numpy (explicit pairwise decays, explicit inverse) and compared with the autograd gradients
of the token-by-token oracle (CPU).

Forward of one chunk (Kimi K3 report walk-through, section 2.5 / Eq. 4), with chunk-start state S0
and G the chunk's inclusive cumulative log-decay, E_rs = e^{G_r - G_s} (per key channel):
  A~_rs = sum_c k_rc k_sc E_rs,c (s < r),  A = Diag(beta) A~,  X = (I + A)^-1,  T = X Diag(beta),
  K^ = K e^G,  Q^ = Q e^G,  K_ = K e^{G_C - G},  W = T K^,  U^ = T V,  U = U^ - W S0,
  M_rs = sum_c q_rc k_sc E_rs,c (s <= r),  O = Q^ S0 + M U,  S_C = Diag(e^{G_C}) S0 + K_^T U.
Reverse, given dO and dS_C: every step below is the transpose of one line above."""
import numpy as np
import torch

from oracle import oracle_kda_backward

C = 8


def _inputs(T, dk, dv, seed):
    gen = torch.Generator().manual_seed(seed)
    n = lambda *s: torch.randn(*s, generator=gen, dtype=torch.float64)
    q = torch.nn.functional.normalize(n(T, 1, dk), dim=-1)
    k = torch.nn.functional.normalize(n(T, 1, dk), dim=-1)
    v = n(T, 1, dv)
    g = -5.0 * torch.sigmoid(n(T, 1, dk) - 1.0)
    beta = torch.sigmoid(n(T, 1))
    h0 = 0.1 * n(1, 1, dk, dv)
    dout = n(T, 1, dv)
    dhT = n(1, 1, dk, dv)
    return q, k, v, g, beta, h0, dout, dhT


def _chunks(x, T):
    """[T, ...] -> list of [C, ...] chunks, the tail padded with zeros (identity tokens)."""
    nc = -(-T // C)
    pad = np.zeros((nc * C,) + x.shape[1:])
    pad[:T] = x
    return [pad[i * C:(i + 1) * C] for i in range(nc)]


def _forward_chunk(q, k, v, g, b, S0):
    G = np.cumsum(g, axis=0)
    E = np.exp(G[:, None, :] - G[None, :, :])                      # [r, s, c]
    strict = np.tril(np.ones((C, C)), -1)
    At = np.einsum("rc,sc,rsc->rs", k, k, E) * strict
    A = b[:, None] * At
    X = np.linalg.inv(np.eye(C) + A)
    T = X * b[None, :]
    Kh, Qh, Kb = k * np.exp(G), q * np.exp(G), k * np.exp(G[-1] - G)
    W, Uh = T @ Kh, T @ v
    U = Uh - W @ S0
    M = np.einsum("rc,sc,rsc->rs", q, k, E) * np.tril(np.ones((C, C)))
    O = Qh @ S0 + M @ U
    SC = np.exp(G[-1])[:, None] * S0 + Kb.T @ U
    return dict(G=G, E=E, At=At, X=X, T=T, Kh=Kh, Qh=Qh, Kb=Kb, W=W, U=U, M=M, O=O, SC=SC)


def _backward_chunk(q, k, v, b, S0, f, dO, dSC):
    G, E, At, X, T = f["G"], f["E"], f["At"], f["X"], f["T"]
    Kh, Qh, Kb, W, U, M = f["Kh"], f["Qh"], f["Kb"], f["W"], f["U"], f["M"]
    dU = M.T @ dO + Kb @ dSC
    dS0 = Qh.T @ dO + np.exp(G[-1])[:, None] * dSC - W.T @ dU
    dQh, dM = dO @ S0.T, (dO @ U.T) * np.tril(np.ones((C, C)))
    dKb, dW = U @ dSC.T, -dU @ S0.T
    dT = dU @ v.T + dW @ Kh.T
    dKh, dv = T.T @ dW, T.T @ dU
    dbeta = np.einsum("rs,rs->s", X, dT)                            # T = X Diag(beta)
    dX = dT * b[None, :]
    dA = -(X.T @ dX @ X.T) * np.tril(np.ones((C, C)), -1)          # X = (I + A)^-1, A strictly lower
    dbeta = dbeta + np.einsum("rs,rs->r", dA, At)                   # A = Diag(beta) A~
    P = b[:, None] * dA
    s1 = np.einsum("rs,sc,rsc->rc", P, k, E)                        # sum_s P_rs k_s E_rs
    s2 = np.einsum("ar,ac,arc->rc", P, k, E)                        # sum_r' P_r'r k_r' E_r'r
    s3 = np.einsum("rs,sc,rsc->rc", dM, k, E)                       # sum_s dM_rs k_s E_rs
    s4 = np.einsum("ar,ac,arc->rc", dM, q, E)                       # sum_r' dM_r'r q_r' E_r'r
    dq = s3 + dQh * np.exp(G)
    dk = s1 + s2 + s4 + dKh * np.exp(G) + dKb * np.exp(G[-1] - G)
    dG = k * (s1 - s2) + q * s3 - k * s4 + dQh * Qh + dKh * Kh - dKb * Kb
    dG[-1] += (dKb * Kb).sum(axis=0) + np.exp(G[-1]) * (dSC * S0).sum(axis=1)
    dg = np.cumsum(dG[::-1], axis=0)[::-1]                          # G_r = sum_{s <= r} g_s
    return dq, dk, dv, dg, dbeta, dS0


def _chunkwise_gradients(q, k, v, g, beta, h0, dout, dhT):
    T = q.shape[0]
    cq, ck, cv, cg, cb, cd = (_chunks(x, T) for x in (q, k, v, g, beta, dout))
    S, fwd = h0, []
    for i in range(len(cq)):  # forward over chunks, keeping each chunk's start state
        f = _forward_chunk(cq[i], ck[i], cv[i], cg[i], cb[i], S)
        fwd.append((S, f))
        S = f["SC"]
    grads = [None] * len(cq)
    dS = dhT
    for i in reversed(range(len(cq))):  # reverse over chunks, carrying dS
        S0, f = fwd[i]
        *gi, dS = _backward_chunk(cq[i], ck[i], cv[i], cb[i], S0, f, cd[i], dS)
        grads[i] = gi
    cat = [np.concatenate([gr[j] for gr in grads])[:T] for j in range(5)]
    return (*cat, dS)


def test_chunkwise_reverse_mode_equals_autograd_with_a_ragged_tail():
    for seed, T in ((0, 20), (1, 8), (2, 3)):
        dk, dv = 5, 4
        q, k, v, g, beta, h0, dout, dhT = _inputs(T, dk, dv, seed)
        ref = oracle_kda_backward(q, k, v, g, beta, dout, h0=h0, dhT=dhT)
        ours = _chunkwise_gradients(q[:, 0].numpy(), k[:, 0].numpy(), v[:, 0].numpy(), g[:, 0].numpy(),
                                    beta[:, 0].numpy(), h0[0, 0].numpy(), dout[:, 0].numpy(), dhT[0, 0].numpy())
        names = ("dq", "dk", "dv", "dg", "dbeta", "dh0")
        for name, r, o in zip(names, ref, ours):
            r = r[0, 0] if name == "dh0" else r[:, 0]
            assert np.abs(r - o).max() <= 1e-10 * max(1.0, np.abs(r).max()), (seed, name)
