"""The decode step's rearrangement (CPU, fp64): the kernel never re-reads the updated state for the
read-out.  With S' = Diag(exp g) S, a = S'^T k, b = S'^T q and delta = beta (v - a):
  S_new = S' + k delta^T   equals   (I - beta k k^T) Diag(exp g) S + beta k v^T   (Eq. 1), and
  o = b + (k . q) delta    equals   S_new^T q                                      (Eq. 3)
(Kimi K3 report walk-through, sections 2.2 and 2.4); checked here against the oracle's step."""
import numpy as np
import torch

from oracle import oracle_kda_decode


def test_rank_one_form_of_the_step_and_its_read_out():
    rng = np.random.default_rng(3)
    N, H, dk, dv = 5, 3, 8, 6
    q = rng.standard_normal((N, H, dk))
    k = rng.standard_normal((N, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((N, H, dv))
    g = -5.0 / (1.0 + np.exp(-rng.standard_normal((N, H, dk))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((N, H))))
    S = 0.1 * rng.standard_normal((N, H, dk, dv))

    Sp = np.exp(g)[..., None] * S
    a = np.einsum("nhij,nhi->nhj", Sp, k)
    b = np.einsum("nhij,nhi->nhj", Sp, q)
    delta = beta[..., None] * (v - a)
    S_new = Sp + k[..., None] * delta[..., None, :]
    o = b + np.einsum("nhi,nhi->nh", k, q)[..., None] * delta

    assert np.abs(o - np.einsum("nhij,nhi->nhj", S_new, q)).max() < 1e-13
    t = lambda x: torch.from_numpy(x)
    ro, rpool, _ = oracle_kda_decode(t(q), t(k), t(v), t(g), t(beta), t(S), np.arange(N))
    assert np.abs(ro - o).max() < 1e-12 and np.abs(rpool - S_new).max() < 1e-12
