"""Pins of the gradient oracle (CPU): its forward is the C oracle's, its gradients are the
finite-difference ones."""
import numpy as np
import torch

from oracle import oracle_kda_backward, oracle_kda_prefill, recurrence_torch


def _inputs(T, H, dk, dv, B=1, seed=0):
    gen = torch.Generator().manual_seed(seed)
    n = lambda *s: torch.randn(*s, generator=gen, dtype=torch.float64)
    q = torch.nn.functional.normalize(n(T, H, dk), dim=-1)
    k = torch.nn.functional.normalize(n(T, H, dk), dim=-1)
    v = n(T, H, dv)
    g = -5.0 * torch.sigmoid(n(T, H, dk))
    beta = torch.sigmoid(n(T, H))
    h0 = 0.1 * n(B, H, dk, dv)
    return q, k, v, g, beta, h0


def test_forward_equals_the_c_oracle():
    q, k, v, g, beta, h0 = _inputs(37, 2, 5, 4, B=2, seed=1)
    cu = torch.tensor([0, 15, 37])
    out, hT = recurrence_torch(q, k, v, g, beta, h0=h0, cu_seqlens=cu)
    ro, rh = oracle_kda_prefill(q, k, v, g, beta, h0=h0, cu_seqlens=cu)
    assert np.abs(out.numpy() - ro).max() < 1e-12 and np.abs(hT.numpy() - rh).max() < 1e-12


def test_gradients_match_finite_differences():
    q, k, v, g, beta, h0 = _inputs(5, 1, 3, 2, seed=2)
    gen = torch.Generator().manual_seed(3)
    dout = torch.randn(5, 1, 2, generator=gen, dtype=torch.float64)
    dhT = torch.randn(1, 1, 3, 2, generator=gen, dtype=torch.float64)

    def loss(q, k, v, g, beta, h0):
        out, hT = recurrence_torch(q, k, v, g, beta, h0=h0)
        return (out * dout).sum() + (hT * dhT).sum()

    args = tuple(x.clone().requires_grad_(True) for x in (q, k, v, g, beta, h0))
    assert torch.autograd.gradcheck(loss, args, eps=1e-6, atol=1e-7, rtol=1e-5)
    # and oracle_kda_backward returns those gradients
    grads = torch.autograd.grad(loss(*args), args)
    ours = oracle_kda_backward(q, k, v, g, beta, dout, h0=h0, dhT=dhT)
    for a, b in zip(grads, ours):
        assert np.abs(a.numpy() - b).max() < 1e-12


def test_gradient_of_the_read_out_alone_is_the_state():
    """With beta = 0 and g = 0 the state is constant (S = h0) and o_t = h0^T q_t, so
    dL/dq_t = h0 dout_t exactly."""
    q, k, v, g, beta, h0 = _inputs(4, 2, 3, 5, seed=4)
    g = torch.zeros_like(g)
    beta = torch.zeros_like(beta)
    dout = torch.randn(4, 2, 5, dtype=torch.float64)
    dq = oracle_kda_backward(q, k, v, g, beta, dout, h0=h0)[0]
    expect = torch.einsum("hij,thj->thi", h0[0], dout).numpy()
    assert np.abs(dq - expect).max() < 1e-12


def test_no_write_gradients_in_closed_form():
    """With beta = 0 the state is S_t = Diag(prod_{s<=t} exp g_s) h0, so k and v get no gradient
    and dL/dh0 = sum_t Diag(prod_{s<=t} exp g_s) q_t dout_t^T + Diag(prod_all exp g) dhT; dL/dbeta
    is the only path through k and v, and is not zero."""
    q, k, v, g, beta, h0 = _inputs(6, 2, 3, 4, seed=5)
    beta = torch.zeros_like(beta)
    gen = torch.Generator().manual_seed(6)
    dout = torch.randn(6, 2, 4, generator=gen, dtype=torch.float64)
    dhT = torch.randn(1, 2, 3, 4, generator=gen, dtype=torch.float64)
    dq, dk, dv, dg, dbeta, dh0 = oracle_kda_backward(q, k, v, g, beta, dout, h0=h0, dhT=dhT)
    assert np.abs(dk).max() == 0.0 and np.abs(dv).max() == 0.0
    assert np.abs(dbeta).max() > 1e-6
    cum = torch.exp(torch.cumsum(g, dim=0))  # [T, H, dk]: prod_{s<=t} exp g_s, per key channel
    expect = torch.einsum("thi,thi,thj->hij", cum, q, dout) + cum[-1][:, :, None] * dhT[0]
    assert np.abs(dh0[0] - expect.numpy()).max() < 1e-12
