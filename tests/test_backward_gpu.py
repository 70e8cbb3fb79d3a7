"""Backward of the prefill recurrence on the GPU vs the fp64 autograd oracle (through the C-ABI)."""
import numpy as np
import pytest
import torch

from gated_delta_rule_08_gb300 import binding, inputs
from gpu_util import assert_no_device_error, rel_err
from oracle import oracle_kda_backward

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["chunked", "token"])
def path(request, monkeypatch):
    """Both backward paths (the library picks the token sweep only beyond 48 GB of chunkwise scratch)."""
    monkeypatch.setenv("KDA_BACKWARD_PATH", request.param)
    return request.param

# the backward runs in fp32 on the given inputs whatever their dtype: the fp32 bound applies
TOL = 1e-3


def _case(lengths, H, dk, dv, dtype, h0, dhT, seed):
    cfg = inputs.PrefillConfig("bwd", H=H, dk=dk, dv=dv, dtype=dtype, lengths=lengths, B=len(lengths),
                               h0_std=0.1 if h0 else 0.0, seed=seed)
    inp = inputs.prefill_inputs(cfg, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(seed + 1)
    T_tot = inp["T_tot"]
    dout = torch.randn(T_tot, H, dv, generator=gen, device="cuda").to(inp["q"].dtype)
    dhT_t = torch.randn(len(lengths), H, dk, dv, generator=gen, device="cuda") if dhT else None
    got = binding.kda_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], dout, h0=inp["h0"],
                                cu_seqlens=inp["cu_seqlens"], dhT=dhT_t, need_dh0=h0)
    assert_no_device_error()
    ref = oracle_kda_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], dout, h0=inp["h0"],
                              cu_seqlens=inp["cu_seqlens"].to("cpu"), dhT=dhT_t)
    names = ("dq", "dk", "dv", "dg", "dbeta", "dh0")
    for name, a, r in zip(names, got, ref):
        if r is None:
            continue
        e = rel_err(a, r)
        assert e <= TOL, (name, e)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_backward_single_sequence_ragged_tail(dtype, path):
    _case((200,), 2, 128, 128, dtype, h0=True, dhT=True, seed=501)


def test_backward_varlen_with_short_sequences(path):
    _case((70, 1, 130), 2, 64, 64, "fp32", h0=False, dhT=False, seed=502)


@pytest.mark.parametrize("dk,dv", [(128, 64), (64, 128)])
def test_backward_rectangular_state(dk, dv, path):
    _case((96, 33), 1, dk, dv, "bf16", h0=True, dhT=True, seed=503 + dk)


def test_backward_gradients_are_deterministic(path):
    cfg = inputs.PrefillConfig("bwd", H=2, dk=128, dv=128, dtype="bf16", lengths=(150,), B=1, seed=510)
    inp = inputs.prefill_inputs(cfg, device="cuda")
    dout = torch.ones(150, 2, 128, device="cuda", dtype=torch.bfloat16)
    a = binding.kda_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], dout, cu_seqlens=inp["cu_seqlens"])
    b = binding.kda_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], dout, cu_seqlens=inp["cu_seqlens"])
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("H", [24, 48, 96])
@pytest.mark.parametrize("dv", [128, 64])
def test_backward_every_value_column_slicing(H, dv, path):
    """Enough (sequence, head) chains to reach every value-column slicing of the serial passes: on a
    152-SM GPU the chunkwise path takes 4, 2 and 2 (64-column) slices at dv = 128 and 2, 2 and 1 at
    dv = 64 for H = 24, 48, 96 (H <= 2 above takes 8 and 4), and the token sweep 4, 2 and 1."""
    _case((100,), H, 128, dv, "bf16", h0=True, dhT=True, seed=520 + H + dv)


def _loss_fd(inp, dout, name, delta, eps):
    """Central difference of L = <dout, o> along `delta` in input `name`, o from the fp64 C oracle."""
    from oracle import oracle_kda_prefill

    vals = []
    for sgn in (1.0, -1.0):
        x = {n: inp[n].double().cpu() for n in ("q", "k", "v", "g", "beta")}
        x[name] = x[name] + sgn * eps * delta
        o, _ = oracle_kda_prefill(x["q"], x["k"], x["v"], x["g"], x["beta"])
        vals.append(float(np.sum(o * dout)))
    return (vals[0] - vals[1]) / (2 * eps)


def test_backward_full_size_directional_derivatives():
    """The 8192-token x 32-head workload: for each input, the GPU gradient's directional derivative
    along (1) the gradient itself and (2) a Gaussian direction on one 512-token block matches the
    central difference of L = <dout, o> evaluated by the fp64 oracle."""
    inp = inputs.prefill_inputs(inputs.PREFILL, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(530)
    dout = torch.randn(inp["T_tot"], 32, 128, generator=gen, device="cuda").to(torch.bfloat16)
    grads = dict(zip(("q", "k", "v", "g", "beta"),
                     binding.kda_chunk_bwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], dout)[:5]))
    assert_no_device_error()
    dout_np = dout.double().cpu().numpy()
    rng = np.random.default_rng(531)
    for name, gr in grads.items():
        gr = gr.double().cpu()
        blk = torch.zeros_like(gr)
        blk[3000:3512] = torch.from_numpy(rng.standard_normal(tuple(blk[3000:3512].shape)))
        for delta in (gr, blk):
            d_gpu = float((gr * delta).sum())
            # a step that moves each input by ~1e-4 of its typical size (g stays inside (-5, 0))
            scale = float(inp[name].double().abs().mean())
            eps = 1e-4 * scale / float(delta.abs().max())
            d_fd = _loss_fd(inp, dout_np, name, delta, eps)
            # a sum of many products of either sign: measured against its own size or, when that
            # happens to be small for a random direction, against the spread sqrt(sum (g_i d_i)^2)
            spread = float(((gr * delta) ** 2).sum().sqrt())
            assert abs(d_gpu - d_fd) <= 2e-3 * max(abs(d_fd), spread), (name, d_gpu, d_fd, spread)
