"""Backward of the prefill recurrence on the GPU vs the fp64 autograd oracle (through the C-ABI)."""
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
