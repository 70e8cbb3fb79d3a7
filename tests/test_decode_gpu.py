"""Decode step on the GPU vs the fp64 oracle (through the C-ABI binding)."""
import dataclasses

import numpy as np
import pytest
import torch

from gated_delta_rule_08_gb300 import binding, inputs
from gpu_util import TOL, assert_no_device_error, parity_err, rel_err
from oracle import oracle_kda_decode

pytestmark = pytest.mark.gpu


def _run_and_check(cfg, epilogue=True):
    inp = inputs.decode_inputs(cfg, device="cuda")
    pool = inp["state_pool"]
    slots = inp["slot_idx"]
    gate = inp["gate"] if epilogue else None
    nw = inp["norm_weight"] if epilogue else None
    # oracle on a compact pool holding only the touched slots, remapped to 0..N-1
    touched = pool[slots.long()].clone()
    untouched_mask = torch.ones(pool.shape[0], dtype=torch.bool, device="cuda")
    untouched_mask[slots.long()] = False
    untouched_before = pool[untouched_mask].clone()
    out = binding.kda_decode_step(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], pool, slots,
                                  gate=gate, norm_weight=nw)
    assert_no_device_error()
    ref_out, ref_pool, skipped = oracle_kda_decode(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], touched,
                                                   np.arange(cfg.N), gate=gate, norm_weight=nw)
    assert skipped == 0
    tol = TOL[inputs.torch_dtype(cfg.dtype)]
    e_out = parity_err(out, ref_out)
    e_state = rel_err(pool[slots.long()], ref_pool)
    assert e_out <= tol, e_out
    assert e_state <= 1e-5, e_state  # fp32 state arithmetic on exact inputs
    # slots not named in slot_idx are byte-identical
    assert torch.equal(pool[untouched_mask], untouched_before)
    return e_out, e_state


def test_decode_config_n256_h32_d128_pool1024():
    _run_and_check(inputs.DECODE)


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 64), (64, 128)])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("epilogue", [True, False])
def test_decode_small_variants(dk, dv, dtype, epilogue):
    cfg = dataclasses.replace(inputs.DECODE, N=7, H=3, dk=dk, dv=dv, num_slots=19, dtype=dtype, epilogue=epilogue,
                              seed=40 + dk + dv)
    _run_and_check(cfg, epilogue=epilogue)


def test_decode_bad_slot_sets_flag_and_skips_row():
    cfg = dataclasses.replace(inputs.DECODE, N=4, H=2, num_slots=6, seed=77)
    inp = inputs.decode_inputs(cfg, device="cuda")
    pool = inp["state_pool"]
    before = pool.clone()
    slots = torch.tensor([1, -3, 6, 4], dtype=torch.int32, device="cuda")
    out = torch.full((4, 2, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    binding.kda_decode_step(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], pool, slots, out=out,
                            gate=inp["gate"], norm_weight=inp["norm_weight"])
    flags = binding.kda_get_device_error()
    assert flags & binding.DEVERR_BAD_SLOT
    assert binding.kda_get_device_error() == 0  # reading clears the word
    assert torch.all(out[1] == 7.0) and torch.all(out[2] == 7.0)
    for s in (0, 2, 3, 5):
        assert torch.equal(pool[s], before[s])
    assert not torch.equal(pool[1], before[1]) and not torch.equal(pool[4], before[4])


def test_decode_is_deterministic():
    cfg = dataclasses.replace(inputs.DECODE, N=32, num_slots=64, seed=78)
    a = inputs.decode_inputs(cfg, device="cuda")
    b = inputs.decode_inputs(cfg, device="cuda")
    oa = binding.kda_decode_step(a["q"], a["k"], a["v"], a["g"], a["beta"], a["state_pool"], a["slot_idx"],
                                 gate=a["gate"], norm_weight=a["norm_weight"])
    ob = binding.kda_decode_step(b["q"], b["k"], b["v"], b["g"], b["beta"], b["state_pool"], b["slot_idx"],
                                 gate=b["gate"], norm_weight=b["norm_weight"])
    assert torch.equal(oa, ob) and torch.equal(a["state_pool"], b["state_pool"])


def test_decode_zero_requests_is_a_no_op():
    pool = torch.zeros(3, 2, 64, 64, device="cuda")
    e = torch.empty(0, 2, 64, device="cuda", dtype=torch.bfloat16)
    f = torch.empty(0, 2, 64, device="cuda")
    out = binding.kda_decode_step(e, e, e, f, torch.empty(0, 2, device="cuda"), pool,
                                  torch.empty(0, dtype=torch.int32, device="cuda"))
    assert out.shape == (0, 2, 64)
    assert_no_device_error()
