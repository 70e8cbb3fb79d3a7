"""Failure reporting of the CUDA path on the GPU: value range of the fp16 tensor-core operands,
bounded device waits that run out, and the debug precondition checks.  Every failure here is
reported through the device error word (kda_get_device_error); none traps or hangs, and the next
ordinary call on the same device is checked against the oracle."""
import dataclasses

import pytest
import torch

from gated_delta_rule_08_gb300 import binding, inputs
from gpu_util import TOL, assert_no_device_error, oracle_prefill, parity_err, rel_err, run_prefill

pytestmark = pytest.mark.gpu


def _scaled(cfg, v_scale, h0_scale):
    inp = inputs.prefill_inputs(cfg, device="cuda")
    inp["v"] = (inp["v"].float() * v_scale).to(inp["v"].dtype).contiguous()
    inp["h0"] = (inp["h0"] * h0_scale).contiguous()
    return inp


# ------------------------------------------------------------------ fp16 operand range
def test_large_values_inside_the_fp16_range_keep_parity():
    """v ~ N(0, 30) and h0 ~ N(0, 30) (h0_std 0.1 scaled by 300): every fp16 operand stays inside its
    range, so the bf16 bound holds as for unit-scale values and no flag is raised."""
    cfg = inputs.PrefillConfig("range", H=4, dk=128, dv=128, dtype="bf16", lengths=(300, 77), B=2, h0_std=0.1,
                               seed=601)
    inp = _scaled(cfg, 30.0, 300.0)
    ref_out, ref_hT = oracle_prefill(inp)
    out, hT = run_prefill(inp, out_dtype=torch.float32)
    assert binding.kda_get_device_error() == 0
    assert rel_err(out, ref_out) <= TOL[torch.bfloat16] and rel_err(hT, ref_hT) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("v_scale,h0_scale", [(1e5, 1.0), (1.0, 1e6)], ids=["values", "initial-state"])
def test_values_beyond_the_fp16_range_set_the_flag(v_scale, h0_scale):
    """|beta v| or |h0| past 65504 cannot be an fp16 operand: it becomes inf, which reaches out and the
    final state, so the call flags KDA_DEVERR_NONFINITE (its results are not valid) and traps on
    nothing; the next call matches the oracle."""
    cfg = inputs.PrefillConfig("range", H=2, dk=128, dv=128, dtype="bf16", lengths=(200,), B=1, h0_std=0.1,
                               seed=602)
    inp = _scaled(cfg, v_scale, h0_scale)
    run_prefill(inp, out_dtype=torch.float32)
    flags = binding.kda_get_device_error()
    assert flags & binding.DEVERR_NONFINITE, hex(flags)
    assert not flags & binding.DEVERR_WAIT_TIMEOUT, hex(flags)
    ok = inputs.prefill_inputs(cfg, device="cuda")
    ref_out, ref_hT = oracle_prefill(ok)
    out, hT = run_prefill(ok, out_dtype=torch.float32)
    assert_no_device_error()
    assert rel_err(out, ref_out) <= TOL[torch.bfloat16] and rel_err(hT, ref_hT) <= TOL[torch.bfloat16]


# ------------------------------------------------------------------ bounded waits that run out
@pytest.mark.parametrize("lengths,H,epilogue", [((300, 70), 2, False), ((8192,), 4, False), ((8192,), 4, True)],
                         ids=["one-pass", "split-into-segments", "split-with-epilogue"])
def test_waits_that_run_out_are_reported_and_the_device_stays_usable(lengths, H, epilogue, monkeypatch):
    """KDA_TEST_WAIT_TIMEOUT=1 launches kernel variants whose waits on work of their own CTA give up at
    once, as a wait that runs out does (the drains of in-flight copies and MMAs keep their normal
    bound).  The call reports
    KDA_DEVERR_WAIT_TIMEOUT; the next ordinary call on the same stream matches the oracle, so every
    CTA released its tensor memory and the context is intact.  The second case runs the segment
    transitions, the merge and the read-out pass (intra-device context parallelism); the third adds
    the gate epilogue, whose helper warps must leave their loop when a TMEM warp's wait gives up."""
    cfg = inputs.PrefillConfig("timeout", H=H, dk=128, dv=128, dtype="bf16", lengths=lengths, B=len(lengths),
                               h0_std=0.1, z_mean=-8.0, seed=603, epilogue=epilogue)
    inp = inputs.prefill_inputs(cfg, device="cuda")
    monkeypatch.setenv("KDA_TEST_WAIT_TIMEOUT", "1")
    run_prefill(inp, out_dtype=torch.float32)
    flags = binding.kda_get_device_error()
    assert flags & binding.DEVERR_WAIT_TIMEOUT, hex(flags)
    monkeypatch.delenv("KDA_TEST_WAIT_TIMEOUT")
    ref_out, ref_hT = oracle_prefill(inp)
    for _ in range(2):
        out, hT = run_prefill(inp, out_dtype=torch.float32)
        assert_no_device_error()
        assert rel_err(out, ref_out) <= TOL[torch.bfloat16] and rel_err(hT, ref_hT) <= TOL[torch.bfloat16]


# ------------------------------------------------------------------ KDA_DEBUG_CHECKS
def test_debug_checks_flag_broken_preconditions(monkeypatch):
    """With KDA_DEBUG_CHECKS set, a planted g = -6 (below the bound g > -5 that the reference-point
    factorisation relies on), a beta outside [0, 1] and two decode requests on one slot each set
    KDA_DEVERR_PRECONDITION; inputs that meet the preconditions set nothing.  Without the switch
    the same planted g is not checked."""
    cfg = inputs.PrefillConfig("dbg", H=2, dk=128, dv=128, dtype="bf16", lengths=(130,), B=1, seed=604)
    inp = inputs.prefill_inputs(cfg, device="cuda")
    monkeypatch.setenv("KDA_DEBUG_CHECKS", "1")
    run_prefill(inp)
    assert binding.kda_get_device_error() == 0
    bad_g = dict(inp, g=inp["g"].clone())
    bad_g["g"][77, 1, 5] = -6.0
    run_prefill(bad_g)
    assert binding.kda_get_device_error() & binding.DEVERR_PRECONDITION
    bad_b = dict(inp, beta=inp["beta"].clone())
    bad_b["beta"][3, 0] = 1.5
    run_prefill(bad_b)
    assert binding.kda_get_device_error() & binding.DEVERR_PRECONDITION

    d = inputs.decode_inputs(dataclasses.replace(inputs.DECODE, N=16, H=2, num_slots=64, seed=605), device="cuda")
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"], d["state_pool"])
    binding.kda_decode_step(*args, d["slot_idx"])
    assert binding.kda_get_device_error() == 0
    dup = d["slot_idx"].clone()
    dup[9] = dup[2]
    binding.kda_decode_step(*args, dup)
    assert binding.kda_get_device_error() & binding.DEVERR_PRECONDITION

    monkeypatch.delenv("KDA_DEBUG_CHECKS")
    run_prefill(bad_g)
    assert not binding.kda_get_device_error() & binding.DEVERR_PRECONDITION
