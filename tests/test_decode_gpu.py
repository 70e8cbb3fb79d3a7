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


# ------------------------------------------------------------------ several tokens per request
def _multi(cfg, n_tok):
    return inputs.decode_inputs(dataclasses.replace(cfg, n_tok=n_tok), device="cuda")


def _oracle_multi(inp, counts, epilogue, pool_before):
    """The single-step oracle applied token by token to the touched states of `pool_before`:
    request n takes its first counts[n] tokens.  Returns (out [N, n_tok, H, dv] with NaN where no
    token applied, final touched states [N, H, dk, dv])."""
    N, n_tok = inp["q"].shape[:2]
    pool = pool_before[inp["slot_idx"].long()].clone()
    outs = np.full((N, n_tok) + tuple(inp["v"].shape[2:]), np.nan)
    for t in range(n_tok):
        slots = np.array([n if counts[n] > t else -1 for n in range(N)])
        tok = {x: inp[x][:, t] for x in ("q", "k", "v", "g", "beta")}
        gate = inp["gate"][:, t] if epilogue else None
        nw = inp["norm_weight"] if epilogue else None
        o, pool, _ = oracle_kda_decode(tok["q"], tok["k"], tok["v"], tok["g"], tok["beta"], pool, slots, gate=gate,
                                       norm_weight=nw)
        live = slots >= 0
        outs[live, t] = o[live]
    return outs, pool


@pytest.mark.parametrize("dk,dv,dtype", [(128, 128, "bf16"), (64, 128, "fp32"), (128, 64, "bf16")])
def test_decode_multi_verify_leaves_the_pool_untouched(dk, dv, dtype):
    """Speculative-decode verify: every draft token of every request is applied in order to a
    private copy of the state; outputs match the oracle, the pool is byte-identical."""
    cfg = dataclasses.replace(inputs.DECODE, N=6, H=3, dk=dk, dv=dv, num_slots=11, dtype=dtype, seed=90 + dk + dv)
    inp = _multi(cfg, 4)
    before = inp["state_pool"].clone()
    out = binding.kda_decode_multi(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["state_pool"],
                                   inp["slot_idx"], commit=False, gate=inp["gate"], norm_weight=inp["norm_weight"])
    assert_no_device_error()
    assert torch.equal(inp["state_pool"], before)
    ref_out, _ = _oracle_multi(inp, [4] * cfg.N, True, before)
    assert parity_err(out, ref_out) <= TOL[inputs.torch_dtype(dtype)]


def test_decode_multi_accept_commits_exactly_the_accepted_prefix():
    """Accept: request n re-applies its first accept[n] tokens and writes that state back; its
    outputs equal the verify outputs bit for bit; rows of rejected tokens are not written."""
    cfg = dataclasses.replace(inputs.DECODE, N=6, H=4, num_slots=13, seed=95)
    inp = _multi(cfg, 4)
    before = inp["state_pool"].clone()
    kw = dict(gate=inp["gate"], norm_weight=inp["norm_weight"])
    verify = binding.kda_decode_multi(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["state_pool"],
                                      inp["slot_idx"], commit=False, **kw)
    accept = [0, 1, 2, 3, 4, 2]
    counts = torch.tensor(accept, dtype=torch.int32, device="cuda")
    out = torch.full_like(verify, 5.0)
    binding.kda_decode_multi(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["state_pool"], inp["slot_idx"],
                             counts, out=out, commit=True, **kw)
    assert_no_device_error()
    for n, a in enumerate(accept):
        assert torch.equal(out[n, :a], verify[n, :a])
        assert torch.all(out[n, a:] == 5.0)
    ref_out, ref_states = _oracle_multi(inp, accept, True, before)
    slots = inp["slot_idx"].long()
    assert rel_err(inp["state_pool"][slots], ref_states) <= 1e-5
    assert torch.equal(inp["state_pool"][slots[0]], before[slots[0]])  # nothing accepted: state kept
    untouched = torch.ones(cfg.num_slots, dtype=torch.bool, device="cuda")
    untouched[slots] = False
    assert torch.equal(inp["state_pool"][untouched], before[untouched])


def test_decode_multi_one_token_is_the_decode_step():
    cfg = dataclasses.replace(inputs.DECODE, N=9, H=2, num_slots=20, seed=97)
    a = inputs.decode_inputs(cfg, device="cuda")
    b = inputs.decode_inputs(cfg, device="cuda")
    kw_a = dict(gate=a["gate"], norm_weight=a["norm_weight"])
    oa = binding.kda_decode_step(a["q"], a["k"], a["v"], a["g"], a["beta"], a["state_pool"], a["slot_idx"], **kw_a)
    ob = binding.kda_decode_multi(b["q"][:, None], b["k"][:, None], b["v"][:, None], b["g"][:, None],
                                  b["beta"][:, None], b["state_pool"], b["slot_idx"], commit=True,
                                  gate=b["gate"][:, None], norm_weight=b["norm_weight"])
    assert torch.equal(oa, ob[:, 0]) and torch.equal(a["state_pool"], b["state_pool"])


def test_decode_multi_bad_count_sets_flag_and_skips_request():
    cfg = dataclasses.replace(inputs.DECODE, N=3, H=2, num_slots=5, seed=98)
    inp = _multi(cfg, 2)
    before = inp["state_pool"].clone()
    counts = torch.tensor([1, 3, -1], dtype=torch.int32, device="cuda")
    out = torch.full((3, 2, 2, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    binding.kda_decode_multi(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["state_pool"], inp["slot_idx"],
                             counts, out=out, commit=True)
    assert binding.kda_get_device_error() & binding.DEVERR_BAD_COUNT
    slots = inp["slot_idx"].long()
    assert torch.all(out[1] == 7.0) and torch.all(out[2] == 7.0) and torch.all(out[0, 1] == 7.0)
    assert torch.equal(inp["state_pool"][slots[1]], before[slots[1]])
    assert torch.equal(inp["state_pool"][slots[2]], before[slots[2]])
    assert not torch.equal(inp["state_pool"][slots[0]], before[slots[0]])


def test_decode_multi_many_items_per_cta():
    """More (request, head) items (1280) than CTAs resident at once, so CTAs warm L2 with the state
    and inputs of the ones that follow them: verify (no write-back) and accept with per-request
    counts from 0 to 4 against the oracle."""
    cfg = dataclasses.replace(inputs.DECODE, N=160, H=8, num_slots=400, seed=99)
    inp = _multi(cfg, 4)
    before = inp["state_pool"].clone()
    kw = dict(gate=inp["gate"], norm_weight=inp["norm_weight"])
    verify = binding.kda_decode_multi(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["state_pool"],
                                      inp["slot_idx"], commit=False, **kw)
    assert_no_device_error()
    assert torch.equal(inp["state_pool"], before)
    ref_out, _ = _oracle_multi(inp, [4] * cfg.N, True, before)
    assert parity_err(verify, ref_out) <= TOL[torch.bfloat16]
    accept = [(7 * n) % 5 for n in range(cfg.N)]  # 0..4, every value many times
    counts = torch.tensor(accept, dtype=torch.int32, device="cuda")
    out = torch.full_like(verify, 5.0)
    binding.kda_decode_multi(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["state_pool"], inp["slot_idx"],
                             counts, out=out, commit=True, **kw)
    assert_no_device_error()
    for n, a in enumerate(accept):
        assert torch.equal(out[n, :a], verify[n, :a])
        assert torch.all(out[n, a:] == 5.0)
    _, ref_states = _oracle_multi(inp, accept, True, before)
    slots = inp["slot_idx"].long()
    assert rel_err(inp["state_pool"][slots], ref_states) <= 1e-5
    untouched = torch.ones(cfg.num_slots, dtype=torch.bool, device="cuda")
    untouched[slots] = False
    assert torch.equal(inp["state_pool"][untouched], before[untouched])


def test_decode_multi_bad_slot_among_many_items():
    """A request with an out-of-range slot is skipped by the multi-token kernel (flag set, its
    outputs untouched) and every other request is still served.  Its items come late enough in the
    grid that earlier CTAs try to prefetch its state, which must skip the bad slot too."""
    cfg = dataclasses.replace(inputs.DECODE, N=100, H=8, num_slots=300, seed=101)
    inp = _multi(cfg, 3)
    good = inp["slot_idx"].clone()
    ref = binding.kda_decode_multi(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["state_pool"], good,
                                   commit=False)
    assert_no_device_error()
    bad = good.clone()
    bad[77] = cfg.num_slots + 5
    out = torch.full_like(ref, 3.0)
    binding.kda_decode_multi(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["state_pool"], bad, out=out,
                             commit=False)
    assert binding.kda_get_device_error() & binding.DEVERR_BAD_SLOT
    assert torch.all(out[77] == 3.0)
    keep = torch.ones(cfg.N, dtype=torch.bool, device="cuda")
    keep[77] = False
    assert torch.equal(out[keep], ref[keep])
