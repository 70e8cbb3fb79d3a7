"""Context parallelism across devices (KCP) on one GPU: the ranks of one long sequence emulated one
after another.  Each range's map (P, b) from kda_chunk_fwd_segment_map, the fold of the maps before a
range by kda_state_compose, and each range's prefill from its folded initial state are checked against
the fp64 oracle on the whole sequence."""
import numpy as np
import pytest
import torch

from gated_delta_rule_08_gb300 import binding, inputs
from gpu_util import assert_no_device_error, parity_err, rel_err
from oracle import oracle_kda_prefill

pytestmark = pytest.mark.gpu
TOL = 2e-2  # bf16 inputs


def _ranges(T, cuts):
    edges = [0] + list(cuts) + [T]
    return list(zip(edges[:-1], edges[1:]))


def test_segment_map_matches_the_oracle():
    """b is the range's final state from a zero state; P is its final state from S_in = I with v = 0
    (a dk x dk state), so that P S_in + b is the final state from any S_in.  Slow decay (z_mean = -8,
    g ~ -2e-3 per token) keeps P of order one over the range: a fast-decaying range's P is far below
    the fp32 range (e^-240 over 1000 tokens at z_mean = -3) and is rightly stored as 0."""
    cfg = inputs.PrefillConfig("map", H=3, dk=128, dv=128, dtype="bf16", B=1, T=1000, z_mean=-8.0, seed=701)
    inp = inputs.prefill_inputs(cfg, device="cuda")
    P, b = binding.kda_chunk_fwd_segment_map(inp["k"], inp["v"], inp["g"], inp["beta"])
    assert_no_device_error()
    _, ref_b = oracle_kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"])
    eye = torch.eye(128, dtype=torch.float32).expand(1, 3, 128, 128).contiguous()
    _, ref_P = oracle_kda_prefill(inp["q"], inp["k"], torch.zeros_like(inp["k"]), inp["g"], inp["beta"], h0=eye)
    assert rel_err(b, ref_b[0]) <= TOL and rel_err(P, ref_P[0]) <= TOL
    # the map applied to a state equals the oracle run from that state
    S = (0.1 * torch.randn(3, 128, 128, generator=torch.Generator().manual_seed(7))).cuda()
    _, ref_S = oracle_kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], h0=S[None])
    got = binding.kda_state_compose(P[None].contiguous(), b[None].contiguous(), S0=S)
    assert rel_err(got, ref_S[0]) <= TOL


def test_empty_range_is_the_identity_map():
    H = 2
    e = torch.empty(0, H, 128, device="cuda", dtype=torch.bfloat16)
    P, b = binding.kda_chunk_fwd_segment_map(e, e, torch.empty(0, H, 128, device="cuda"),
                                             torch.empty(0, H, device="cuda"))
    assert_no_device_error()
    assert torch.equal(P, torch.eye(128, device="cuda").expand(H, 128, 128)) and torch.all(b == 0)


def test_state_compose_is_the_fold_of_the_maps():
    """S = P[n-1](... (P[0] S0 + b[0]) ...) + b[n-1] against an fp64 fold (all four (dk, dv))."""
    gen = torch.Generator().manual_seed(702)
    for dk, dv in ((128, 128), (128, 64), (64, 128), (64, 64)):
        n, H = 3, 2
        P = torch.randn(n, H, dk, dk, generator=gen) / dk ** 0.5
        b = torch.randn(n, H, dk, dv, generator=gen)
        S0 = torch.randn(H, dk, dv, generator=gen)
        ref = S0.double()
        for i in range(n):
            ref = P[i].double() @ ref + b[i].double()
        got = binding.kda_state_compose(P.cuda(), b.cuda(), S0=S0.cuda())
        assert rel_err(got, ref.numpy()) <= 1e-5, (dk, dv)
        got0 = binding.kda_state_compose(P[:0].cuda(), b[:0].cuda(), S0=None, out=torch.ones(H, dk, dv).cuda())
        assert torch.all(got0 == 0)
        alias = S0.cuda().contiguous()
        binding.kda_state_compose(P.cuda(), b.cuda(), S0=alias, out=alias)
        assert rel_err(alias, ref.numpy()) <= 1e-5


@pytest.mark.parametrize("cuts,h0", [((4096,), False), ((3000, 5500), True), ((1000, 2048, 6000), True)],
                         ids=["2-ranks", "3-ranks-ragged", "4-ranks-ragged"])
def test_ranks_of_one_sequence_reproduce_the_whole_sequence(cuts, h0):
    """An 8192-token sequence (H = 4, slow decay so that every range's initial state matters: g ~ -2e-3
    per token) cut into 2-4 consecutive ranges, as KCP would place them on 2-4 GPUs: every range's
    outputs and the last range's final state match the oracle on the whole sequence."""
    T, H = 8192, 4
    cfg = inputs.PrefillConfig("kcp", H=H, dk=128, dv=128, dtype="bf16", B=1, T=T, h0_std=0.1 if h0 else 0.0,
                               z_mean=-8.0, seed=703)
    inp = inputs.prefill_inputs(cfg, device="cuda")
    ref_out, ref_hT = oracle_kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], h0=inp["h0"])
    rng = _ranges(T, cuts)
    maps = [binding.kda_chunk_fwd_segment_map(*(inp[x][a:e].contiguous() for x in ("k", "v", "g", "beta")))
            for a, e in rng]
    Ps = torch.stack([m[0] for m in maps])
    bs = torch.stack([m[1] for m in maps])
    S0 = inp["h0"][0].contiguous() if h0 else None
    outs, last = [], None
    for r, (a, e) in enumerate(rng):
        S_in = binding.kda_state_compose(Ps[:r].contiguous(), bs[:r].contiguous(), S0=S0)
        o, hT = binding.kda_chunk_fwd(*(inp[x][a:e].contiguous() for x in ("q", "k", "v", "g", "beta")),
                                      h0=S_in[None].contiguous(), out_dtype=torch.float32)
        outs.append(o)
        last = hT
    assert_no_device_error()
    out = torch.cat(outs)
    assert parity_err(out, ref_out) <= TOL and rel_err(last, ref_hT) <= TOL
    # the fold of every range's map is the sequence's final state too
    S_all = binding.kda_state_compose(Ps, bs, S0=S0)
    assert rel_err(S_all, ref_hT[0]) <= TOL
