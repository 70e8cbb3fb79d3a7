"""Chunked prefill on the GPU vs the fp64 oracle (through the C-ABI binding)."""
import dataclasses
import math

import numpy as np
import pytest
import torch

from gated_delta_rule_08_gb300 import binding, inputs
from gpu_util import TOL, assert_no_device_error, oracle_prefill, parity_err, rel_err, run_prefill
from oracle import oracle_kda_prefill

pytestmark = pytest.mark.gpu


def _check(cfg, *, epilogue=None, device_gen=False, out_dtypes=(torch.float32, torch.bfloat16)):
    """GPU vs oracle on the same inputs.  The tolerance is the one for the input dtype
    (1e-3 fp32, 2e-2 bf16) on max|err|/RMS, per output tensor; a bf16-stored output is
    allowed its own storage rounding on top (see gpu_util.parity_err)."""
    inp = inputs.prefill_inputs(cfg, device="cuda" if device_gen else "cpu")
    inp_d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    ref_out, ref_hT = oracle_prefill(inp_d, epilogue=epilogue)
    tol = TOL[inputs.torch_dtype(cfg.dtype)]
    res = None
    for odt in out_dtypes:
        out, hT = run_prefill(inp_d, epilogue=epilogue, out_dtype=odt)
        assert_no_device_error()
        e_o, e_h = parity_err(out, ref_out), rel_err(hT, ref_hT)
        assert e_o <= tol and e_h <= tol, (cfg.name, odt, e_o, e_h)
        res = res or (inp_d, out, hT)
    return res


# ------------------------------------------------------------------ the named workloads
def test_tiny_fp32_h2_t256_d64():
    _check(inputs.TINY)


def test_prefill_bf16_h32_t8192_d128():
    _check(inputs.PREFILL, device_gen=True)


def test_prefill_bf16_h32_t8192_d64():
    """The prefill workload's shape with 64-dim heads: the CUDA-core path (tensor-core products,
    value-column clusters) over 128 chunks per chain."""
    _check(dataclasses.replace(inputs.PREFILL, dk=64, dv=64, h0_std=0.1, name="prefill d64"), device_gen=True)


def test_prefill_bf16_h32_t8192_d128_epilogue():
    """The prefill workload with the fused RMSNorm + sigmoid gate: the tensor-core read-out's
    epilogue specialisation (staged gate logits, batched row reductions) over the whole sequence."""
    cfg = dataclasses.replace(inputs.PREFILL, epilogue=True, name="prefill epilogue")
    _check(cfg, epilogue=True, device_gen=True)


def test_varlen_bf16_8seqs_h32_d128_h0():
    _check(inputs.VARLEN, device_gen=True)


# ------------------------------------------------------------------ sweeps: lengths, dims, states, epilogue
@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 127, 200])
@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_single_sequence_lengths(T, dtype):
    cfg = inputs.PrefillConfig("len sweep", H=3, dk=128, dv=128, dtype=dtype, B=1, T=T, h0_std=0.1, seed=100 + T)
    _check(cfg)


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 64), (64, 128), (128, 128)])
@pytest.mark.parametrize("epilogue", [False, True])
def test_dims_and_epilogue(dk, dv, epilogue):
    cfg = inputs.PrefillConfig("dims", H=2, dk=dk, dv=dv, dtype="bf16", lengths=(130, 64, 1, 77), B=4,
                               h0_std=0.1, epilogue=epilogue, seed=200 + dk + dv)
    _check(cfg, epilogue=epilogue)


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128)])
def test_fp32_inputs_with_the_epilogue(dk, dv):
    """fp32 inputs take the CUDA-core path: its serial pass runs each chain as a cluster of dv/16
    CTAs that exchange the RMSNorm's partial sums through distributed shared memory (one stage of
    records at dk = 128, two at dk = 64)."""
    cfg = inputs.PrefillConfig("fp32 epi", H=3, dk=dk, dv=dv, dtype="fp32", lengths=(200, 64, 1, 333), B=4,
                               h0_std=0.1, epilogue=True, seed=240 + dk + dv)
    _check(cfg, epilogue=True)


def test_varlen_with_empty_and_short_sequences():
    cfg = inputs.PrefillConfig("varlen edge", H=4, dk=128, dv=128, dtype="bf16",
                               lengths=(0, 1, 63, 64, 65, 0, 129, 3), B=8, h0_std=0.1, epilogue=True, seed=300)
    inp, out, hT = _check(cfg, epilogue=True)
    # empty sequences: final state equals initial state, bit for bit
    assert torch.equal(hT[0], inp["h0"][0]) and torch.equal(hT[5], inp["h0"][5])


def test_many_sequences_beyond_the_length_ordering_limit():
    # more sequences than the plan sorts by length (512): the serial pass keeps their given order
    rng = np.random.default_rng(320)
    lengths = tuple(int(x) for x in rng.integers(0, 131, size=600))
    cfg = inputs.PrefillConfig("many", H=1, dk=128, dv=128, dtype="bf16", lengths=lengths, B=600, h0_std=0.1,
                               seed=320)
    _check(cfg, out_dtypes=(torch.bfloat16,))


def test_length_ordering_with_ties_matches_oracle():
    # equal lengths among unequal ones: the rank order breaks ties by index
    cfg = inputs.PrefillConfig("ties", H=2, dk=128, dv=128, dtype="bf16", lengths=(200, 65, 200, 1, 65, 300, 200),
                               B=7, h0_std=0.1, seed=321)
    _check(cfg, out_dtypes=(torch.bfloat16,))


def test_equal_lengths_without_cu_seqlens():
    cfg = inputs.PrefillConfig("equal", H=2, dk=128, dv=128, dtype="bf16", B=3, T=100, h0_std=0.1, seed=301)
    inp = inputs.prefill_inputs(cfg, device="cuda")
    out_a, h_a = binding.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], h0=inp["h0"], B=3)
    out_b, h_b = binding.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], h0=inp["h0"],
                                       cu_seqlens=inp["cu_seqlens"])
    assert torch.equal(out_a, out_b) and torch.equal(h_a, h_b)


# ------------------------------------------------------------------ bit-exact properties
def test_packed_equals_each_sequence_alone():
    cfg = inputs.PrefillConfig("pack", H=2, dk=128, dv=128, dtype="bf16", lengths=(70, 5, 128, 200), B=4,
                               h0_std=0.1, seed=302)
    inp = inputs.prefill_inputs(cfg, device="cuda")
    out, hT = run_prefill(inp)
    cu = inp["cu_seqlens"].tolist()
    for b in range(4):
        a, e = cu[b], cu[b + 1]
        o1, h1 = binding.kda_chunk_fwd(inp["q"][a:e].contiguous(), inp["k"][a:e].contiguous(),
                                       inp["v"][a:e].contiguous(), inp["g"][a:e].contiguous(),
                                       inp["beta"][a:e].contiguous(), h0=inp["h0"][b:b + 1].contiguous())
        assert torch.equal(o1, out[a:e]), b
        assert torch.equal(h1[0], hT[b]), b


def test_run_to_run_deterministic():
    cfg = inputs.PrefillConfig("det", H=4, dk=128, dv=128, dtype="bf16", lengths=(300, 17), B=2, h0_std=0.1,
                               epilogue=True, seed=303)
    inp = inputs.prefill_inputs(cfg, device="cuda")
    o1, h1 = run_prefill(inp)
    o2, h2 = run_prefill(inp)
    assert torch.equal(o1, o2) and torch.equal(h1, h2)


def test_final_state_may_alias_initial_state():
    cfg = inputs.PrefillConfig("alias", H=2, dk=128, dv=128, dtype="bf16", lengths=(90, 33), B=2, h0_std=0.1,
                               seed=304)
    inp = inputs.prefill_inputs(cfg, device="cuda")
    out, hT = run_prefill(inp)
    state = inp["h0"].clone()
    out2, _ = binding.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], h0=state,
                                    cu_seqlens=inp["cu_seqlens"], hT=state)
    assert torch.equal(out, out2) and torch.equal(state, hT)


def test_split_run_resumes_from_final_state():
    """Prefill of a prefix, then of the rest from its final state == one prefill (checkpoint/resume)."""
    cfg = inputs.PrefillConfig("resume", H=2, dk=128, dv=128, dtype="bf16", B=1, T=256, h0_std=0.1, seed=305)
    inp = inputs.prefill_inputs(cfg, device="cuda")
    out, hT = run_prefill(inp)
    o1, h1 = binding.kda_chunk_fwd(*(inp[x][:128].contiguous() for x in ("q", "k", "v", "g", "beta")),
                                   h0=inp["h0"])
    o2, h2 = binding.kda_chunk_fwd(*(inp[x][128:].contiguous() for x in ("q", "k", "v", "g", "beta")), h0=h1)
    assert torch.equal(torch.cat([o1, o2]), out) and torch.equal(h2, hT)


def test_decode_steps_match_prefill():
    cfg = inputs.PrefillConfig("dec", H=2, dk=128, dv=128, dtype="bf16", B=1, T=20, h0_std=0.1, seed=306)
    inp = inputs.prefill_inputs(cfg, device="cuda")
    out, hT = run_prefill(inp)
    pool = torch.zeros(3, 2, 128, 128, device="cuda")
    pool[1] = inp["h0"][0]
    slot = torch.tensor([1], dtype=torch.int32, device="cuda")
    outs = []
    for t in range(20):
        outs.append(binding.kda_decode_step(*(inp[x][t:t + 1].contiguous() for x in ("q", "k", "v", "g", "beta")),
                                            pool, slot))
    dec = torch.cat(outs)
    assert parity_err(dec, out.double().cpu().numpy()) <= 2e-2
    assert rel_err(pool[1], hT[0].double().cpu().numpy()) <= 2e-2


def test_bad_cu_seqlens_sets_flag():
    cfg = inputs.PrefillConfig("bad", H=2, dk=128, dv=128, dtype="bf16", lengths=(10, 20), B=2, seed=307)
    inp = inputs.prefill_inputs(cfg, device="cuda")
    bad = torch.tensor([0, 25, 20], dtype=torch.int32, device="cuda")  # decreasing
    hT = torch.full((2, 2, 128, 128), 3.0, device="cuda")
    binding.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], cu_seqlens=bad, hT=hT)
    assert binding.kda_get_device_error() & binding.DEVERR_BAD_SEQLENS
    assert torch.all(hT == 3.0)  # skipped, untouched


# ------------------------------------------------------------------ long context: 1M tokens, H=16
def _window_start(g_host_f64, p, eps_log=math.log(1e-12), max_w=8192):
    """Smallest window start a such that prod_{t=a..p} max_c alpha_t < 1e-12 (all heads).
    For |k| = 1 and beta in [0, 1] each token's transition has operator norm <= max_c alpha_t,
    so restarting the recurrence from zero at a changes S_p by < 1e-12 * |S_{a-1}|."""
    acc = np.zeros(g_host_f64.shape[1])
    a = p
    while a >= 0 and p - a < max_w:
        acc += g_host_f64[a].max(axis=-1)
        if acc.max() < eps_log:
            return a
        a -= 1
    return max(a, 0)


@pytest.mark.slow
@pytest.mark.parametrize("cfg", [inputs.LONG, inputs.LONG_SLOW], ids=["z_mean+2", "z_mean-2"])
def test_long_context_1m_tokens(cfg):
    inp = inputs.prefill_inputs(cfg, device="cuda")
    T = inp["T_tot"]
    # (i) the first 65,536 tokens against the full oracle
    P = 65536
    pre = {x: inp[x][:P].contiguous() for x in ("q", "k", "v", "g", "beta")}
    o_p, h_p = binding.kda_chunk_fwd(pre["q"], pre["k"], pre["v"], pre["g"], pre["beta"])
    assert_no_device_error()
    ref_o, ref_h = oracle_kda_prefill(pre["q"], pre["k"], pre["v"], pre["g"], pre["beta"])
    assert parity_err(o_p, ref_o) <= 2e-2 and rel_err(h_p, ref_h) <= 2e-2
    del pre, o_p, h_p, ref_o, ref_h
    # (ii) the full sequence; spot rows against the oracle restarted on a provably sufficient window
    out, hT = binding.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"])
    assert_no_device_error()
    for p in [70000, 262143, 500001, 777777, T - 1]:
        gw = inp["g"][max(0, p - 8192):p + 1].double().cpu().numpy()
        a = max(0, p - 8192) + _window_start(gw, gw.shape[0] - 1)
        sl = slice(a, p + 1)
        ro, rh = oracle_kda_prefill(*(inp[x][sl] for x in ("q", "k", "v", "g", "beta")))
        assert parity_err(out[p], ro[-1]) <= 2e-2, p
        if p == T - 1:
            assert rel_err(hT[0], rh[0]) <= 2e-2


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_strong_decay_inside_chunk_with_weak_decay_across_the_half_boundary(dtype):
    """g near the bound over tokens 16..30 and 33..47 of every chunk but ~0 at 31..32: the
    off-diagonal-block entry for (r, s) = (32, 31) is O(1) while the cumulative decay between the
    two centred references (e^{G_47 - G_15} ~ e^{-142}) underflows fp32."""
    cfg = inputs.PrefillConfig("decay edge", H=2, dk=128, dv=128, dtype=dtype, B=1, T=256, h0_std=0.1, seed=308)
    inp = inputs.prefill_inputs(cfg, device="cpu")
    pos = torch.arange(256) % 64
    strong = ((pos >= 16) & (pos <= 30)) | ((pos >= 33) & (pos <= 47))
    g = torch.where(strong[:, None, None], torch.full_like(inp["g"], -4.9), torch.full_like(inp["g"], -0.01))
    inp["g"] = (g + 0.05 * inp["g"] / 5.0).contiguous()  # keep a little per-channel variation, g in (-5, 0)
    inp = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    ref_out, ref_hT = oracle_prefill(inp)
    out, hT = run_prefill(inp, out_dtype=torch.float32)
    assert_no_device_error()
    tol = TOL[inputs.torch_dtype(dtype)]
    assert rel_err(out, ref_out) <= tol and rel_err(hT, ref_hT) <= tol


@pytest.mark.parametrize("lengths,H,epilogue,z_mean", [
    ((16384,), 4, False, 0.0),
    ((20000, 300), 2, True, 0.0),
    ((8192,), 4, False, -8.0),
    ((6400,), 64, False, -8.0),             # two segments: the run of segment 0 from h0 is S_in(1), no merge
    ((4096, 4096), 16, False, -8.0),        # three segments planned, every sequence ends in segment 1
    ((2730, 2730, 2730), 16, False, -8.0),  # two segments planned, every sequence fits in segment 0
])
def test_sequence_split_across_sms_matches_oracle(lengths, H, epilogue, z_mean):
    """Few (sequence, head) chains with long sequences: the state pass is split into segments
    whose transitions are merged (intra-device context parallelism); results must not change.
    z_mean = -8 gives g close to 0 (decay ~e^-0.002 per token), so each segment's initial state,
    recovered by the merge, still shapes the segment's outputs and final state.  The segment
    counts in the comments are those of a 152-SM GPU; the last two cases leave every merge CTA,
    and in the last case every transition CTA, with nothing to do."""
    cfg = inputs.PrefillConfig("cp", H=H, dk=128, dv=128, dtype="bf16", lengths=lengths, B=len(lengths),
                               h0_std=0.1, epilogue=epilogue, z_mean=z_mean, seed=309)
    _check(cfg, epilogue=epilogue, device_gen=True)


# ------------------------------------------------------------------ prefix-cache checkpoints
@pytest.mark.parametrize("lengths,H,dk,dtype,ckpt_chunks,z_mean", [
    ((700, 1300, 64, 2000), 2, 128, "bf16", 4, 0.0),   # tensor-core path, varlen
    ((700, 1300, 64, 2000), 2, 64, "fp32", 4, 0.0),    # CUDA-core path
    ((700, 1300, 64, 2000), 2, 128, "fp32", 2, 0.0),   # CUDA-core path, one record stage, 8-CTA clusters
    ((8192,), 4, 128, "bf16", 8, -8.0),                # split into segments, slow decay
])
def test_checkpoints_match_the_oracle_on_each_prefix(lengths, H, dk, dtype, ckpt_chunks, z_mean):
    """Each stored state equals the oracle's final state on the sequence's prefix of
    j * 64 * ckpt_chunks tokens (from h0); out and hT are unchanged by storing them."""
    cfg = inputs.PrefillConfig("ckpt", H=H, dk=dk, dv=dk, dtype=dtype, lengths=lengths, B=len(lengths), h0_std=0.1,
                               z_mean=z_mean, seed=321)
    inp = inputs.prefill_inputs(cfg, device="cuda")
    kw = dict(h0=inp["h0"], cu_seqlens=inp["cu_seqlens"], B=len(lengths))
    out0, hT0 = binding.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], **kw)
    out, hT, states = binding.kda_chunk_fwd_checkpoints(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                                        ckpt_chunks=ckpt_chunks, **kw)
    assert_no_device_error()
    assert torch.equal(out, out0) and torch.equal(hT, hT0)
    span = 64 * ckpt_chunks
    # the checkpoint prefixes as one packed batch for the oracle
    starts = inp["cu_seqlens"].to("cpu").tolist()
    pieces, h0s = [], []
    for b, L in enumerate(lengths):
        for j in range(1, L // span + 1):
            pieces.append((starts[b], starts[b] + j * span))
            h0s.append(inp["h0"][b])
    assert states.shape[0] == len(pieces)
    sl = lambda x: torch.cat([inp[x][a:e] for a, e in pieces])
    cu = torch.tensor([0] + list(np.cumsum([e - a for a, e in pieces])), dtype=torch.int64)
    _, ref = oracle_kda_prefill(sl("q"), sl("k"), sl("v"), sl("g"), sl("beta"), h0=torch.stack(h0s), cu_seqlens=cu)
    assert rel_err(states, ref) <= TOL[inputs.torch_dtype(dtype)]
    # a checkpoint at a sequence's end is its final state
    idx = 0
    for b, L in enumerate(lengths):
        idx += L // span
        if L % span == 0 and L // span > 0:
            assert torch.equal(states[idx - 1], hT[b])
