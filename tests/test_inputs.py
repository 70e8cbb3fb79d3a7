"""The seeded synthetic inputs (CPU): shapes, dtypes and value ranges of each workload's recipe,
reproducibility, and the varlen workload's drawn lengths."""
import dataclasses

import torch

from gated_delta_rule_08_gb300 import inputs


def _check_prefill(inp, cfg, unit_tol):
    T, H = inp["T_tot"], cfg.H
    dt = inputs.torch_dtype(cfg.dtype)
    assert inp["q"].shape == (T, H, cfg.dk) and inp["k"].shape == (T, H, cfg.dk)
    assert inp["v"].shape == (T, H, cfg.dv) and inp["g"].shape == (T, H, cfg.dk)
    assert inp["beta"].shape == (T, H)
    assert inp["q"].dtype == dt and inp["v"].dtype == dt
    assert inp["g"].dtype == torch.float32 and inp["beta"].dtype == torch.float32
    for x in ("q", "k"):  # L2-normalised per (token, head)
        norms = inp[x].float().norm(dim=-1)
        assert torch.all((norms - 1).abs() < unit_tol), x
    assert torch.all((inp["beta"] > 0) & (inp["beta"] < 1))
    assert torch.all((inp["g"] > -5) & (inp["g"] < 0))
    cu = inp["cu_seqlens"]
    assert cu.dtype == torch.int32 and int(cu[0]) == 0 and int(cu[-1]) == T
    assert torch.all(cu[1:] >= cu[:-1])


def test_tiny_workload_recipe_and_reproducibility():
    a = inputs.prefill_inputs(inputs.TINY)
    b = inputs.prefill_inputs(inputs.TINY)
    _check_prefill(a, inputs.TINY, 1e-6)
    assert a["T_tot"] == 256 and a["h0"] is None and a["gate"] is None
    for x in ("q", "k", "v", "g", "beta"):
        assert torch.equal(a[x], b[x]), x


def test_bf16_prefill_recipe_on_a_short_copy():
    cfg = dataclasses.replace(inputs.PREFILL, T=300)
    inp = inputs.prefill_inputs(cfg)
    _check_prefill(inp, cfg, 1e-2)  # unit norms up to the bf16 rounding of each element


def test_varlen_lengths_and_initial_states():
    lengths = inputs.sequence_lengths(inputs.VARLEN)
    assert len(lengths) == 8 and all(512 <= n <= 8192 for n in lengths)
    assert sum(lengths) == 27654  # the token count the varlen measurements are quoted on
    cfg = dataclasses.replace(inputs.VARLEN, lengths=tuple(n // 64 for n in lengths))  # same recipe, short
    inp = inputs.prefill_inputs(cfg)
    _check_prefill(inp, cfg, 1e-2)
    assert inp["h0"].shape == (8, 32, 128, 128) and abs(float(inp["h0"].std()) - 0.1) < 0.01


def test_slow_decay_variant_decays_slower():
    fast = inputs.prefill_inputs(dataclasses.replace(inputs.LONG, T=128))
    slow = inputs.prefill_inputs(dataclasses.replace(inputs.LONG_SLOW, T=128))
    assert float(fast["g"].mean()) < -3.5 and float(slow["g"].mean()) > -1.5


def test_decode_recipe_one_and_several_tokens():
    cfg = dataclasses.replace(inputs.DECODE, N=8, H=2, num_slots=16)
    d = inputs.decode_inputs(cfg)
    assert d["q"].shape == (8, 2, 128) and d["g"].shape == (8, 2, 128) and d["beta"].shape == (8, 2)
    assert d["state_pool"].shape == (16, 2, 128, 128) and d["state_pool"].dtype == torch.float32
    s = d["slot_idx"]
    assert s.dtype == torch.int32 and len(set(s.tolist())) == 8 and int(s.min()) >= 0 and int(s.max()) < 16
    assert torch.all((d["g"] > -5) & (d["g"] < 0)) and torch.all((d["beta"] > 0) & (d["beta"] < 1))
    assert d["gate"].shape == (8, 2, 128) and d["norm_weight"].shape == (128,)
    m = inputs.decode_inputs(dataclasses.replace(cfg, n_tok=4))
    assert m["q"].shape == (8, 4, 2, 128) and m["beta"].shape == (8, 4, 2) and m["gate"].shape == (8, 4, 2, 128)
