"""Seeded synthetic KDA workloads.

This module only draws random tensors; it holds none of the method's arithmetic
(no decay, no recurrence, no chunking).  Both the CUDA path and the fp64 oracle
are fed from here.

Recipe (the five workloads of the KDA hot path, plus one labelled extra):
  - q, k ~ N(0, 1), then L2-normalised over the key dimension per (token, head)
    (upstream ShortConv + Swish + L2-norm of section 2.4 / Eq. 2 is outside the
    kernel; only its output norm is reproduced);
  - v ~ N(0, 1);  beta = sigmoid(N(0, 1));
  - g = -5 * sigmoid(z), z ~ N(z_mean, 1) per key channel (the lower-bounded
    decay of section 3.2 / Eq. 5 with g_min = -5 and log-scale A = 0);
  - h0 ~ N(0, h0_std) (standard deviation), or no initial state;
  - gate logits ~ N(0, 1) in the input dtype, RMSNorm weight = 1 + 0.1 N(0, 1);
  - variable lengths ~ U{lo..hi}; decode slots = a random permutation prefix.

Draw order: lengths (varlen only); then, per block of at most 65,536 tokens,
q, k, v, beta-logits, z and (when the epilogue is on) gate logits; then h0,
norm weight, slot permutation.  One torch.Generator seeded per workload; on a
CUDA device the generator lives on that device, so the values differ from a CPU
draw of the same recipe (each test hands the oracle host copies of exactly the
tensors the GPU consumed).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

BLOCK_TOKENS = 65536


@dataclasses.dataclass(frozen=True)
class PrefillConfig:
    name: str
    H: int
    dk: int
    dv: int
    dtype: str                 # "bf16" or "fp32" for q, k, v (and gate)
    B: int = 1
    T: int = 0                 # per-sequence length when lengths are equal
    len_range: Optional[tuple] = None   # (lo, hi) inclusive -> variable lengths
    lengths: Optional[tuple] = None     # explicit lengths (tests)
    z_mean: float = 0.0
    h0_std: float = 0.0
    epilogue: bool = False
    C: int = 64
    seed: int = 0


@dataclasses.dataclass(frozen=True)
class DecodeConfig:
    name: str
    N: int
    H: int
    dk: int
    dv: int
    num_slots: int
    dtype: str = "bf16"
    z_mean: float = 0.0
    state_std: float = 0.1
    epilogue: bool = True
    seed: int = 4
    n_tok: int = 1  # tokens per request (> 1: the multi-token layout [N, n_tok, H, ..])


# The hot path's workloads.
TINY = PrefillConfig("tiny fp32: B=1 H=2 T=256 dk=dv=64 C=64", H=2, dk=64, dv=64, dtype="fp32",
                     B=1, T=256, seed=0)
PREFILL = PrefillConfig("prefill bf16: B=1 H=32 T=8192 dk=dv=128 C=64", H=32, dk=128, dv=128,
                        dtype="bf16", B=1, T=8192, seed=1)
VARLEN = PrefillConfig("varlen bf16: 8 seqs len U[512,8192] H=32 dk=dv=128 h0~N(0,0.1)", H=32, dk=128,
                       dv=128, dtype="bf16", B=8, len_range=(512, 8192), h0_std=0.1, seed=2)
LONG = PrefillConfig("long bf16: B=1 H=16 T=1048576 dk=dv=128 z~N(2,1)", H=16, dk=128, dv=128,
                     dtype="bf16", B=1, T=1048576, z_mean=2.0, seed=3)
LONG_SLOW = PrefillConfig("long bf16 slow decay: B=1 H=16 T=1048576 dk=dv=128 z~N(-2,1)", H=16, dk=128,
                          dv=128, dtype="bf16", B=1, T=1048576, z_mean=-2.0, seed=5)
DECODE = DecodeConfig("decode bf16: N=256 H=32 dk=dv=128 pool=1024 fp32 states, RMSNorm+gate",
                      N=256, H=32, dk=128, dv=128, num_slots=1024, seed=4)

_TORCH_DTYPE = {"bf16": torch.bfloat16, "fp32": torch.float32}


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH_DTYPE[name]


def _gen(seed: int, device) -> torch.Generator:
    dev = torch.device(device)
    g = torch.Generator(device=dev) if dev.type == "cuda" else torch.Generator()
    g.manual_seed(seed)
    return g


def _unit(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)


def sequence_lengths(cfg: PrefillConfig) -> list:
    """Per-sequence lengths (drawn first, on a CPU generator, so that CPU and
    GPU draws of the same workload agree on the shapes)."""
    if cfg.lengths is not None:
        return [int(x) for x in cfg.lengths]
    if cfg.len_range is not None:
        lo, hi = cfg.len_range
        g = torch.Generator().manual_seed(cfg.seed)
        return [int(x) for x in torch.randint(lo, hi + 1, (cfg.B,), generator=g)]
    return [cfg.T] * cfg.B


def prefill_inputs(cfg: PrefillConfig, device="cpu") -> dict:
    """Returns a dict with q, k, v ([T_tot, H, d]), g ([T_tot, H, dk] fp32), beta ([T_tot, H] fp32),
    h0 ([B, H, dk, dv] fp32 or None), cu_seqlens (int32 [B+1] on device), lengths (list),
    gate ([T_tot, H, dv] or None), norm_weight ([dv] fp32 or None)."""
    lengths = sequence_lengths(cfg)
    T_tot = int(sum(lengths))
    gen = _gen(cfg.seed, device)
    dt = _TORCH_DTYPE[cfg.dtype]
    f32 = dict(device=device, dtype=torch.float32)
    q = torch.empty(T_tot, cfg.H, cfg.dk, device=device, dtype=dt)
    k = torch.empty_like(q)
    v = torch.empty(T_tot, cfg.H, cfg.dv, device=device, dtype=dt)
    g = torch.empty(T_tot, cfg.H, cfg.dk, **f32)
    beta = torch.empty(T_tot, cfg.H, **f32)
    gate = torch.empty(T_tot, cfg.H, cfg.dv, device=device, dtype=dt) if cfg.epilogue else None
    for t0 in range(0, T_tot, BLOCK_TOKENS):
        n = min(BLOCK_TOKENS, T_tot - t0)
        sl = slice(t0, t0 + n)
        q[sl] = _unit(torch.randn(n, cfg.H, cfg.dk, generator=gen, **f32)).to(dt)
        k[sl] = _unit(torch.randn(n, cfg.H, cfg.dk, generator=gen, **f32)).to(dt)
        v[sl] = torch.randn(n, cfg.H, cfg.dv, generator=gen, **f32).to(dt)
        beta[sl] = torch.sigmoid(torch.randn(n, cfg.H, generator=gen, **f32))
        z = torch.randn(n, cfg.H, cfg.dk, generator=gen, **f32) + cfg.z_mean
        g[sl] = -5.0 * torch.sigmoid(z)
        if gate is not None:
            gate[sl] = torch.randn(n, cfg.H, cfg.dv, generator=gen, **f32).to(dt)
    h0 = None
    if cfg.h0_std > 0:
        h0 = torch.randn(cfg.B, cfg.H, cfg.dk, cfg.dv, generator=gen, **f32) * cfg.h0_std
    norm_weight = None
    if cfg.epilogue:
        norm_weight = 1.0 + 0.1 * torch.randn(cfg.dv, generator=gen, **f32)
    cu = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    if lengths:
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    return dict(q=q, k=k, v=v, g=g, beta=beta, h0=h0, cu_seqlens=cu.to(device), lengths=lengths,
                gate=gate, norm_weight=norm_weight, T_tot=T_tot)


def decode_inputs(cfg: DecodeConfig, device="cpu") -> dict:
    """Returns q, k, v, g, beta for N requests, a state pool [num_slots, H, dk, dv] fp32
    (~N(0, state_std)), slot_idx (int32 [N], distinct), gate and norm_weight."""
    gen = _gen(cfg.seed, device)
    dt = _TORCH_DTYPE[cfg.dtype]
    f32 = dict(device=device, dtype=torch.float32)
    lead = (cfg.N, cfg.H) if cfg.n_tok == 1 else (cfg.N, cfg.n_tok, cfg.H)
    q = _unit(torch.randn(*lead, cfg.dk, generator=gen, **f32)).to(dt)
    k = _unit(torch.randn(*lead, cfg.dk, generator=gen, **f32)).to(dt)
    v = torch.randn(*lead, cfg.dv, generator=gen, **f32).to(dt)
    beta = torch.sigmoid(torch.randn(*lead, generator=gen, **f32))
    g = -5.0 * torch.sigmoid(torch.randn(*lead, cfg.dk, generator=gen, **f32) + cfg.z_mean)
    gate = torch.randn(*lead, cfg.dv, generator=gen, **f32).to(dt) if cfg.epilogue else None
    pool = torch.empty(cfg.num_slots, cfg.H, cfg.dk, cfg.dv, **f32)
    for s0 in range(0, cfg.num_slots, 64):  # bounded temporaries
        s1 = min(cfg.num_slots, s0 + 64)
        pool[s0:s1] = torch.randn(s1 - s0, cfg.H, cfg.dk, cfg.dv, generator=gen, **f32) * cfg.state_std
    norm_weight = (1.0 + 0.1 * torch.randn(cfg.dv, generator=gen, **f32)) if cfg.epilogue else None
    perm = torch.randperm(cfg.num_slots, generator=gen, device=device)
    slot_idx = perm[: cfg.N].to(torch.int32)
    return dict(q=q, k=k, v=v, g=g, beta=beta, state_pool=pool, slot_idx=slot_idx, gate=gate,
                norm_weight=norm_weight)
