"""Helpers for the GPU parity tests: run the CUDA path through the binding, run the
fp64 oracle on host copies of exactly the same tensors, and compare."""
from __future__ import annotations

import numpy as np
import torch

from gated_delta_rule_08_gb300 import binding
from oracle import oracle_kda_decode, oracle_kda_prefill

# max|gpu - oracle| / RMS(oracle), per output tensor
TOL = {torch.float32: 1e-3, torch.bfloat16: 2e-2}


# unit roundoff of the storage format of a result: rounding the exact value into it
# moves it by at most this fraction of its magnitude
STORAGE_ROUNDOFF = {torch.float32: 0.0, torch.bfloat16: 2.0 ** -8}


def rel_err(gpu, ref) -> float:
    """max|gpu - ref| / RMS(ref)."""
    return parity_err(gpu, ref, torch.float32)


def parity_err(gpu, ref, stored=None) -> float:
    """max_i (|gpu_i - ref_i| - u |ref_i|) / RMS(ref), u = unit roundoff of the dtype the
    GPU result is stored in (0 for fp32).  For fp32 storage this is the plain
    max|err|/RMS; for bf16 storage it removes the one rounding that even the exact
    result incurs when written as bf16, and bounds everything else."""
    if stored is None:
        stored = gpu.dtype if hasattr(gpu, "dtype") else torch.float32
    g = gpu.detach().to("cpu").double().numpy() if hasattr(gpu, "detach") else np.asarray(gpu, np.float64)
    r = np.asarray(ref, dtype=np.float64)
    if not r.size:
        return 0.0
    rms = float(np.sqrt(np.mean(r * r)))
    excess = np.abs(g - r) - STORAGE_ROUNDOFF[stored] * np.abs(r)
    if rms == 0.0:
        return float(max(0.0, excess.max()))
    return float(max(0.0, excess.max()) / rms)


def run_prefill(inp, *, epilogue=None, h0=None, out_final=True, out_dtype=None):
    gate = inp.get("gate") if epilogue is None else (inp.get("gate") if epilogue else None)
    nw = inp.get("norm_weight") if gate is not None else None
    B = len(inp["lengths"])
    return binding.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                 h0=inp.get("h0") if h0 is None else h0, cu_seqlens=inp["cu_seqlens"], B=B,
                                 gate=gate, norm_weight=nw, output_final_state=out_final, out_dtype=out_dtype)


def oracle_prefill(inp, *, epilogue=None, h0=None):
    gate = inp.get("gate") if epilogue is None else (inp.get("gate") if epilogue else None)
    nw = inp.get("norm_weight") if gate is not None else None
    return oracle_kda_prefill(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                              h0=inp.get("h0") if h0 is None else h0,
                              cu_seqlens=inp["cu_seqlens"].to("cpu").to(torch.int64), gate=gate, norm_weight=nw)


def to_device(inp, device="cuda"):
    out = {}
    for key, val in inp.items():
        out[key] = val.to(device) if isinstance(val, torch.Tensor) else val
    return out


def assert_no_device_error():
    flags = binding.kda_get_device_error()
    assert flags == 0, f"device error word = {flags:#x}"
