"""One workload of the hot path, run alone a few times: a target for a profiler (ncu) that should
see one kernel family on a small device footprint.

    python -m gated_delta_rule_08_gb300.profile_cases prefill|prefill_epi|varlen|decode|verify|backward|prefill_d64|
        prefill_d64_epi
        [--calls N]

prefill      B=1, H=32, T=8192, dk=dv=128, bf16 (q, k, v, g, beta: 337 MB; records 310 MB)
prefill_epi  the same with the RMSNorm + sigmoid gate epilogue
varlen       8 sequences, 27,654 tokens, H=32, dk=dv=128, bf16, h0
decode       N=256 requests, H=32, 1024-slot fp32 pool (2 GiB), RMSNorm + gate
verify       the decode workload with 4 draft tokens per request, pool not written
backward     the prefill workload's gradients (chunkwise path)
prefill_d64  B=1, H=32, T=8192, dk=dv=64, bf16 (the CUDA-core prefill path)
prefill_d64_epi  the same with the RMSNorm + sigmoid gate epilogue

Every call goes through the C-ABI binding; the first call is a warm-up.  Nothing is timed here.
"""
from __future__ import annotations

import argparse
import dataclasses
import sys

import torch

from . import binding, inputs


def _prefill(cfg, calls, dev):
    P = inputs.prefill_inputs(cfg, device=dev)
    varlen = cfg.len_range is not None or cfg.lengths is not None
    kw = {"cu_seqlens": P["cu_seqlens"]} if varlen else {"B": len(P["lengths"])}
    if cfg.epilogue:
        kw.update(gate=P["gate"], norm_weight=P["norm_weight"])
    for _ in range(calls + 1):
        binding.kda_chunk_fwd(P["q"], P["k"], P["v"], P["g"], P["beta"], h0=P["h0"], **kw)


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["prefill", "prefill_epi", "varlen", "decode", "verify", "backward", "prefill_d64",
                                     "prefill_d64_epi"])
    ap.add_argument("--calls", type=int, default=2)
    args = ap.parse_args(argv)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if args.case in ("prefill", "prefill_epi"):
        _prefill(dataclasses.replace(inputs.PREFILL, epilogue=args.case == "prefill_epi"), args.calls, dev)
    elif args.case == "varlen":
        _prefill(inputs.VARLEN, args.calls, dev)
    elif args.case in ("prefill_d64", "prefill_d64_epi"):
        _prefill(dataclasses.replace(inputs.PREFILL, dk=64, dv=64, name="prefill d64",
                                     epilogue=args.case.endswith("_epi")), args.calls, dev)
    elif args.case in ("decode", "verify"):
        cfg = inputs.DECODE if args.case == "decode" else dataclasses.replace(inputs.DECODE, n_tok=4)
        D = inputs.decode_inputs(cfg, device=dev)
        for _ in range(args.calls + 1):
            if args.case == "decode":
                binding.kda_decode_step(D["q"], D["k"], D["v"], D["g"], D["beta"], D["state_pool"], D["slot_idx"],
                                        gate=D["gate"], norm_weight=D["norm_weight"])
            else:
                binding.kda_decode_multi(D["q"], D["k"], D["v"], D["g"], D["beta"], D["state_pool"], D["slot_idx"],
                                         commit=False, gate=D["gate"], norm_weight=D["norm_weight"])
    else:
        P = inputs.prefill_inputs(inputs.PREFILL, device=dev)
        gen = torch.Generator(device=dev).manual_seed(11)
        dout = torch.randn(P["T_tot"], 32, 128, generator=gen, device=dev).to(torch.bfloat16)
        for _ in range(args.calls + 1):
            binding.kda_chunk_bwd(P["q"], P["k"], P["v"], P["g"], P["beta"], dout)
    torch.cuda.synchronize()
    flags = binding.kda_get_device_error(dev)
    if flags:
        sys.stderr.write(f"device error word {flags:#x}\n")
        return 1
    return 0


if __name__ == "__main__":
    sys.exit(main())
