"""KDA hot-path benchmark: chunked prefill + pooled decode on GB300.

One step = one kda_chunk_fwd over the prefill workload (B=1, H=32, T=8192,
dk=dv=128, bf16 q/k/v, fp32 g/beta, h0=0, C=64, out + final fp32 state) followed by
one kda_decode_step over the decode workload (N=256, H=32, dk=dv=128, fp32 state
pool of 1024 slots, fused RMSNorm + sigmoid gate).  `value` is prefill tokens/s
(the metric's first half, timed on the prefill calls of the timed steps); decode
steps/s is reported beside it.  Inputs are synthetic (seeded), resident in HBM and
larger than L2 (prefill 404 MB, decode 1.07 GB of touched state), so no L2 flush
is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the only reference implementation this
method has here) on the host cores, on the same workload and metric.
Under torchrun (N > 1) every rank runs the same per-GPU workload (independent
problems: weak scaling, no collective on the data path); timing is the max over
ranks and value aggregates all ranks.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s (bf16, H=32, dk=dv=128) + decode steps/s, % of roofline"
PREFILL_BYTES_PER_TOKEN_HEAD = 3 * 2 * 128 + 4 * 128 + 4 + 2 * 128        # q,k,v bf16 + g fp32 + beta + out bf16
PREFILL_FLOPS_PER_TOKEN_HEAD = 2 * (5 * 64 * 128 + 3 * 128 * 128)          # method's flop count at C=64, d=128
PREP_BYTES_PER_TOKEN_HEAD = 3 * 2 * 128 + 4 * 128 + 4                      # the chunk-parallel kernel's inputs
STATE_BYTES = 128 * 128 * 4                                                # one fp32 state (h0 or hT)


def prefill_bytes_per_token_head(dk: int, dv: int) -> int:
    """q, k (bf16, dk each), v (bf16, dv), g (fp32, dk), beta (fp32), out (bf16, dv)."""
    return 2 * (2 * dk + dv) + 4 * dk + 4 + 2 * dv
DECODE_STATE_BYTES = 2 * 128 * 128 * 4                                    # read + write of one fp32 state
DECODE_IO_BYTES_PER_TOKEN_HEAD = 3 * 2 * 128 + 4 * 128 + 4 + 2 * 128 + 2 * 128  # q,k,v,g,beta,gate,out
# chunkwise backward, per (chunk, head) at C=64, d=128: 14 C x C x d products (records A, M, W, U_hat;
# M^T dO; dM, dU V^T, T^T dU; dW K_hat^T, T^T dW and the four A/M-term products), 8 C x d x d
# (U, the state update, K_bar dS, Q_hat^T dO, W^T dU, dQ_hat, dW, dK_bar) and 2 C^3 (X^T dX X^T)
BWD_FLOPS_PER_CHUNK_HEAD = 2 * (14 * 64 * 64 * 128 + 8 * 64 * 128 * 128 + 2 * 64 ** 3)
FP32_LANES_PER_SM = 128                                                   # FP32 FMA lanes per SM (4 x 32)
TF32_PER_BF16_NOMINAL = 1.1 / 2.25                                        # dense tensor peaks, tf32 / bf16


def _env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", 0)), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


# the files that define each profiled kernel and its launch shape; a kernel's recorded traffic
# stands only while these hash to the digest recorded with it
_TC_HEADERS = ("kda_tc_common.cuh", "tc_ptx.cuh", "kda_device.cuh", "kda_internal.h")
KERNEL_SOURCES = {
    "kda_tc_chunk_prep": ("kda_prefill_tc.cu",) + _TC_HEADERS,
    "kda_tc_chunk_scan_transition": ("kda_scan_tc.cu",) + _TC_HEADERS,
    "kda_cp_merge": ("kda_scan_tc.cu",) + _TC_HEADERS,
    "kda_tc_chunk_scan": ("kda_scan_tc.cu",) + _TC_HEADERS,
    "kda_decode": ("kda_decode.cu", "kda_device.cuh", "kda_internal.h"),
}


def source_digest(names) -> str:
    """sha256 over the named sources (names and contents, in the given order)."""
    import hashlib
    d = os.path.join(ROOT, "gated_delta_rule_08_gb300", "csrc")
    hsh = hashlib.sha256()
    for name in names:
        hsh.update(name.encode())
        with open(os.path.join(d, name), "rb") as f:
            hsh.update(f.read())
    return hsh.hexdigest()


def measured_traffic() -> dict:
    """Per-kernel DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from the
    committed ncu capture, for the kernels whose sources are unchanged since it was taken."""
    path = os.path.join(ROOT, "profiles", "kda_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return {}
    out = {}
    for k, v in rec.get("kernels", {}).items():
        if k in KERNEL_SOURCES and v.get("source_sha256") == source_digest(KERNEL_SOURCES[k]):
            out[k] = v["dram_bytes_per_launch"]
    return out


def call_traffic(traffic: dict, kernels: dict):
    """DRAM bytes of one prefill call: the sum over its kernels of the captured bytes per launch, or
    None unless every kernel of the call has a capture that matches its current sources."""
    if not kernels or any(k not in traffic for k in kernels):
        return None
    calls = min(v[0] for v in kernels.values())
    return int(sum(traffic[k] * v[0] / calls for k, v in kernels.items()))


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while the GPU works.  It is entered
    before the warm-up steps and waits for nvidia-smi's first sample, so that the timed steps and
    the traced pass after them are sampled in full (a few tens of milliseconds of GPU time)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (FileNotFoundError, OSError):
            self.proc = None
            return self
        import threading
        self._lines = []
        self._reader = threading.Thread(target=lambda: self._lines.extend(iter(self.proc.stdout.readline, "")),
                                        daemon=True)
        self._reader.start()
        t_end = time.monotonic() + 5.0
        while not self._lines and time.monotonic() < t_end and self.proc.poll() is None:
            time.sleep(0.01)
        return self

    def __exit__(self, *exc):
        if self.proc is None:  # never started, or already stopped
            self.lines = getattr(self, "lines", [])
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        self._reader.join(timeout=5)
        self.lines = [ln for ln in self._lines if ln.strip()]
        self.proc = None

    def summary(self):
        if not getattr(self, "lines", None):
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm),
                "window": "warm-up steps, timed steps and the traced pass"}


def _dist():
    world = _env_int("WORLD_SIZE", 1)
    rank = _env_int("RANK", 0)
    local = _env_int("LOCAL_RANK", 0)
    return world, rank, local


def dist_max(value: float, world: int) -> float:
    """Max of a per-rank float over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return units_per_rank * world / max_seconds


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def run_ours(args, world, rank, local):
    import torch

    from gated_delta_rule_08_gb300 import binding, inputs

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    hbm_gbs, bf16_tflops, _, peak_kind = _peaks()

    pcfg, dcfg = inputs.PREFILL, inputs.DECODE
    P = inputs.prefill_inputs(pcfg, device=dev)
    D = inputs.decode_inputs(dcfg, device=dev)
    T, H = P["T_tot"], pcfg.H
    out = torch.empty(T, H, pcfg.dv, device=dev, dtype=torch.bfloat16)
    hT = torch.empty(1, H, pcfg.dk, pcfg.dv, device=dev, dtype=torch.float32)
    ws = torch.empty(binding.kda_chunk_fwd_workspace_size(1, T, H, pcfg.dk, pcfg.dv), device=dev, dtype=torch.uint8)
    dout = torch.empty(dcfg.N, dcfg.H, dcfg.dv, device=dev, dtype=torch.bfloat16)

    def prefill():
        binding.kda_chunk_fwd(P["q"], P["k"], P["v"], P["g"], P["beta"], out=out, hT=hT, workspace=ws)

    def decode():
        binding.kda_decode_step(D["q"], D["k"], D["v"], D["g"], D["beta"], D["state_pool"], D["slot_idx"], out=dout,
                                gate=D["gate"], norm_weight=D["norm_weight"])

    clocks = ClockSampler(local).__enter__()  # sampling from the warm-up through the traced pass
    try:
        for _ in range(args.warmup):
            prefill()
            decode()
        torch.cuda.synchronize()
        assert binding.kda_get_device_error(dev) == 0

        stream = torch.cuda.current_stream(dev)

        def timed_steps():
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
                   torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
            for i in range(args.steps):
                ev[i][0].record(stream)
                prefill()
                ev[i][1].record(stream)
                decode()
                ev[i][2].record(stream)
            return ev

        # the headline: K steps with nothing between the kernels of a call (the state-pass kernels
        # start while their predecessor drains)
        _barrier(world)
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        ev = timed_steps()
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
        _barrier(world)
        # the same K steps again with every kernel bracketed by CUDA events on its stream: per-kernel
        # durations for the roofline (the events cost the overlap above, so this pass is not the value)
        binding.kda_trace_enable(True)
        binding.kda_trace_collect()  # drop anything recorded before this pass
        ev_traced = timed_steps()
        torch.cuda.synchronize()
        _barrier(world)
        trace = binding.kda_trace_collect()
        binding.kda_trace_enable(False)
    finally:
        clocks.__exit__(None, None, None)
    pre_ms = [a.elapsed_time(b) for a, b, _ in ev]
    dec_ms = [b.elapsed_time(c) for _, b, c in ev]
    pre_s = dist_max(sum(pre_ms) / 1e3, world)
    dec_s = dist_max(sum(dec_ms) / 1e3, world)
    step_s = dist_max(sum(a.elapsed_time(c) for a, _, c in ev) / 1e3, world)

    value = aggregate(T * args.steps, world, pre_s)
    dec_steps_per_s = aggregate(args.steps, world, dec_s)

    # the whole prefill call against the HBM roofline (the headline), and its dominant kernel on its
    # own inputs (the largest summed time among the prefill-side kernels)
    pre_k = {k: v for k, v in trace.items() if k != "kda_decode"}
    dom = max(pre_k.items(), key=lambda kv: kv[1][1])
    dom_ms = dom[1][1] / dom[1][0]
    alg_bytes = PREFILL_BYTES_PER_TOKEN_HEAD * T * H
    call_ms = pre_s * 1e3 / args.steps
    achieved = alg_bytes / (call_ms * 1e-3) / 1e9
    dom_bytes = PREP_BYTES_PER_TOKEN_HEAD * T * H if dom[0] == "kda_tc_chunk_prep" else None
    dec_launch = trace.get("kda_decode", (1, float("nan")))
    dec_ms_k = dec_launch[1] / dec_launch[0]
    dec_bytes = DECODE_STATE_BYTES * dcfg.N * dcfg.H + dcfg.N * dcfg.H * (3 * 2 * 128 + 4 * 128 + 4 + 2 * 128 + 2 * 128)
    dec_achieved = dec_bytes / (dec_ms_k * 1e-3) / 1e9
    pre_flops = PREFILL_FLOPS_PER_TOKEN_HEAD * T * H
    launches = sum(v[0] for v in trace.values())
    traffic = measured_traffic()

    # end to end through the public API with host buffers: every step uploads its inputs from
    # pinned host memory, makes the call and downloads its outputs.  Two buffer sets and three
    # streams let step i+1's upload and step i-1's download overlap step i's call.
    host = {k: P[k].to("cpu").pin_memory() for k in ("q", "k", "v", "g", "beta")}
    nb = 2
    dev_in = [{k: torch.empty_like(P[k]) for k in host} for _ in range(nb)]
    outs = [torch.empty_like(out) for _ in range(nb)]
    hTs = [torch.empty_like(hT) for _ in range(nb)]
    out_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(nb)]
    hT_h = [torch.empty(hT.shape, dtype=hT.dtype).pin_memory() for _ in range(nb)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h[0].numel() * out_h[0].element_size() + hT_h[0].numel() * hT_h[0].element_size()
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    in_done = [torch.cuda.Event() for _ in range(nb)]
    call_done = [torch.cuda.Event() for _ in range(nb)]
    out_done = [torch.cuda.Event() for _ in range(nb)]

    def e2e_run(nsteps, start_event=None, end_event=None):
        if start_event is not None:
            start_event.record(s_in)
        for i in range(nsteps):
            b = i % nb
            if i >= nb:
                s_in.wait_event(call_done[b])  # the call nb steps back has read this input set
            with torch.cuda.stream(s_in):
                for k in host:
                    dev_in[b][k].copy_(host[k], non_blocking=True)
            in_done[b].record(s_in)
            stream.wait_event(in_done[b])
            if i >= nb:
                stream.wait_event(out_done[b])  # the download nb steps back has read this output set
            binding.kda_chunk_fwd(dev_in[b]["q"], dev_in[b]["k"], dev_in[b]["v"], dev_in[b]["g"], dev_in[b]["beta"],
                                  out=outs[b], hT=hTs[b], workspace=ws)
            call_done[b].record(stream)
            s_out.wait_event(call_done[b])
            with torch.cuda.stream(s_out):
                out_h[b].copy_(outs[b], non_blocking=True)
                hT_h[b].copy_(hTs[b], non_blocking=True)
            out_done[b].record(s_out)
        if end_event is not None:
            stream.wait_stream(s_out)
            end_event.record(stream)

    e2e_run(max(1, args.warmup))
    torch.cuda.synchronize()
    _barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_run(args.steps, e0, e1)
    torch.cuda.synchronize()
    e2e_s = dist_max(e0.elapsed_time(e1) / 1e3, world)
    e2e_value = aggregate(T * args.steps, world, e2e_s)
    assert binding.kda_get_device_error(dev) == 0
    # the pipelined calls computed what the resident-input calls did
    assert torch.equal(out_h[(args.steps - 1) % nb], out.cpu()) and torch.equal(hT_h[(args.steps - 1) % nb], hT.cpu())

    # the next rows, each timed beside the step (not part of the metric) against its own roofline
    def time_calls(fn, calls):
        fn()
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for _ in range(calls):
            fn()
        c1.record(stream)
        torch.cuda.synchronize()
        assert binding.kda_get_device_error(dev) == 0
        return dist_max(c0.elapsed_time(c1) / calls, world)

    # prefill with the prefix-cache checkpoints (the state every 512 tokens)
    ckpt_chunks = 8
    n_ckpt = T // (64 * ckpt_chunks)
    states = torch.empty(n_ckpt, H, pcfg.dk, pcfg.dv, device=dev, dtype=torch.float32)
    ckpt_ms = time_calls(lambda: binding.kda_chunk_fwd_checkpoints(
        P["q"], P["k"], P["v"], P["g"], P["beta"], out=out, hT=hT, states=states, ckpt_chunks=ckpt_chunks,
        workspace=ws), max(3, args.steps))
    ckpt_bytes = alg_bytes + states.numel() * 4
    # speculative-decode verify: 4 draft tokens per request, the pool read once and not written
    vcfg = dataclasses.replace(dcfg, n_tok=4)
    V = inputs.decode_inputs(vcfg, device=dev)
    vout = torch.empty(vcfg.N, vcfg.n_tok, vcfg.H, vcfg.dv, device=dev, dtype=torch.bfloat16)
    ver_ms = time_calls(lambda: binding.kda_decode_multi(
        V["q"], V["k"], V["v"], V["g"], V["beta"], V["state_pool"], V["slot_idx"], out=vout, commit=False,
        gate=V["gate"], norm_weight=V["norm_weight"]), max(3, args.steps))
    ver_bytes = vcfg.N * vcfg.H * DECODE_STATE_BYTES // 2 + \
        vcfg.N * vcfg.n_tok * vcfg.H * DECODE_IO_BYTES_PER_TOKEN_HEAD
    del V
    # backward of the prefill recurrence (no epilogue) on the same workload, fp32 on the CUDA cores
    gen = torch.Generator(device=dev).manual_seed(11)
    dout = torch.randn(out.shape, generator=gen, device=dev).to(out.dtype)
    bws = torch.empty(binding.kda_chunk_bwd_workspace_size(1, T, H, pcfg.dk, pcfg.dv), device=dev, dtype=torch.uint8)
    bwd_ms = time_calls(lambda: binding.kda_chunk_bwd(P["q"], P["k"], P["v"], P["g"], P["beta"], dout,
                                                      workspace=bws), 2)
    del bws
    bwd_flops = BWD_FLOPS_PER_CHUNK_HEAD * (T // 64) * H
    del P, D, ws
    torch.cuda.empty_cache()
    # the other prefill workloads, each timed on its own with its whole-call HBM roofline
    others = {}
    if not args.skip_other_workloads:
        others["varlen"] = prefill_workload(inputs.VARLEN, max(3, args.steps), dev, hbm_gbs, peak_kind, world,
                                            time_calls)
        others["long"] = prefill_workload(inputs.LONG, 3, dev, hbm_gbs, peak_kind, world, time_calls)
        # the prefill workload with the fused RMSNorm + sigmoid-gate epilogue
        others["prefill_epilogue"] = prefill_workload(
            dataclasses.replace(inputs.PREFILL, epilogue=True, name="prefill B=1 H=32 T=8192 dk=dv=128 bf16 "
                                                                  "+ RMSNorm + gate"),
            max(3, args.steps), dev, hbm_gbs, peak_kind, world, time_calls)
        # 64-dim heads: the same shape as the prefill workload, carried by the CUDA-core prefill
        others["prefill_d64"] = prefill_workload(
            dataclasses.replace(inputs.PREFILL, dk=64, dv=64, name="prefill B=1 H=32 T=8192 dk=dv=64 bf16"),
            max(3, args.steps), dev, hbm_gbs, peak_kind, world, time_calls)
    csum = clocks.summary() or {}
    sm_max_mhz = csum.get("sm_max_mhz") or 2070.0
    fp32_tflops = torch.cuda.get_device_properties(dev).multi_processor_count * FP32_LANES_PER_SM * 2 * \
        sm_max_mhz * 1e6 / 1e12
    tf32_tflops = bf16_tflops * TF32_PER_BF16_NOMINAL
    bwd_tflops = bwd_flops / (bwd_ms * 1e-3) / 1e12

    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_s * 1e3 / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; q,k L2-normalised N(0,1), v N(0,1), beta=sigmoid(N), g=-5*sigmoid(N))",
        "config": {"workload": "prefill B=1 H=32 T=8192 dk=dv=128 C=64 bf16, h0=0, out+hT; then decode N=256 "
                               "H=32 dk=dv=128 pool=1024 fp32 slots, RMSNorm+gate",
                   "prefill_ms_per_step": round(pre_s * 1e3 / args.steps, 4),
                   "prefill_ms_per_step_traced": round(sum(x.elapsed_time(y) for x, y, _ in ev_traced) / args.steps, 4),
                   "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{world}"},
        "decode": {"steps_per_s": round(dec_steps_per_s, 1),
                   "tokens_per_s": round(dec_steps_per_s * dcfg.N, 1),
                   "ms_per_step": round(dec_s * 1e3 / args.steps, 4),
                   "roofline": {"bound": "hbm", "achieved": round(dec_achieved, 1), "peak": hbm_gbs, "unit": "GB/s",
                                "frac": round(dec_achieved / hbm_gbs, 4), "traffic": traffic.get("kda_decode"),
                                "kernel": "kda_decode", "peak_kind": peak_kind}},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_gbs, "unit": "GB/s",
                     "frac": round(achieved / hbm_gbs, 4), "traffic": call_traffic(traffic, pre_k),
                     "kernel": "kda_chunk_fwd (whole call: " + ", ".join(sorted(pre_k)) + ")",
                     "scope": "whole call", "call_ms": round(call_ms, 4), "peak_kind": peak_kind,
                     "algorithmic_bytes_per_call": alg_bytes,
                     "dominant_kernel": {
                         "kernel": dom[0], "kernel_ms": round(dom_ms, 4), "traffic": traffic.get(dom[0]),
                         "algorithmic_bytes_per_launch": dom_bytes,
                         "achieved": round(dom_bytes / (dom_ms * 1e-3) / 1e9, 1) if dom_bytes else None,
                         "frac": round(dom_bytes / (dom_ms * 1e-3) / 1e9 / hbm_gbs, 4) if dom_bytes else None,
                         "bytes": "its inputs q, k, v, g, beta (1284 B per token and head); the records it "
                                  "writes are not algorithmic bytes"}},
        "prefill_tensor": {"flops_per_step": pre_flops,
                           "achieved_tflops": round(pre_flops / (pre_s / args.steps) / 1e12, 2),
                           "peak_tflops": bf16_tflops,
                           "frac": round(pre_flops / (pre_s / args.steps) / 1e12 / bf16_tflops, 4)},
        "kernels": {k: {"launches": v[0], "total_ms": round(v[1], 4)} for k, v in trace.items()},
        "gpu_launches": launches,
        "checkpoints": {"workload": f"the prefill workload, state stored every {64 * ckpt_chunks} tokens "
                                    f"({n_ckpt} x {H} fp32 states)",
                        "ms_per_call": round(ckpt_ms, 4), "tokens_per_s": round(aggregate(T, world, ckpt_ms / 1e3), 1),
                        "roofline": {"bound": "hbm", "achieved": round(ckpt_bytes / (ckpt_ms * 1e-3) / 1e9, 1),
                                     "peak": hbm_gbs, "unit": "GB/s", "peak_kind": peak_kind,
                                     "frac": round(ckpt_bytes / (ckpt_ms * 1e-3) / 1e9 / hbm_gbs, 4),
                                     "algorithmic_bytes_per_call": ckpt_bytes, "scope": "whole call"}},
        "verify": {"workload": f"decode N={vcfg.N} requests x {vcfg.n_tok} draft tokens, H={vcfg.H}, pool not "
                               "written (commit=0), RMSNorm+gate",
                   "ms_per_call": round(ver_ms, 4),
                   "tokens_per_s": round(aggregate(vcfg.N * vcfg.n_tok, world, ver_ms / 1e3), 1),
                   "roofline": {"bound": "hbm", "achieved": round(ver_bytes / (ver_ms * 1e-3) / 1e9, 1),
                                "peak": hbm_gbs, "unit": "GB/s", "peak_kind": peak_kind,
                                "frac": round(ver_bytes / (ver_ms * 1e-3) / 1e9 / hbm_gbs, 4),
                                "algorithmic_bytes_per_call": ver_bytes, "scope": "whole call"}},
        "backward": {"ms_per_call": round(bwd_ms, 3), "tokens_per_s": round(aggregate(T, world, bwd_ms / 1e3), 1),
                     "kernel": "chunkwise: per-chunk records, serial state passes over chunks, per-chunk "
                               "gradients; products as three-term tf32 warp MMAs, the rest fp32",
                     "roofline": {"bound": "tensor", "achieved": round(bwd_tflops, 2),
                                  "peak": round(tf32_tflops, 1), "unit": "TFLOP/s",
                                  "peak_kind": f"tf32 dense = measured bf16 x nominal {TF32_PER_BF16_NOMINAL:.3f}",
                                  "frac": round(bwd_tflops / tf32_tflops, 4),
                                  "frac_of_fp32_fma": round(bwd_tflops / fp32_tflops, 4),
                                  "algorithmic_flops_per_call": bwd_flops, "scope": "whole call"}},
        **others,
        "e2e": {"value": round(e2e_value, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "clocks": csum or None,
        "wall_s": round(t_wall, 3),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args)
        if "long" in line:
            line["long"]["cpu_baseline"] = cpu_baseline_long(args)
    return line


def prefill_workload(cfg, calls, dev, hbm_gbs, peak_kind, world, time_calls):
    """ms per kda_chunk_fwd call on a prefill workload (inputs resident in HBM), its tokens/s and
    its whole-call HBM roofline (q, k, v, g, beta in, out written, plus h0 read and hT written)."""
    import torch

    from gated_delta_rule_08_gb300 import binding, inputs

    P = inputs.prefill_inputs(cfg, device=dev)
    T_tot, H, B = P["T_tot"], cfg.H, len(P["lengths"])
    varlen = cfg.len_range is not None or cfg.lengths is not None
    kw = {"cu_seqlens": P["cu_seqlens"]} if varlen else {"B": B}
    out = torch.empty(T_tot, H, cfg.dv, device=dev, dtype=torch.bfloat16)
    hT = torch.empty(B, H, cfg.dk, cfg.dv, device=dev, dtype=torch.float32)
    ws = torch.empty(binding.kda_chunk_fwd_workspace_size(B, T_tot if varlen else T_tot // B, H, cfg.dk, cfg.dv),
                     device=dev, dtype=torch.uint8)
    if cfg.epilogue:
        kw.update(gate=P["gate"], norm_weight=P["norm_weight"])
    ms = time_calls(lambda: binding.kda_chunk_fwd(P["q"], P["k"], P["v"], P["g"], P["beta"], h0=P["h0"], out=out,
                                                  hT=hT, workspace=ws, **kw), calls)
    nbytes = prefill_bytes_per_token_head(cfg.dk, cfg.dv) * T_tot * H + \
        B * H * cfg.dk * cfg.dv * 4 * (2 if P["h0"] is not None else 1) + \
        (2 * cfg.dv * T_tot * H + 4 * cfg.dv if cfg.epilogue else 0)  # gate logits (bf16) and the norm weight
    achieved = nbytes / (ms * 1e-3) / 1e9
    del P, out, hT, ws
    torch.cuda.empty_cache()
    return {"workload": cfg.name + f" ({T_tot} tokens)", "ms_per_call": round(ms, 4),
            "tokens_per_s": round(aggregate(T_tot, world, ms / 1e3), 1),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_gbs, "unit": "GB/s",
                         "frac": round(achieved / hbm_gbs, 4), "peak_kind": peak_kind,
                         "algorithmic_bytes_per_call": nbytes, "scope": "whole call"}}


def _oracle_prefill_sample(tokens: int):
    """The oracle on the first `tokens` tokens of the prefill workload (all 32 heads)."""
    import dataclasses

    from gated_delta_rule_08_gb300 import inputs
    from oracle import oracle_kda_prefill, oracle_threads

    cfg = dataclasses.replace(inputs.PREFILL, T=tokens)
    P = inputs.prefill_inputs(cfg, device="cpu")
    t0 = time.perf_counter()
    oracle_kda_prefill(P["q"], P["k"], P["v"], P["g"], P["beta"])
    return time.perf_counter() - t0, oracle_threads()


def cpu_baseline(args):
    tokens = args.cpu_tokens
    secs, cores = _oracle_prefill_sample(tokens)
    return {"value": round(tokens / secs, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"fp64 token-by-token oracle on the first {tokens} of the 8192 prefill tokens, all 32 heads "
                      f"(OpenMP over heads; {secs:.2f} s wall)"}


def cpu_baseline_long(args):
    """The oracle on the 65,536-token prefix of the long-context workload (H = 16)."""
    import dataclasses

    from gated_delta_rule_08_gb300 import inputs
    from oracle import oracle_kda_prefill, oracle_threads

    tokens = args.cpu_tokens_long
    P = inputs.prefill_inputs(dataclasses.replace(inputs.LONG, T=tokens), device="cpu")
    t0 = time.perf_counter()
    oracle_kda_prefill(P["q"], P["k"], P["v"], P["g"], P["beta"])
    secs = time.perf_counter() - t0
    return {"value": round(tokens / secs, 1), "unit": "tokens/s", "cores": oracle_threads(), "kind": "oracle",
            "sample": f"fp64 token-by-token oracle on the first {tokens} tokens of the long-context workload, "
                      f"all 16 heads ({secs:.2f} s wall); a 1,048,576-token call would take about "
                      f"{secs * (1 << 20) / tokens:.0f} s (extrapolated)"}


def run_reference(args, world, rank):
    if rank != 0:
        return None
    tokens = args.cpu_tokens
    times = []
    cores = 1
    for i in range(args.warmup + args.steps):
        s, cores = _oracle_prefill_sample(tokens)
        if i >= args.warmup:
            times.append(s)
    total = sum(times)
    value = tokens * len(times) / total
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total * 1e3 / len(times), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": "prefill B=1 H=32 T=8192 dk=dv=128 (oracle sample: first "
                               f"{tokens} tokens, all heads)"},
        "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"first {tokens} of 8192 tokens, all 32 heads, per step"},
        "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-tokens", type=int, default=8192)
    ap.add_argument("--cpu-tokens-long", type=int, default=65536)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--skip-other-workloads", action="store_true",
                    help="time only the prefill + decode step (no varlen / long-context lines)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    world, rank, local = _dist()
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # one process per GPU: relaunch this command under torch.distributed.run
        port = str(_env_int("MASTER_PORT", 29511))
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={args.gpus}",
               "--master-addr", "127.0.0.1", "--master-port", port, os.path.abspath(__file__)] + \
            (list(argv) if argv is not None else sys.argv[1:])
        return subprocess.call(cmd)
    if world != args.gpus:
        sys.stderr.write(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}; launch one process per GPU\n")
        return 2
    if args.impl == "reference":
        line = run_reference(args, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    line = run_ours(args, world, rank, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
