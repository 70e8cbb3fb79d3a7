"""kda_chunk_fwd_noalloc: the prefill for callers that cannot allocate device memory.

Some callers (code under an allocator that owns all device memory, hosts whose
execution path forbids cudaMalloc) cannot hand kda_chunk_fwd a workspace; the
no-allocation entry point uses the library's fixed device scratch instead.  This
test calls it through the C-ABI (ctypes, raw device pointers, no workspace
argument) twice in a row and checks each result against kda_chunk_fwd on the same
inputs, with the parity tolerance the other tests use.  The file is named so that
pytest collects it last.
"""
import ctypes

import pytest
import torch

from gated_delta_rule_08_gb300 import binding, inputs
from gpu_util import TOL, parity_err, rel_err

pytestmark = pytest.mark.gpu


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc_call(lib, inp, out, hT):
    T_tot, H, dk = inp["q"].shape
    dv = inp["v"].shape[2]
    B = len(inp["lengths"])
    epi = binding._Epilogue(inp["gate"].data_ptr(), inp["norm_weight"].data_ptr(), 1e-6)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.kda_chunk_fwd_noalloc(_p(inp["q"]), _p(inp["k"]), _p(inp["v"]), _p(inp["g"]), _p(inp["beta"]),
                                     _p(inp["h0"]), _p(inp["cu_seqlens"]), _p(out), _p(hT), B, T_tot, H, dk, dv,
                                     64, binding.KDA_DTYPE_BF16, binding.KDA_DTYPE_FP32, ctypes.byref(epi), stream)


def test_noalloc_matches_workspace_entry_point_twice():
    lib = binding.load_library()
    assert lib.kda_noalloc_scratch_bytes() == 64 << 20
    runs = []
    for seed in (501, 502):  # two calls in a row, different inputs, same scratch
        cfg = inputs.PrefillConfig("noalloc", H=4, dk=128, dv=128, dtype="bf16", lengths=(70, 1, 130), B=3,
                                   h0_std=0.1, epilogue=True, seed=seed)
        inp = inputs.prefill_inputs(cfg, device="cuda")
        T_tot, H, dv = inp["T_tot"], cfg.H, cfg.dv
        out = torch.empty(T_tot, H, dv, device="cuda", dtype=torch.float32)
        hT = torch.empty(3, H, cfg.dk, dv, device="cuda", dtype=torch.float32)
        assert _noalloc_call(lib, inp, out, hT) == 0
        ref_out, ref_hT = binding.kda_chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], h0=inp["h0"],
                                                cu_seqlens=inp["cu_seqlens"], gate=inp["gate"],
                                                norm_weight=inp["norm_weight"], out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert binding.kda_get_device_error() == 0
        tol = TOL[torch.bfloat16]
        assert parity_err(out, ref_out.double().cpu().numpy()) <= tol
        assert rel_err(hT, ref_hT.double().cpu().numpy()) <= tol
        runs.append(torch.equal(out, ref_out) and torch.equal(hT, ref_hT))
    assert all(runs)  # same kernels on the same inputs: identical results


def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = binding.load_library()
    # H=32, T=1M needs far more than 64 MiB of scratch: refused before any launch
    dummy = ctypes.c_void_p(0x1000)
    st = lib.kda_chunk_fwd_noalloc(dummy, dummy, dummy, dummy, dummy, None, None, ctypes.c_void_p(0x2000), None,
                                   1, 1 << 20, 32, 128, 128, 64, binding.KDA_DTYPE_BF16, binding.KDA_DTYPE_BF16,
                                   None, None)
    assert st == 5  # KDA_ERR_WORKSPACE
