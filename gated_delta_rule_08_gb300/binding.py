"""Thin Python binding of libkda (ctypes): argument marshalling only.

Every function here checks shapes/dtypes/devices of torch tensors, passes their
device pointers and the current CUDA stream to the C-ABI entry point of the same
name (include/kda.h), and raises on a non-OK status.  No arithmetic of the method
happens in Python.  There is no fallback: without a built libkda.so or a CUDA
device the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkda.so")

KDA_DTYPE_BF16 = 0
KDA_DTYPE_FP32 = 1
STATUS = {0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED", 3: "KDA_ERR_CUDA",
          4: "KDA_ERR_DEVICE", 5: "KDA_ERR_WORKSPACE"}
DEVERR_BAD_SLOT = 0x1
DEVERR_BAD_SEQLENS = 0x2
DEVERR_WAIT_TIMEOUT = 0x4
DEVERR_BAD_COUNT = 0x8
DEVERR_NONFINITE = 0x10
DEVERR_PRECONDITION = 0x20

# Exported symbols, as declared in include/kda.h.
EXPORTS = ("kda_chunk_fwd_workspace_size", "kda_chunk_fwd", "kda_decode_step", "kda_decode_multi",
           "kda_chunk_fwd_checkpoints", "kda_chunk_bwd", "kda_chunk_bwd_workspace_size", "kda_get_device_error",
           "kda_status_string", "kda_trace_enable", "kda_trace_collect", "kda_chunk_fwd_noalloc",
           "kda_noalloc_scratch_bytes", "kda_chunk_fwd_segment_map", "kda_state_compose")


class KdaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")
        self.status = status


class _Epilogue(ctypes.Structure):
    _fields_ = [("gate_logits", ctypes.c_void_p), ("norm_weight", ctypes.c_void_p), ("eps", ctypes.c_float)]


_lock = threading.Lock()
_lib = None


def load_library(path: Optional[str] = None):
    """Load libkda.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libkda.so not built ({p}); run __graft_entry__.build()")
        lib = ctypes.CDLL(p)
        P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
        lib.kda_chunk_fwd_workspace_size.argtypes = [I, I64, I, I, I, I, I]
        lib.kda_chunk_fwd_workspace_size.restype = SZ
        lib.kda_chunk_fwd.argtypes = [P, P, P, P, P, P, P, P, P, I, I64, I, I, I, I, I, I, P, P, SZ, P]
        lib.kda_chunk_fwd.restype = I
        lib.kda_decode_step.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, P, P]
        lib.kda_decode_step.restype = I
        lib.kda_decode_multi.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, P, P]
        lib.kda_decode_multi.restype = I
        lib.kda_chunk_fwd_checkpoints.argtypes = [P, P, P, P, P, P, P, P, P, P, I64, I, I64, I, I, I, I, I, I, P, P,
                                                  SZ, P]
        lib.kda_chunk_fwd_checkpoints.restype = I
        lib.kda_chunk_bwd_workspace_size.argtypes = [I, I64, I, I, I]
        lib.kda_chunk_bwd_workspace_size.restype = SZ
        lib.kda_chunk_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, I, I64, I, I, I, I, P, SZ, P]
        lib.kda_chunk_bwd.restype = I
        lib.kda_get_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
        lib.kda_get_device_error.restype = I
        lib.kda_chunk_fwd_noalloc.argtypes = [P, P, P, P, P, P, P, P, P, I, I64, I, I, I, I, I, I, P, P]
        lib.kda_chunk_fwd_noalloc.restype = I
        lib.kda_chunk_fwd_segment_map.argtypes = [P, P, P, P, P, P, I64, I, I, I, I, I, P, SZ, P]
        lib.kda_chunk_fwd_segment_map.restype = I
        lib.kda_state_compose.argtypes = [P, P, P, P, I, I, I, I, P]
        lib.kda_state_compose.restype = I
        lib.kda_noalloc_scratch_bytes.argtypes = []
        lib.kda_noalloc_scratch_bytes.restype = SZ
        lib.kda_trace_enable.argtypes = [I]
        lib.kda_trace_enable.restype = I
        lib.kda_trace_collect.argtypes = [I, ctypes.c_char_p, ctypes.POINTER(I), ctypes.POINTER(ctypes.c_double),
                                          ctypes.POINTER(I)]
        lib.kda_trace_collect.restype = I
        lib.kda_status_string.argtypes = [I]
        lib.kda_status_string.restype = ctypes.c_char_p
        if path is None:
            _lib = lib
        return lib


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_DTYPE_BF16
    if t.dtype == torch.float32:
        return KDA_DTYPE_FP32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(t: Optional[torch.Tensor], name: str, dtype=None, shape=None, device=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def kda_chunk_fwd_workspace_size(B: int, T: int, H: int, dk: int, dv: int, C: int = 64,
                                 dtype: torch.dtype = torch.bfloat16) -> int:
    code = KDA_DTYPE_BF16 if dtype == torch.bfloat16 else KDA_DTYPE_FP32
    return int(load_library().kda_chunk_fwd_workspace_size(B, T, H, dk, dv, C, code))


def kda_chunk_fwd(q, k, v, g, beta, h0=None, cu_seqlens=None, out=None, hT=None, *, B: Optional[int] = None,
                  C: int = 64, gate=None, norm_weight=None, eps: float = 1e-6, workspace=None,
                  output_final_state: bool = True, out_dtype: Optional[torch.dtype] = None, _ckpt=None):
    """Chunked KDA prefill.  q, k: [T_tot, H, dk]; v: [T_tot, H, dv]; g: [T_tot, H, dk] fp32;
    beta: [T_tot, H] fp32; h0: [B, H, dk, dv] fp32 or None; cu_seqlens: int32 [B+1] on the device
    or None (then B sequences of T_tot/B tokens).  gate/norm_weight enable the fused epilogue.
    out_dtype: element type of out (default: the dtype of q; bf16 or fp32).
    Returns (out [T_tot, H, dv], hT [B, H, dk, dv] or None)."""
    lib = load_library()
    dev = q.device
    T_tot, H, dk = q.shape
    dv = v.shape[2]
    dt = q.dtype
    code = _dtype_code(q)
    if cu_seqlens is not None:
        _check(cu_seqlens, "cu_seqlens", torch.int32, device=dev)
        nB = cu_seqlens.numel() - 1
        if B is not None and B != nB:
            raise ValueError("B does not match cu_seqlens")
        B = nB
        T_arg = T_tot
    else:
        B = 1 if B is None else B
        if T_tot % B:
            raise ValueError("without cu_seqlens, T_tot must be a multiple of B")
        T_arg = T_tot // B
    _check(q, "q", dt, (T_tot, H, dk), dev)
    _check(k, "k", dt, (T_tot, H, dk), dev)
    _check(v, "v", dt, (T_tot, H, dv), dev)
    _check(g, "g", torch.float32, (T_tot, H, dk), dev)
    _check(beta, "beta", torch.float32, (T_tot, H), dev)
    _check(h0, "h0", torch.float32, (B, H, dk, dv), dev)
    _check(gate, "gate", dt, (T_tot, H, dv), dev)
    _check(norm_weight, "norm_weight", torch.float32, (dv,), dev)
    odt = out.dtype if out is not None else (out_dtype or dt)
    if out is None:
        out = torch.empty(T_tot, H, dv, device=dev, dtype=odt)
    _check(out, "out", odt, (T_tot, H, dv), dev)
    ocode = _dtype_code(out)
    if hT is None and output_final_state:
        hT = torch.empty(B, H, dk, dv, device=dev, dtype=torch.float32)
    _check(hT, "hT", torch.float32, (B, H, dk, dv), dev)
    need = int(lib.kda_chunk_fwd_workspace_size(B, T_arg, H, dk, dv, C, code))
    if need == 0:
        raise KdaError("kda_chunk_fwd_workspace_size", 2)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, device=dev, dtype=torch.uint8)
    _check(workspace, "workspace", torch.uint8, None, dev)
    epi = None
    if gate is not None:
        epi = _Epilogue(gate.data_ptr(), norm_weight.data_ptr() if norm_weight is not None else None, float(eps))
    if _ckpt is None:
        st = lib.kda_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(cu_seqlens),
                               _ptr(out), _ptr(hT), B, T_arg, H, dk, dv, C, code, ocode,
                               ctypes.byref(epi) if epi is not None else None, _ptr(workspace),
                               workspace.numel(), _stream(dev))
        if st != 0:
            raise KdaError("kda_chunk_fwd", st)
        return out, hT
    states, ckpt_chunks = _ckpt
    span = 64 * ckpt_chunks
    if cu_seqlens is not None:
        lens = (cu_seqlens[1:] - cu_seqlens[:-1]).to("cpu").to(torch.int64)
        n_ckpt = int((lens // span).sum())
    else:
        n_ckpt = B * (T_arg // span)
    if states is None:
        states = torch.empty(n_ckpt, H, dk, dv, device=dev, dtype=torch.float32)
    _check(states, "states", torch.float32, (n_ckpt, H, dk, dv), dev)
    st = lib.kda_chunk_fwd_checkpoints(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(cu_seqlens),
                                       _ptr(out), _ptr(hT), ctypes.c_void_p(states.data_ptr()), int(ckpt_chunks), B,
                                       T_arg, H, dk, dv, C, code, ocode,
                                       ctypes.byref(epi) if epi is not None else None, _ptr(workspace),
                                       workspace.numel(), _stream(dev))
    if st != 0:
        raise KdaError("kda_chunk_fwd_checkpoints", st)
    return out, hT, states


def kda_chunk_fwd_checkpoints(q, k, v, g, beta, h0=None, cu_seqlens=None, out=None, hT=None, *, ckpt_chunks: int,
                              states=None, **kw):
    """kda_chunk_fwd that also returns the fp32 state of every sequence after each 64 * ckpt_chunks
    of its tokens: states [n_ckpt, H, dk, dv], sequences in order, each in token order.
    Returns (out, hT, states)."""
    if ckpt_chunks < 1:
        raise ValueError("ckpt_chunks must be >= 1")
    return kda_chunk_fwd(q, k, v, g, beta, h0, cu_seqlens, out, hT, _ckpt=(states, int(ckpt_chunks)), **kw)


def kda_decode_step(q, k, v, g, beta, state_pool, slot_idx, out=None, *, gate=None, norm_weight=None,
                    eps: float = 1e-6, out_dtype: Optional[torch.dtype] = None):
    """One decode step.  q, k: [N, H, dk]; v: [N, H, dv]; g: [N, H, dk] fp32; beta: [N, H] fp32;
    state_pool: [num_slots, H, dk, dv] fp32 (updated in place); slot_idx: int32 [N].
    Returns out [N, H, dv]."""
    lib = load_library()
    dev = q.device
    N, H, dk = q.shape
    dv = v.shape[2]
    dt = q.dtype
    code = _dtype_code(q)
    num_slots = state_pool.shape[0]
    _check(q, "q", dt, (N, H, dk), dev)
    _check(k, "k", dt, (N, H, dk), dev)
    _check(v, "v", dt, (N, H, dv), dev)
    _check(g, "g", torch.float32, (N, H, dk), dev)
    _check(beta, "beta", torch.float32, (N, H), dev)
    _check(state_pool, "state_pool", torch.float32, (num_slots, H, dk, dv), dev)
    _check(slot_idx, "slot_idx", torch.int32, (N,), dev)
    _check(gate, "gate", dt, (N, H, dv), dev)
    _check(norm_weight, "norm_weight", torch.float32, (dv,), dev)
    odt = out.dtype if out is not None else (out_dtype or dt)
    if out is None:
        out = torch.empty(N, H, dv, device=dev, dtype=odt)
    _check(out, "out", odt, (N, H, dv), dev)
    ocode = _dtype_code(out)
    epi = None
    if gate is not None:
        epi = _Epilogue(gate.data_ptr(), norm_weight.data_ptr() if norm_weight is not None else None, float(eps))
    st = lib.kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_pool), _ptr(slot_idx),
                             _ptr(out), N, H, dk, dv, num_slots, code, ocode,
                             ctypes.byref(epi) if epi is not None else None, _stream(dev))
    if st != 0:
        raise KdaError("kda_decode_step", st)
    return out


def kda_chunk_bwd_workspace_size(B: int, T: int, H: int, dk: int, dv: int) -> int:
    return int(load_library().kda_chunk_bwd_workspace_size(B, T, H, dk, dv))


def kda_chunk_bwd(q, k, v, g, beta, dout, h0=None, cu_seqlens=None, dhT=None, *, B: Optional[int] = None,
                  need_dh0: bool = True, workspace=None):
    """Gradients of sum <dout, out> + <dhT, hT> for the prefill recurrence (no epilogue).
    Returns (dq, dk, dv, dg, dbeta, dh0 or None), all fp32."""
    lib = load_library()
    dev = q.device
    T_tot, H, dk = q.shape
    dv = v.shape[2]
    dt = q.dtype
    code = _dtype_code(q)
    if cu_seqlens is not None:
        _check(cu_seqlens, "cu_seqlens", torch.int32, device=dev)
        B = cu_seqlens.numel() - 1
        T_arg = T_tot
    else:
        B = 1 if B is None else B
        if T_tot % B:
            raise ValueError("without cu_seqlens, T_tot must be a multiple of B")
        T_arg = T_tot // B
    for name, t, d, shape in (("q", q, dt, (T_tot, H, dk)), ("k", k, dt, (T_tot, H, dk)), ("v", v, dt, (T_tot, H, dv)),
                              ("g", g, torch.float32, (T_tot, H, dk)), ("beta", beta, torch.float32, (T_tot, H)),
                              ("dout", dout, dt, (T_tot, H, dv))):
        _check(t, name, d, shape, dev)
    _check(h0, "h0", torch.float32, (B, H, dk, dv), dev)
    _check(dhT, "dhT", torch.float32, (B, H, dk, dv), dev)
    f32 = dict(device=dev, dtype=torch.float32)
    dq, dk_, dg = (torch.empty(T_tot, H, dk, **f32) for _ in range(3))
    dv_ = torch.empty(T_tot, H, dv, **f32)
    dbeta = torch.empty(T_tot, H, **f32)
    dh0 = torch.empty(B, H, dk, dv, **f32) if need_dh0 else None
    need = int(lib.kda_chunk_bwd_workspace_size(B, T_arg, H, dk, dv))
    if need == 0:
        raise KdaError("kda_chunk_bwd_workspace_size", 2)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, device=dev, dtype=torch.uint8)
    st = lib.kda_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(cu_seqlens), _ptr(dout),
                           _ptr(dhT), _ptr(dq), _ptr(dk_), _ptr(dv_), _ptr(dg), _ptr(dbeta), _ptr(dh0), B, T_arg, H, dk,
                           dv, code, _ptr(workspace), workspace.numel(), _stream(dev))
    if st != 0:
        raise KdaError("kda_chunk_bwd", st)
    return dq, dk_, dv_, dg, dbeta, dh0


def kda_decode_multi(q, k, v, g, beta, state_pool, slot_idx, ntok_per_req=None, out=None, *, commit: bool,
                     gate=None, norm_weight=None, eps: float = 1e-6, out_dtype: Optional[torch.dtype] = None):
    """Several tokens per request (speculative-decode verify / accept).  q, k: [N, n_tok, H, dk];
    v: [N, n_tok, H, dv]; g: [N, n_tok, H, dk] fp32; beta: [N, n_tok, H] fp32; state_pool:
    [num_slots, H, dk, dv] fp32; slot_idx: int32 [N]; ntok_per_req: int32 [N] (tokens applied per
    request) or None (all n_tok).  commit=False leaves the pool untouched (verify); commit=True
    writes each request's state after its applied tokens back (accept).
    Returns out [N, n_tok, H, dv]; rows of tokens not applied are left as they were in `out`."""
    lib = load_library()
    dev = q.device
    N, n_tok, H, dk = q.shape
    dv = v.shape[3]
    dt = q.dtype
    code = _dtype_code(q)
    num_slots = state_pool.shape[0]
    _check(q, "q", dt, (N, n_tok, H, dk), dev)
    _check(k, "k", dt, (N, n_tok, H, dk), dev)
    _check(v, "v", dt, (N, n_tok, H, dv), dev)
    _check(g, "g", torch.float32, (N, n_tok, H, dk), dev)
    _check(beta, "beta", torch.float32, (N, n_tok, H), dev)
    _check(state_pool, "state_pool", torch.float32, (num_slots, H, dk, dv), dev)
    _check(slot_idx, "slot_idx", torch.int32, (N,), dev)
    _check(ntok_per_req, "ntok_per_req", torch.int32, (N,), dev)
    _check(gate, "gate", dt, (N, n_tok, H, dv), dev)
    _check(norm_weight, "norm_weight", torch.float32, (dv,), dev)
    odt = out.dtype if out is not None else (out_dtype or dt)
    if out is None:
        out = torch.empty(N, n_tok, H, dv, device=dev, dtype=odt)
    _check(out, "out", odt, (N, n_tok, H, dv), dev)
    ocode = _dtype_code(out)
    epi = None
    if gate is not None:
        epi = _Epilogue(gate.data_ptr(), norm_weight.data_ptr() if norm_weight is not None else None, float(eps))
    st = lib.kda_decode_multi(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state_pool), _ptr(slot_idx),
                              _ptr(ntok_per_req), _ptr(out), N, n_tok, H, dk, dv, num_slots, 1 if commit else 0,
                              code, ocode, ctypes.byref(epi) if epi is not None else None, _stream(dev))
    if st != 0:
        raise KdaError("kda_decode_multi", st)
    return out


def kda_get_device_error(device=None) -> int:
    """Synchronise the current stream and read + clear the device error word."""
    lib = load_library()
    flags = ctypes.c_uint32(0)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    st = lib.kda_get_device_error(_stream(dev), ctypes.byref(flags))
    if st != 0:
        raise KdaError("kda_get_device_error", st)
    return int(flags.value)


def kda_status_string(status: int) -> str:
    return load_library().kda_status_string(status).decode()


def kda_trace_enable(enable: bool = True) -> None:
    """Bracket every internal kernel launch with CUDA events (profiling aid)."""
    st = load_library().kda_trace_enable(1 if enable else 0)
    if st != 0:
        raise KdaError("kda_trace_enable", st)


def kda_trace_collect(max_entries: int = 32) -> dict:
    """{kernel name: (launches, total ms)} since the previous collect (synchronises)."""
    lib = load_library()
    names = ctypes.create_string_buffer(64 * max_entries)
    launches = (ctypes.c_int * max_entries)()
    total = (ctypes.c_double * max_entries)()
    n = ctypes.c_int(0)
    st = lib.kda_trace_collect(max_entries, names, launches, total, ctypes.byref(n))
    if st != 0:
        raise KdaError("kda_trace_collect", st)
    raw = names.raw
    return {raw[64 * i:64 * i + 64].split(b"\0", 1)[0].decode(): (int(launches[i]), float(total[i]))
            for i in range(n.value)}


def kda_chunk_fwd_noalloc(q, k, v, g, beta, h0=None, cu_seqlens=None, out=None, hT=None, *,
                          B: Optional[int] = None, C: int = 64, gate=None, norm_weight=None, eps: float = 1e-6,
                          out_dtype: Optional[torch.dtype] = None):
    """kda_chunk_fwd without a caller workspace: the library's fixed device scratch is used
    instead, so the C call itself allocates nothing (out/hT are allocated here only when the
    caller passes None).  For callers that cannot allocate at call time; problems needing more
    than kda_noalloc_scratch_bytes() of scratch are rejected.  Same arguments and results as
    kda_chunk_fwd."""
    lib = load_library()
    dev = q.device
    T_tot, H, dk = q.shape
    dv = v.shape[2]
    code = _dtype_code(q)
    if cu_seqlens is not None:
        _check(cu_seqlens, "cu_seqlens", torch.int32, device=dev)
        B = cu_seqlens.numel() - 1
        T_arg = T_tot
    else:
        B = 1 if B is None else B
        if T_tot % B:
            raise ValueError("without cu_seqlens, T_tot must be a multiple of B")
        T_arg = T_tot // B
    for t, name, dt_, shp in ((q, "q", q.dtype, (T_tot, H, dk)), (k, "k", q.dtype, (T_tot, H, dk)),
                              (v, "v", q.dtype, (T_tot, H, dv)), (g, "g", torch.float32, (T_tot, H, dk)),
                              (beta, "beta", torch.float32, (T_tot, H)), (h0, "h0", torch.float32, (B, H, dk, dv)),
                              (gate, "gate", q.dtype, (T_tot, H, dv)),
                              (norm_weight, "norm_weight", torch.float32, (dv,))):
        _check(t, name, dt_, shp, dev)
    odt = out.dtype if out is not None else (out_dtype or q.dtype)
    if out is None:
        out = torch.empty(T_tot, H, dv, device=dev, dtype=odt)
    _check(out, "out", odt, (T_tot, H, dv), dev)
    if hT is None:
        hT = torch.empty(B, H, dk, dv, device=dev, dtype=torch.float32)
    _check(hT, "hT", torch.float32, (B, H, dk, dv), dev)
    epi = None
    if gate is not None:
        epi = _Epilogue(gate.data_ptr(), norm_weight.data_ptr() if norm_weight is not None else None, float(eps))
    st = lib.kda_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(cu_seqlens),
                                   _ptr(out), _ptr(hT), B, T_arg, H, dk, dv, C, code, _dtype_code(out),
                                   ctypes.byref(epi) if epi is not None else None, _stream(dev))
    if st != 0:
        raise KdaError("kda_chunk_fwd_noalloc", st)
    return out, hT


def kda_chunk_fwd_segment_map(k, v, g, beta, *, C: int = 64, P=None, b=None, workspace=None):
    """The affine map of one token range's state pass (context parallelism across devices):
    S_out = P S_in + b.  k: [T, H, dk]; v: [T, H, dv]; g: [T, H, dk] fp32; beta: [T, H] fp32.
    Returns (P [H, dk, dk], b [H, dk, dv]), both fp32."""
    lib = load_library()
    dev = k.device
    T, H, dk = k.shape
    dv = v.shape[2]
    dt = k.dtype
    code = _dtype_code(k)
    _check(k, "k", dt, (T, H, dk), dev)
    _check(v, "v", dt, (T, H, dv), dev)
    _check(g, "g", torch.float32, (T, H, dk), dev)
    _check(beta, "beta", torch.float32, (T, H), dev)
    if P is None:
        P = torch.empty(H, dk, dk, device=dev, dtype=torch.float32)
    if b is None:
        b = torch.empty(H, dk, dv, device=dev, dtype=torch.float32)
    _check(P, "P", torch.float32, (H, dk, dk), dev)
    _check(b, "b", torch.float32, (H, dk, dv), dev)
    need = int(lib.kda_chunk_fwd_workspace_size(1, T, H, dk, dv, C, code))
    if need == 0:
        raise KdaError("kda_chunk_fwd_workspace_size", 2)
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, device=dev, dtype=torch.uint8)
    st = lib.kda_chunk_fwd_segment_map(_ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(P), _ptr(b), T, H, dk, dv, C,
                                       code, _ptr(workspace), workspace.numel(), _stream(dev))
    if st != 0:
        raise KdaError("kda_chunk_fwd_segment_map", st)
    return P, b


def kda_state_compose(P, b, S0=None, out=None):
    """Fold n range maps into an initial state: S = P[n-1](...(P[0] S0 + b[0])...) + b[n-1].
    P: [n, H, dk, dk] fp32; b: [n, H, dk, dv] fp32; S0: [H, dk, dv] fp32 or None (zero).
    Returns S [H, dk, dv] fp32 (`out` if given; it may be S0)."""
    lib = load_library()
    n, H, dk, _ = P.shape
    dv = b.shape[3]
    dev = P.device
    _check(P, "P", torch.float32, (n, H, dk, dk), dev)
    _check(b, "b", torch.float32, (n, H, dk, dv), dev)
    _check(S0, "S0", torch.float32, (H, dk, dv), dev)
    if out is None:
        out = torch.empty(H, dk, dv, device=dev, dtype=torch.float32)
    _check(out, "out", torch.float32, (H, dk, dv), dev)
    st = lib.kda_state_compose(_ptr(P), _ptr(b), _ptr(S0), _ptr(out), n, H, dk, dv, _stream(dev))
    if st != 0:
        raise KdaError("kda_state_compose", st)
    return out
