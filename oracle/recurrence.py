"""ctypes wrapper around the fp64 token-by-token KDA oracle (``kda_oracle.c``).

TEST INFRASTRUCTURE: see the package docstring for who may call this.

The recurrence (Kimi K3 report walk-through, section 2.2 Eq. 1, section 2.3,
section 2.4 Eq. 3, section 3.3 Eq. 6):
    S_t = (I - beta_t k_t k_t^T) Diag(exp g_t) S_{t-1} + beta_t k_t v_t^T
    o_t = S_t^T q_t            [optionally RMSNorm over dv, times sigmoid(gate)]
All arithmetic is fp64 on the host.  Inputs of any dtype are upcast to fp64
before the call (bf16 values are exact in fp64).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None


def build_oracle(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` with gcc (-O2, OpenMP, fp64, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build_oracle()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            lib.oracle_kda_prefill.argtypes = [P, P, P, P, P, P, P, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, P, P, ctypes.c_double,
                                               P, P, ctypes.c_int]
            lib.oracle_kda_prefill.restype = ctypes.c_int
            lib.oracle_kda_decode.argtypes = [P, P, P, P, P, P, P, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int, P, P,
                                              ctypes.c_double, P, ctypes.c_int]
            lib.oracle_kda_decode.restype = ctypes.c_int
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x):
    """Contiguous fp64 numpy copy of a numpy array or a (CPU/GPU) torch tensor."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def oracle_threads() -> int:
    return int(_load().oracle_max_threads())


def oracle_kda_prefill(q, k, v, g, beta, h0=None, cu_seqlens=None, gate=None, norm_weight=None,
                       eps: float = 1e-6, num_threads: int = 0):
    """fp64 prefill over a packed batch.

    q, k, g: [T_tot, H, dk]; v: [T_tot, H, dv]; beta: [T_tot, H];
    h0: [B, H, dk, dv] or None; cu_seqlens: [B+1] (None = one sequence of T_tot);
    gate: [T_tot, H, dv] or None (None = no epilogue); norm_weight: [dv] or None.
    Returns (out [T_tot, H, dv], hT [B, H, dk, dv]) as fp64 numpy arrays.
    """
    q, k, v, g, beta = (_f64(t) for t in (q, k, v, g, beta))
    T_tot, H, dk = q.shape
    dv = v.shape[2]
    if cu_seqlens is None:
        cu = np.array([0, T_tot], dtype=np.int64)
    else:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().to("cpu").numpy()
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    B = len(cu) - 1
    h0 = _f64(h0)
    gate = _f64(gate)
    w = _f64(norm_weight)
    out = np.zeros((T_tot, H, dv), dtype=np.float64)
    hT = np.zeros((B, H, dk, dv), dtype=np.float64)
    rc = _load().oracle_kda_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(cu),
                                    B, H, dk, dv, _ptr(gate), _ptr(w), float(eps), _ptr(out), _ptr(hT),
                                    int(num_threads))
    if rc != 0:
        raise ValueError("oracle_kda_prefill: bad arguments")
    return out, hT


def oracle_kda_decode(q, k, v, g, beta, state_pool, slot_idx, gate=None, norm_weight=None,
                      eps: float = 1e-6, num_threads: int = 0):
    """fp64 single-token decode step on a state pool.

    q, k, g: [N, H, dk]; v: [N, H, dv]; beta: [N, H]; state_pool: [num_slots, H, dk, dv]
    (a fp64 copy is updated and returned); slot_idx: [N].
    Returns (out [N, H, dv], new_pool, n_skipped_rows).
    """
    q, k, v, g, beta = (_f64(t) for t in (q, k, v, g, beta))
    N, H, dk = q.shape
    dv = v.shape[2]
    pool = _f64(state_pool).copy()
    if hasattr(slot_idx, "detach"):
        slot_idx = slot_idx.detach().to("cpu").numpy()
    slots = np.ascontiguousarray(np.asarray(slot_idx, dtype=np.int64))
    gate = _f64(gate)
    w = _f64(norm_weight)
    out = np.zeros((N, H, dv), dtype=np.float64)
    rc = _load().oracle_kda_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(pool), _ptr(slots),
                                   N, H, dk, dv, pool.shape[0], _ptr(gate), _ptr(w), float(eps), _ptr(out),
                                   int(num_threads))
    if rc < 0:
        raise ValueError("oracle_kda_decode: bad arguments")
    return out, pool, rc
