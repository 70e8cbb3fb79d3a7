"""The fp64 oracle against what the pages and the mathematics fix (CPU only)."""
import numpy as np
import pytest
import torch

import pins
from oracle import oracle_kda_decode, oracle_kda_prefill
from oracle.chunkwise_bruteforce import chunkwise_prefill


def oracle_prefill(q, k, v, g, beta, h0, cu):
    return oracle_kda_prefill(q, k, v, g, beta, h0=h0, cu_seqlens=cu)


def chunkwise(q, k, v, g, beta, h0, cu, C):
    return chunkwise_prefill(q, k, v, g, beta, h0=h0, cu_seqlens=cu, C=C)


# ---------------------------------------------------------------- the pins
def test_hand_example():
    assert pins.check_hand_example(oracle_prefill) < 1e-12


def test_beta_zero_closed_form():
    assert pins.check_beta_zero(oracle_prefill) < 1e-12


def test_unit_key_beta_one_overwrites():
    assert pins.check_overwrite(oracle_prefill) < 1e-12


def test_delta_rule_is_a_gradient_step():
    assert pins.check_gradient_step(oracle_prefill) < 1e-12


@pytest.mark.parametrize("seed,T,dk,dv", [(4, 24, 5, 3), (7, 48, 8, 8), (9, 33, 3, 6)])
def test_chunkwise_equals_recurrence_for_every_chunk_size(seed, T, dk, dv):
    assert pins.check_chunkwise(oracle_prefill, chunkwise, seed=seed, T=T, dk=dk, dv=dv) < 1e-10


def test_chunkwise_strong_decay_long_chunk():
    """g near the lower bound -5 over a 64-token chunk: cumulative decay exp(-320)
    stays representable in fp64, and the chunkwise form still matches."""
    rng = np.random.default_rng(11)
    T, dk, dv = 64, 4, 3
    q, k, v, g, b, h0 = pins.rand_inputs(rng, T, 1, dk, dv)
    g = np.full_like(g, -4.99)
    out, hT = oracle_prefill(q, k, v, g, b, h0, np.array([0, T]))
    o2, h2 = chunkwise(q, k, v, g, b, h0, np.array([0, T]), 64)
    assert np.abs(out - o2).max() < 1e-10 and np.abs(hT - h2).max() < 1e-10


def test_linearity_in_values_and_initial_state():
    assert pins.check_linearity(oracle_prefill) < 1e-12


def test_value_columns_are_independent():
    assert pins.check_column_split(oracle_prefill) < 1e-13


def test_no_decay_no_write_keeps_state():
    rng = np.random.default_rng(12)
    T, H, dk, dv = 10, 2, 4, 3
    q, k, v, _, _, h0 = pins.rand_inputs(rng, T, H, dk, dv)
    out, hT = oracle_prefill(q, k, v, np.zeros((T, H, dk)), np.zeros((T, H)), h0, np.array([0, T]))
    assert np.array_equal(hT, h0)
    assert np.allclose(out, np.einsum("hij,thi->thj", h0[0], q), rtol=0, atol=1e-13)


# ---------------------------------------------------------------- epilogue
def test_epilogue_matches_torch_rms_norm_and_sigmoid():
    rng = np.random.default_rng(13)
    T, H, dk, dv = 12, 3, 5, 8
    q, k, v, g, b, h0 = pins.rand_inputs(rng, T, H, dk, dv)
    gate = rng.standard_normal((T, H, dv))
    w = 1.0 + 0.1 * rng.standard_normal(dv)
    eps = 1e-6
    raw, hT = oracle_kda_prefill(q, k, v, g, b, h0=h0)
    y, hT2 = oracle_kda_prefill(q, k, v, g, b, h0=h0, gate=gate, norm_weight=w, eps=eps)
    ref = torch.nn.functional.rms_norm(torch.tensor(raw), (dv,), torch.tensor(w), eps) * torch.sigmoid(
        torch.tensor(gate))
    assert np.abs(y - ref.numpy()).max() < 1e-12
    assert np.array_equal(hT, hT2)  # the epilogue never feeds back into the state
    y1, _ = oracle_kda_prefill(q, k, v, g, b, h0=h0, gate=gate, norm_weight=None, eps=eps)
    ref1 = torch.nn.functional.rms_norm(torch.tensor(raw), (dv,), None, eps) * torch.sigmoid(torch.tensor(gate))
    assert np.abs(y1 - ref1.numpy()).max() < 1e-12


# ---------------------------------------------------------------- batching
def test_packed_varlen_equals_separate_runs():
    rng = np.random.default_rng(14)
    lens = [5, 0, 1, 17, 64, 65]
    T = sum(lens)
    H, dk, dv = 2, 4, 3
    q, k, v, g, b, _ = pins.rand_inputs(rng, T, H, dk, dv)
    h0 = rng.standard_normal((len(lens), H, dk, dv))
    cu = np.concatenate([[0], np.cumsum(lens)])
    out, hT = oracle_kda_prefill(q, k, v, g, b, h0=h0, cu_seqlens=cu)
    for i, (a, e) in enumerate(zip(cu[:-1], cu[1:])):
        o_i, h_i = oracle_kda_prefill(q[a:e], k[a:e], v[a:e], g[a:e], b[a:e], h0=h0[i:i + 1])
        assert np.array_equal(out[a:e], o_i)
        assert np.array_equal(hT[i], h_i[0])
    assert np.array_equal(hT[1], h0[1])  # empty sequence: final state is the initial state


def test_decode_steps_equal_prefill():
    rng = np.random.default_rng(15)
    T, H, dk, dv = 9, 2, 4, 3
    q, k, v, g, b, h0 = pins.rand_inputs(rng, T, H, dk, dv)
    out, hT = oracle_kda_prefill(q, k, v, g, b, h0=h0)
    pool = np.zeros((3, H, dk, dv))
    pool[2] = h0[0]
    for t in range(T):
        o, pool, skipped = oracle_kda_decode(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1], b[t:t + 1],
                                             pool, np.array([2]))
        assert skipped == 0
        assert np.array_equal(o[0], out[t])
    assert np.array_equal(pool[2], hT[0])
    assert not pool[:2].any()


def test_decode_bad_slot_is_skipped():
    rng = np.random.default_rng(16)
    N, H, dk, dv = 4, 2, 4, 3
    q, k, v, g, b, _ = pins.rand_inputs(rng, N, H, dk, dv)
    pool = rng.standard_normal((5, H, dk, dv))
    out, new_pool, skipped = oracle_kda_decode(q, k, v, g, b, pool, np.array([1, -1, 5, 3]))
    assert skipped == 2
    assert not out[1].any() and not out[2].any()
    for s in (0, 2, 4):
        assert np.array_equal(new_pool[s], pool[s])
    assert not np.array_equal(new_pool[1], pool[1]) and not np.array_equal(new_pool[3], pool[3])


# ---------------------------------------------------------------- the pins catch planted mistakes
def _mutant(kind):
    """A small recurrence with one planted mistake (CPU, test only)."""

    def step(S, q, k, v, g, beta):
        a = np.exp(-g) if kind == "decay_sign" else np.exp(g)
        dv = S.shape[1]
        if kind == "erase_before_decay":
            S = S - beta * np.outer(k, k @ S)
            S = a[:, None] * S
        else:
            if kind == "decay_columns":
                S = S * np.resize(a, dv)[None, :]
            elif kind != "no_decay":
                S = a[:, None] * S
            if kind == "erase_without_beta":
                S = S - np.outer(k, k @ S)
            elif kind == "erase_sign":
                S = S + beta * np.outer(k, k @ S)
            elif kind != "no_erase":
                S = S - beta * np.outer(k, k @ S)
        if kind == "write_without_beta":
            S = S + np.outer(k, v)
        elif kind == "write_wrong_key_index":
            S = S + beta * np.outer(np.roll(k, 1), v)
        else:
            S = S + beta * np.outer(k, v)
        return S

    def prefill(q, k, v, g, beta, h0, cu):
        T, H, dk = q.shape
        dv = v.shape[2]
        out = np.zeros((T, H, dv))
        hT = np.zeros((1, H, dk, dv))
        for h in range(H):
            S = h0[0, h].copy()
            for t in range(T):
                S_prev = S
                S = step(S, q[t, h], k[t, h], v[t, h], g[t, h], beta[t, h])
                if kind == "read_before_update":
                    out[t, h] = S_prev.T @ q[t, h]
                elif kind == "read_wrong_query_index":
                    out[t, h] = S.T @ np.roll(q[t, h], 1)
                else:
                    out[t, h] = S.T @ q[t, h]
            hT[0, h] = S
        return out, hT

    return prefill


MUTANTS = ["erase_before_decay", "decay_columns", "decay_sign", "no_decay", "erase_without_beta",
           "erase_sign", "no_erase", "write_without_beta", "write_wrong_key_index", "read_before_update",
           "read_wrong_query_index"]


def _run_all(prefill):
    return {
        "hand_example": pins.check_hand_example(prefill),
        "beta_zero": pins.check_beta_zero(prefill),
        "overwrite": pins.check_overwrite(prefill),
        "gradient_step": pins.check_gradient_step(prefill),
        "chunkwise": pins.check_chunkwise(prefill, chunkwise),
        "linearity": pins.check_linearity(prefill),
        "column_split": pins.check_column_split(prefill),
    }


def test_correct_small_recurrence_passes_all_pins():
    errs = _run_all(_mutant("none"))
    assert max(errs.values()) < 1e-10, errs


@pytest.mark.parametrize("kind", MUTANTS)
def test_every_planted_mistake_fails_some_pin(kind):
    errs = _run_all(_mutant(kind))
    failed = [name for name, e in errs.items() if not (e < 1e-8)]
    assert failed, f"mutant {kind} passed every pin: {errs}"
