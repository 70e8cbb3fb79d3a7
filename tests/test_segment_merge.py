"""The algebra behind splitting one sequence's state pass into segments (CPU, fp64, on the
oracle): each token maps the state affinely, so a segment maps S_in to P S_in + b with
  b = the segment's final state from S_in = 0,
  P = the segment's final state from S_in = I with v = 0 (a dk x dk state);
and the sequence's final state is recovered by S_in(p+1) = P_p S_in(p) + b_p, where S_in(1) may
instead be taken directly as segment 0's final state from h0 (segment 0's input is known).
(Kimi K3 report walk-through, section 13.3.1: segments evaluate their transitions independently,
then a merge recovers every segment's initial state.)"""
import numpy as np
import torch

from oracle import oracle_kda_prefill


def _seq(T, H, dk, dv, seed, z_mean):
    gen = torch.Generator().manual_seed(seed)
    n = lambda *s: torch.randn(*s, generator=gen, dtype=torch.float64)
    q = torch.nn.functional.normalize(n(T, H, dk), dim=-1)
    k = torch.nn.functional.normalize(n(T, H, dk), dim=-1)
    v = n(T, H, dv)
    g = -5.0 * torch.sigmoid(n(T, H, dk) + z_mean)
    beta = torch.sigmoid(n(T, H))
    h0 = 0.1 * n(1, H, dk, dv)
    return q, k, v, g, beta, h0


def _final(q, k, v, g, beta, h0):
    return oracle_kda_prefill(q, k, v, g, beta, h0=h0)[1][0]  # [H, dk, dv]


def test_segments_compose_to_the_full_sequence():
    T, H, dk, dv = 96, 2, 6, 5
    q, k, v, g, beta, h0 = _seq(T, H, dk, dv, seed=11, z_mean=-3.0)  # slow decay: S_in matters
    full = _final(q, k, v, g, beta, h0)
    bounds = [0, 30, 61, 96]  # three segments of unequal length
    eye = torch.eye(dk, dtype=torch.float64).expand(1, H, dk, dk).contiguous()
    segs = []
    for p in range(3):
        sl = slice(bounds[p], bounds[p + 1])
        args = tuple(x[sl] for x in (q, k, v, g, beta))
        b = _final(*args, torch.zeros(1, H, dk, dv, dtype=torch.float64))
        P = _final(args[0], args[1], torch.zeros(args[2].shape[0], H, dk, dtype=torch.float64), args[3], args[4], eye)
        segs.append((P, b, args))
    # S_in(1): segment 0 run from h0, or P_0 h0 + b_0 -- the same state
    s_direct = _final(*segs[0][2], h0)
    s_merged = np.einsum("hij,hjk->hik", segs[0][0], h0[0].numpy()) + segs[0][1]
    assert np.abs(s_direct - s_merged).max() < 1e-12
    s = s_direct
    for p in (1, 2):
        P, b, _ = segs[p]
        s = np.einsum("hij,hjk->hik", P, s) + b
    assert np.abs(s - full).max() < 1e-12 * max(1.0, np.abs(full).max())


def test_a_later_segment_rerun_from_its_merged_input_gives_the_same_outputs():
    T, H, dk, dv = 80, 1, 4, 3
    q, k, v, g, beta, h0 = _seq(T, H, dk, dv, seed=12, z_mean=-3.0)
    out_full, _ = oracle_kda_prefill(q, k, v, g, beta, h0=h0)
    cut = 37
    s_in = torch.from_numpy(_final(*(x[:cut] for x in (q, k, v, g, beta)), h0))[None]
    out_tail, _ = oracle_kda_prefill(*(x[cut:] for x in (q, k, v, g, beta)), h0=s_in)
    assert np.abs(out_tail - out_full[cut:]).max() < 1e-12
