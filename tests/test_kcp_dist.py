"""The exchange step of context parallelism across devices (KCP), on CPU: two gloo ranks.

Each rank holds a consecutive range of one sequence.  Here each rank computes its range's map
(P, b) with the fp64 oracle (P: final state from S_in = I with v = 0; b: final state from 0), the
ranks exchange the maps with gated_delta_rule_08_gb300.kcp.exchange_segment_maps (the same call the
GPU path makes, here over gloo), and each rank folds the maps of the ranges before its own.  The
folded initial state of rank 1 and the fold of both maps must equal the oracle's state at the range
boundary and at the end of the sequence."""
import os
import socket
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

T, H, D, CUT = 96, 2, 8, 40


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs():
    g = torch.Generator().manual_seed(801)
    q = torch.nn.functional.normalize(torch.randn(T, H, D, generator=g, dtype=torch.float64), dim=-1)
    k = torch.nn.functional.normalize(torch.randn(T, H, D, generator=g, dtype=torch.float64), dim=-1)
    v = torch.randn(T, H, D, generator=g, dtype=torch.float64)
    beta = torch.sigmoid(torch.randn(T, H, generator=g, dtype=torch.float64))
    dec = -5.0 * torch.sigmoid(torch.randn(T, H, D, generator=g, dtype=torch.float64) - 4.0)
    h0 = 0.1 * torch.randn(1, H, D, D, generator=g, dtype=torch.float64)
    return q, k, v, dec, beta, h0


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    from gated_delta_rule_08_gb300.kcp import exchange_segment_maps
    from oracle import oracle_kda_prefill

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q, k, v, dec, beta, h0 = _inputs()
        sl = slice(0, CUT) if rank == 0 else slice(CUT, T)
        x = [t[sl].contiguous() for t in (q, k, v, dec, beta)]
        _, b = oracle_kda_prefill(x[0], x[1], x[2], x[3], x[4])
        eye = torch.eye(D, dtype=torch.float64).expand(1, H, D, D).contiguous()
        _, P = oracle_kda_prefill(x[0], x[1], torch.zeros_like(x[1]), x[3], x[4], h0=eye)
        Ps, bs = exchange_segment_maps(torch.from_numpy(np.ascontiguousarray(P[0])),
                                       torch.from_numpy(np.ascontiguousarray(b[0])))
        S = h0[0].numpy()
        for i in range(rank):  # fold the ranges before this rank's
            S = np.einsum("hij,hjk->hik", Ps[i].numpy(), S) + bs[i].numpy()
        S_all = h0[0].numpy()
        for i in range(world):
            S_all = np.einsum("hij,hjk->hik", Ps[i].numpy(), S_all) + bs[i].numpy()
        results[rank] = (tuple(Ps.shape), S, S_all)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_exchange_and_fold_the_segment_maps():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=180)
        codes = [p.exitcode for p in procs]
        for p in procs:
            if p.is_alive():
                p.kill()
        assert codes == [0, 0], codes
        got = dict(results)
    from oracle import oracle_kda_prefill

    q, k, v, dec, beta, h0 = _inputs()
    _, at_cut = oracle_kda_prefill(q[:CUT], k[:CUT], v[:CUT], dec[:CUT], beta[:CUT], h0=h0)
    _, at_end = oracle_kda_prefill(q, k, v, dec, beta, h0=h0)
    assert got[0][0] == got[1][0] == (world, H, D, D)
    np.testing.assert_allclose(got[0][1], h0[0].numpy(), rtol=0, atol=0)  # rank 0 starts from h0
    np.testing.assert_allclose(got[1][1], at_cut[0], rtol=1e-12, atol=1e-12)
    for r in range(world):
        np.testing.assert_allclose(got[r][2], at_end[0], rtol=1e-12, atol=1e-12)
