"""Multi-rank host logic on CPU with gloo, world size 2 (no GPU).

The step's only cross-rank exchange is the 8-byte local sum of squares of
each rank (ZeRO-2/3 global grad-norm clipping).  Two gloo ranks check that
the shard ranges they compute partition the flat buffer, that
gather_sqnorms returns every rank's value in rank order and the same vector
on every rank, that the rank-order total equals the oracle's norm over the
whole buffer, and that a non-finite grad on one rank makes every rank skip.
"""
import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

WORLD = 2


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        import oracle
        import workloads as W
        from fsdp_sharded_mixed_flatparameter_gb300 import gather_sqnorms, zero_shard as zs
        wl = W.small_ragged(n_tensors=200, world_size=WORLD, rank=rank, grad_dtype="f32")
        s, e = zs.zero_shard_range(wl.total, WORLD, rank)
        # every rank's view of the partition
        rng = torch.tensor([s, e], dtype=torch.int64)
        ranges = [torch.empty(2, dtype=torch.int64) for _ in range(WORLD)]
        dist.all_gather(ranges, rng)
        out = {"ranges": [tuple(int(x) for x in r) for r in ranges]}
        for case in ("finite", "nonfinite"):
            g = W.flat_grads(wl, 1, 0, s, e).numpy().copy()
            if case == "nonfinite" and rank == 1:
                g[len(g) // 2] = np.inf
            local = torch.tensor([oracle.sqnorm(g)], dtype=torch.float64)
            gathered = gather_sqnorms(local, None)
            total = 0.0
            for v in gathered.tolist():
                total += v  # rank order, binary64: what zero_grad_sqnorm_combine does
            cr = oracle.clip(total, 0.0, wl.max_norm)
            out[case] = {"gathered": gathered.tolist(), "local": float(local), "norm": cr.norm,
                         "coef": cr.coef, "finite": cr.finite}
        results[rank] = out
    finally:
        dist.destroy_process_group()


def test_two_ranks_exchange_and_skip_policy():
    import oracle
    import workloads as W
    from fsdp_sharded_mixed_flatparameter_gb300 import build
    build.build()  # once, before the ranks start (they only load it)
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    mp.start_processes(_rank_main, args=(_free_port(), results), nprocs=WORLD, start_method="spawn", join=True)
    r0, r1 = results[0], results[1]
    wl = W.small_ragged(n_tensors=200, world_size=WORLD, rank=0, grad_dtype="f32")
    # the ranges partition [0, total) in rank order and both ranks agree on them
    assert r0["ranges"] == r1["ranges"]
    (a0, b0), (a1, b1) = r0["ranges"]
    assert a0 == 0 and b0 == a1 and b1 == wl.total
    # the gathered vector: each rank's own value at its index, identical on both ranks
    for case in ("finite", "nonfinite"):
        g0, g1 = r0[case]["gathered"], r1[case]["gathered"]
        assert g0 == g1 or (case == "nonfinite" and all(
            (math.isinf(x) and math.isinf(y)) or x == y for x, y in zip(g0, g1)))
        assert g0[0] == r0[case]["local"] and (g0[1] == r1[case]["local"] or math.isinf(r1[case]["local"]))
        assert r0[case]["coef"] == r1[case]["coef"] and r0[case]["finite"] == r1[case]["finite"]
    # the rank-order total is the norm over the whole flat buffer
    full = W.flat_grads(wl, 1, 0, 0, wl.total).numpy()
    ref = oracle.clip(oracle.sqnorm(full), 0.0, wl.max_norm)
    assert abs(r0["finite"]["norm"] - ref.norm) <= 1e-14 * ref.norm
    assert r0["finite"]["finite"]
    # one rank's overflow makes every rank skip
    assert not r0["nonfinite"]["finite"] and not r1["nonfinite"]["finite"]
