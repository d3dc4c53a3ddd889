"""Host logic of the ZeRO-2/3 data plane on CPU with gloo, world size 2 (no GPU).

Checks the padded chunk layout against the oracle's shard ranges, that the
all-to-all exchange delivers to rank q every rank's chunk q in rank order,
that the in-place all-gather leaves every rank's block on every rank, and
that ZeroDataPlane places each rank's low-precision parameter slice at its
shard's offset inside the full FlatParameter (so the AdamW write-back lands
where the all-gather sends it from).
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle

WORLD = 2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fsdp_sharded_mixed_flatparameter_gb300 import build
    build.build()


def test_chunk_layout_matches_shard_ranges():
    from fsdp_sharded_mixed_flatparameter_gb300 import chunk_layout
    for total in (0, 1, 2, 5, 7, 8, 9, 100, 10_007, 124_439_808, 6_738_415_616):
        for world in (1, 2, 3, 4, 7, 8, 64):
            chunk, padded = chunk_layout(total, world)
            assert chunk == -(-total // world) and padded == chunk * world
            assert padded >= total and padded - total < max(world, 1) or total == 0
            for r in range(world):
                s, e = oracle.shard_range(total, world, r)
                # rank r's shard is the head of its padded chunk (short or empty at the tail)
                assert s == min(r * chunk, total) and e - s <= chunk


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        from fsdp_sharded_mixed_flatparameter_gb300 import ZeroDataPlane, exchange_chunks, gather_shards
        chunk = 7
        send = torch.tensor([1000.0 * rank + k for k in range(WORLD * chunk)])
        recv = torch.full_like(send, -1.0)
        exchange_chunks(send, recv, dist.group.WORLD)
        full = torch.full((WORLD * chunk,), -1.0)
        full[rank * chunk:(rank + 1) * chunk] = 10.0 * (rank + 1)
        gather_shards(full, dist.group.WORLD)
        numels = [5, 4, 3]  # total 12: chunk 6, rank 1's shard [6, 12)
        dp = ZeroDataPlane(numels, group=dist.group.WORLD, device="cpu", lr=1e-3)
        # checkpoint round trip: a rank restores its own shard, the all-gather restores the rest
        dp.opt.lowp.copy_(torch.full((dp.opt.n,), float(rank + 1)))
        dp.opt.master.copy_(torch.arange(dp.opt.n, dtype=torch.float32) + 100 * rank)
        sd = dp.state_dict()
        dp2 = ZeroDataPlane(numels, group=dist.group.WORLD, device="cpu", lr=1e-3)
        dp2.load_state_dict(sd)
        ckpt = {"flat_param": dp2.flat_param.float().tolist(), "master": dp2.opt.master.tolist()}
        try:
            bad = dict(sd, rank=1 - rank)
            dp2.load_state_dict(bad)
            ckpt["refused"] = False
        except ValueError:
            ckpt["refused"] = True
        results[rank] = {
            "recv": recv.tolist(), "full": full.tolist(),
            "chunk": dp.chunk, "padded": dp.padded, "range": (dp.opt.start, dp.opt.end),
            "lowp_at": (dp.opt.lowp.data_ptr() - dp.flat_param.data_ptr()) // dp.flat_param.element_size(),
            "lowp_n": dp.opt.lowp.numel(), "grad_n": dp.opt.grad.numel(), "recv_n": dp.recv.numel(),
            "views": [(v.data_ptr() - dp.flat_grad.data_ptr()) // dp.flat_grad.element_size()
                      for v in dp.grad_views()],
            "ckpt": ckpt,
        }
    finally:
        dist.destroy_process_group()


def test_two_ranks_exchange_gather_and_layout():
    ctx = mp.get_context("spawn")
    results = ctx.Manager().dict()
    mp.start_processes(_rank_main, args=(_free_port(), results), nprocs=WORLD, start_method="spawn", join=True)
    chunk = 7
    for q in range(WORLD):
        r = results[q]
        # block j of rank q's receive buffer is rank j's chunk q
        want = [1000.0 * j + q * chunk + k for j in range(WORLD) for k in range(chunk)]
        assert r["recv"] == want, q
        assert r["full"] == [10.0 * (j + 1) for j in range(WORLD) for _ in range(chunk)]
        s, e = oracle.shard_range(12, WORLD, q)
        assert (r["chunk"], r["padded"]) == (6, 12) and tuple(r["range"]) == (s, e)
        assert r["lowp_at"] == s and r["lowp_n"] == e - s == r["grad_n"]
        assert r["recv_n"] == 12 and r["views"] == [0, 5, 9]
        # every rank's restored slice, gathered into every rank's full FlatParameter
        assert r["ckpt"]["flat_param"] == [1.0] * 6 + [2.0] * 6
        assert r["ckpt"]["master"] == [100.0 * q + k for k in range(6)] and r["ckpt"]["refused"]


def test_units_layout_on_the_host():
    """ZeroUnits builds one FlatParameter per unit, each with its own shard layout, and
    refuses a master list of the wrong length."""
    from fsdp_sharded_mixed_flatparameter_gb300 import ZeroUnits
    units = [[5], [4, 3, 9], [2]]
    zu = ZeroUnits(units, device="cpu", lr=1e-3)
    assert [u.total for u in zu.units] == [5, 16, 2]
    assert [u.flat_param.numel() for u in zu.units] == [5, 16, 2]  # one rank: no padding
    assert [u.opt.n for u in zu.units] == [5, 16, 2]
    with pytest.raises(ValueError):
        ZeroUnits(units, device="cpu", masters=[torch.zeros(5)])
