"""The product's multi-rank step across real processes: two ranks on one GPU.

Two processes, one rank each, both on cuda:0, exchange through a gloo
process group (the ranks' only exchange is the 8-byte local sum of squares
of ZeRO-2/3 global grad-norm clipping; gloo stages it through host memory).
No kernel waits on another rank: each process runs its own kernels and the
exchange happens on the host between them.  Each rank steps its own shard
with ``FlatShardAdamW.step(process_group=...)`` (flatten with the fused norm
first) or ``step_tensors(process_group=...)``, on a side stream rather than
torch's current stream, for four steps; at step 3 a grad inside rank 1's
shard is infinite, so both ranks must skip that step together.  Every rank's
norm, coefficient and skip decision must be the same, and every rank's state
must equal the oracle's global-norm step bit for bit.
"""
import datetime
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu
WORLD = 2
STEPS = 4
BAD_STEP = 3


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _workload():
    import workloads as W
    return W.small_ragged(n_tensors=300, world_size=WORLD, rank=0, max_norm=0.5)


def _grads(wl, t, dev):
    import workloads as W
    tg = W.tensor_grads(wl, t, 0, device=dev)
    if t == BAD_STEP:
        tg.tensors[-1][0] = float("inf")  # the last tensor lies in rank 1's shard
    return tg


def _rank_main(rank, port, mode, results):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD, timeout=datetime.timedelta(seconds=180))
    try:
        import workloads as W
        from fsdp_sharded_mixed_flatparameter_gb300 import FlatShardAdamW
        dev = torch.device("cuda:0")
        torch.cuda.set_device(dev)
        wl = _workload().with_(rank=rank)
        opt = FlatShardAdamW(wl.numels, world_size=WORLD, rank=rank, lr=wl.lr, betas=wl.betas, eps=wl.eps,
                             weight_decay=wl.weight_decay, max_norm=wl.max_norm, device=dev, master=None)
        opt.master.copy_(W.master_init(wl, opt.start, opt.end))
        side = torch.cuda.Stream(device=dev)
        norms = []
        for t in range(1, STEPS + 1):
            tg = _grads(wl, t, dev)
            side.wait_stream(torch.cuda.current_stream(dev))  # the grads were written on the current stream
            if mode == "step":
                opt.flatten(tg.tensors, accumulate=False, fuse_norm=True, stream=side)
                r = opt.step(stream=side, process_group=dist.group.WORLD)
            else:
                r = opt.step_tensors(tg.tensors, stream=side, process_group=dist.group.WORLD)
            norms.append((r.sqnorm, r.norm, r.clip_coef, r.finite, opt.t))
        torch.cuda.synchronize(dev)
        results[rank] = {"norms": norms, "range": (opt.start, opt.end),
                         **{k: getattr(opt, k).cpu().view(torch.int32 if k != "lowp" else torch.int16)
                            .numpy().tobytes() for k in ("master", "exp_avg", "exp_avg_sq", "lowp")}}
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("mode", ["step", "step_tensors"])
def test_two_processes_global_norm_step(mode):
    import oracle
    from _helpers import raw
    from fsdp_sharded_mixed_flatparameter_gb300 import build
    import workloads as W
    build.build()  # once, before the ranks start (they only load it)
    ctx = mp.get_context("spawn")
    results = ctx.Manager().dict()
    mp.start_processes(_rank_main, args=(_free_port(), mode, results), nprocs=WORLD, start_method="spawn", join=True)
    r0, r1 = results[0], results[1]
    # every rank saw the same norm, coefficient and skip decision at every step
    # (repr: a skipped step's norm is NaN on both ranks, and NaN != NaN)
    assert repr(r0["norms"]) == repr(r1["norms"])
    assert [x[3] for x in r0["norms"]] == [t != BAD_STEP for t in range(1, STEPS + 1)]
    assert [x[4] for x in r0["norms"]] == [1, 2, 2, 3]

    wl = _workload()
    states = {}
    for rank, res in ((0, r0), (1, r1)):
        s, e = oracle.shard_range(wl.total, WORLD, rank)
        assert tuple(res["range"]) == (s, e)
        states[rank] = oracle.new_state(raw(W.master_init(wl, s, e)))
    for t in range(1, STEPS + 1):
        tg = _grads(wl, t, torch.device("cuda:0"))  # the ranks' draws (CPU and CUDA generators differ)
        full = np.zeros(wl.total, np.float32)
        oracle.flatten([raw(x) for x in tg.tensors], wl.numels, "bf16", 0, wl.total, 1.0, full, False)
        cr = oracle.clip(oracle.sqnorm(full), 0.0, wl.max_norm)
        sq, nv, coef, fin, _ = r0["norms"][t - 1]
        assert fin == cr.finite
        if not cr.finite:
            continue
        assert abs(nv - cr.norm) <= 1e-12 * cr.norm and coef == cr.coef
        for rank in (0, 1):
            st = states[rank]
            s, e = oracle.shard_range(wl.total, WORLD, rank)
            st.t += 1
            sc = oracle.adamw_scalars(wl.lr, wl.betas[0], wl.betas[1], wl.eps, wl.weight_decay, st.t)
            oracle.adamw(st.p, st.m, st.v, np.ascontiguousarray(full[s:e]), sc, cr.coef, st.lowp)
    for rank, res in ((0, r0), (1, r1)):
        st = states[rank]
        assert st.t == 3
        assert res["master"] == st.p.tobytes(), f"rank {rank} master"
        assert res["exp_avg"] == st.m.tobytes(), f"rank {rank} exp_avg"
        assert res["exp_avg_sq"] == st.v.tobytes(), f"rank {rank} exp_avg_sq"
        assert res["lowp"] == st.lowp.tobytes(), f"rank {rank} lowp"


# ------------------------------------------------------------------ ZeRO-2 data plane
M_DP = 2  # micro-batches, each reduced as it comes


def _dp_grads(wl, rank, t, j, dev):
    """Rank `rank`'s full flat bf16 grad of micro-batch j (rank 1's holds an inf at step BAD_STEP,
    inside rank 0's chunk: the exchange carries it to rank 0)."""
    import workloads as W
    g = W.flat_grads(wl.with_(seed=100 + rank), t, j, 0, wl.total, device=dev)
    if t == BAD_STEP and rank == 1 and j == 0:
        g[5] = float("inf")
    return g


def _dp_rank_main(rank, port, results):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD, timeout=datetime.timedelta(seconds=180))
    try:
        import workloads as W
        from fsdp_sharded_mixed_flatparameter_gb300 import ZeroDataPlane, zero_shard_range
        dev = torch.device("cuda:0")
        torch.cuda.set_device(dev)
        wl = _workload()
        s, e = zero_shard_range(wl.total, WORLD, rank)
        dp = ZeroDataPlane(wl.numels, group=dist.group.WORLD, device=dev, lr=wl.lr, betas=wl.betas, eps=wl.eps,
                           weight_decay=wl.weight_decay, max_norm=wl.max_norm, master=W.master_init(wl, s, e).to(dev))
        side = torch.cuda.Stream(device=dev)
        norms = []
        for t in range(1, STEPS + 1):
            for j in range(M_DP):
                dp.flat_grad[:wl.total] = _dp_grads(wl, rank, t, j, dev)  # what backward leaves
                side.wait_stream(torch.cuda.current_stream(dev))
                dp.reduce_scatter_grads(accumulate=j > 0, scale=1.0 / (WORLD * M_DP), fuse_norm=j == M_DP - 1,
                                        stream=side)
                torch.cuda.current_stream(dev).wait_stream(side)  # flat_grad is rewritten next
            r = dp.step(stream=side)
            norms.append((r.sqnorm, r.norm, r.clip_coef, r.finite, dp.opt.t))
        torch.cuda.synchronize(dev)
        results[rank] = {"norms": norms, "range": (s, e), "flat_param": dp.flat_param.cpu().view(torch.int16)
                         .numpy().tobytes(), "padded": dp.padded,
                         **{k: getattr(dp.opt, k).cpu().view(torch.int32).numpy().tobytes()
                            for k in ("master", "exp_avg", "exp_avg_sq")}}
    finally:
        dist.destroy_process_group()


def test_two_processes_zero2_data_plane():
    """ZeroDataPlane across two processes: all-to-all of the padded flat bf16 grads, fp32
    rank-order reduction with the fused norm over two micro-batches, global norm, AdamW
    into the shard's slice of the bf16 FlatParameter, in-place all-gather -- on a side
    stream, with a non-finite grad exchanged into the other rank's shard at step 3."""
    import oracle
    from _helpers import raw
    from fsdp_sharded_mixed_flatparameter_gb300 import build
    import workloads as W
    build.build()
    ctx = mp.get_context("spawn")
    results = ctx.Manager().dict()
    mp.start_processes(_dp_rank_main, args=(_free_port(), results), nprocs=WORLD, start_method="spawn", join=True)
    r0, r1 = results[0], results[1]
    assert repr(r0["norms"]) == repr(r1["norms"])  # NaN-aware: a skipped step's norm is NaN
    assert [x[3] for x in r0["norms"]] == [t != BAD_STEP for t in range(1, STEPS + 1)]
    assert [x[4] for x in r0["norms"]] == [1, 2, 2, 3]
    assert r0["flat_param"] == r1["flat_param"], "ranks hold different parameters after the all-gather"

    wl = _workload()
    total = wl.total
    chunk = -(-total // WORLD)
    dev = torch.device("cuda:0")
    states = {}
    for rank in range(WORLD):
        s, e = oracle.shard_range(total, WORLD, rank)
        states[rank] = oracle.new_state(raw(W.master_init(wl, s, e)))
    for t in range(1, STEPS + 1):
        acc = {q: np.zeros(max(states[q].p.size, 1), np.float32) for q in range(WORLD)}
        for j in range(M_DP):
            full = [np.concatenate([raw(_dp_grads(wl, r, t, j, dev)), np.zeros(WORLD * chunk - total, np.uint16)])
                    for r in range(WORLD)]
            for q in range(WORLD):
                blocks = np.ascontiguousarray(np.stack([f[q * chunk:(q + 1) * chunk] for f in full]))
                oracle.reduce_chunks(acc[q], blocks, "bf16", states[q].p.size, 1.0 / (WORLD * M_DP), j > 0)
        grad = np.concatenate([acc[q][:states[q].p.size] for q in range(WORLD)])
        cr = oracle.clip(oracle.sqnorm(grad), 0.0, wl.max_norm)
        _, nv, coef, fin, _ = r0["norms"][t - 1]
        assert fin == cr.finite
        if not cr.finite:
            continue
        assert abs(nv - cr.norm) <= 1e-12 * cr.norm and coef == cr.coef
        for q in range(WORLD):
            st = states[q]
            st.t += 1
            sc = oracle.adamw_scalars(wl.lr, wl.betas[0], wl.betas[1], wl.eps, wl.weight_decay, st.t)
            oracle.adamw(st.p, st.m, st.v, np.ascontiguousarray(acc[q][:st.p.size]), sc, cr.coef, st.lowp)
    lowp = np.frombuffer(r0["flat_param"], np.uint16)
    assert np.array_equal(lowp[:total], np.concatenate([states[q].lowp for q in range(WORLD)]))
    assert not lowp[total:].any()
    for q, res in ((0, r0), (1, r1)):
        st = states[q]
        assert res["master"] == st.p.tobytes() and res["exp_avg"] == st.m.tobytes()
        assert res["exp_avg_sq"] == st.v.tobytes()


# ------------------------------------------------------------------ several FSDP units
def _unit_workload():
    import workloads as W
    return W.small_llama(layers=2, hidden=256, mlp=688, vocab=1000, max_norm=0.05)


def _units_of(numels):
    return [list(numels[:1]), list(numels[1:10]), list(numels[10:19]), list(numels[19:])]


def _units_rank_main(rank, port, results):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=WORLD, timeout=datetime.timedelta(seconds=180))
    try:
        import workloads as W
        from fsdp_sharded_mixed_flatparameter_gb300 import ZeroUnits, zero_shard_range
        dev = torch.device("cuda:0")
        torch.cuda.set_device(dev)
        wl = _unit_workload()
        units = _units_of(wl.numels)
        offs = np.concatenate([[0], np.cumsum([sum(u) for u in units])]).astype(np.int64)
        masters = []
        for i, u in enumerate(units):
            s, e = zero_shard_range(sum(u), WORLD, rank)
            masters.append(W.master_init(wl, int(offs[i]) + s, int(offs[i]) + e).to(dev))
        zu = ZeroUnits(units, group=dist.group.WORLD, device=dev, lr=wl.lr, betas=wl.betas, eps=wl.eps,
                       weight_decay=wl.weight_decay, max_norm=wl.max_norm, masters=masters)
        norms = []
        for t in range(1, 3):
            for i, u in enumerate(zu.units):
                u.flat_grad[:sum(units[i])] = W.flat_grads(wl.with_(seed=300 + rank), t, 0, int(offs[i]),
                                                           int(offs[i + 1]), device=dev)
            zu.reduce_scatter_grads()
            r = zu.step()
            norms.append((r.norm, r.clip_coef, r.finite))
        torch.cuda.synchronize(dev)
        results[rank] = {"norms": norms,
                         "params": [u.flat_param.cpu().view(torch.int16).numpy().tobytes() for u in zu.units],
                         "masters": [u.opt.master.cpu().numpy().tobytes() for u in zu.units]}
    finally:
        dist.destroy_process_group()


def test_two_processes_units_with_one_global_clip():
    """Four FSDP units across two processes (gloo): every unit exchanged and reduced on its
    own, one global norm over every unit of both ranks, every rank's parameters after the
    units' all-gathers equal to the oracle's, bit for bit."""
    import oracle
    from _helpers import raw
    from fsdp_sharded_mixed_flatparameter_gb300 import build
    import workloads as W
    build.build()
    ctx = mp.get_context("spawn")
    results = ctx.Manager().dict()
    mp.start_processes(_units_rank_main, args=(_free_port(), results), nprocs=WORLD, start_method="spawn",
                       join=True)
    r0, r1 = results[0], results[1]
    assert repr(r0["norms"]) == repr(r1["norms"]) and r0["params"] == r1["params"]
    wl = _unit_workload()
    units = _units_of(wl.numels)
    offs = np.concatenate([[0], np.cumsum([sum(u) for u in units])]).astype(np.int64)
    dev = torch.device("cuda:0")
    states = {}
    for i, u in enumerate(units):
        for rank in range(WORLD):
            s, e = oracle.shard_range(sum(u), WORLD, rank)
            states[i, rank] = oracle.new_state(raw(W.master_init(wl, int(offs[i]) + s, int(offs[i]) + e)))
    for t in range(1, 3):
        accs = {}
        for i, u in enumerate(units):
            total = sum(u)
            chunk = -(-total // WORLD)
            full = [np.concatenate([raw(W.flat_grads(wl.with_(seed=300 + r), t, 0, int(offs[i]), int(offs[i + 1]),
                                                     device=dev)), np.zeros(WORLD * chunk - total, np.uint16)])
                    for r in range(WORLD)]
            for q in range(WORLD):
                n = states[i, q].p.size
                a = np.zeros(max(n, 1), np.float32)
                oracle.reduce_chunks(a, np.ascontiguousarray(np.stack([f[q * chunk:(q + 1) * chunk] for f in full])),
                                     "bf16", n, 1.0 / WORLD, False)
                accs[i, q] = a[:n]
        cr = oracle.clip(oracle.sqnorm(np.concatenate([accs[k] for k in sorted(accs)])), 0.0, wl.max_norm)
        nv, coef, fin = r0["norms"][t - 1]
        assert fin and cr.finite and abs(nv - cr.norm) <= 1e-12 * cr.norm and coef == cr.coef and cr.coef < 1.0
        for k, st in states.items():
            st.t += 1
            sc = oracle.adamw_scalars(wl.lr, wl.betas[0], wl.betas[1], wl.eps, wl.weight_decay, st.t)
            oracle.adamw(st.p, st.m, st.v, np.ascontiguousarray(accs[k]), sc, cr.coef, st.lowp)
    for i, u in enumerate(units):
        lowp = np.frombuffer(r0["params"][i], np.uint16)
        assert np.array_equal(lowp[:sum(u)], np.concatenate([states[i, q].lowp for q in range(WORLD)]))
        for q, res in ((0, r0), (1, r1)):
            assert res["masters"][i] == states[i, q].p.tobytes(), (i, q)
