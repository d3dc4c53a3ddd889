"""The ZeRO-2/3 data plane on one GPU against the oracle.

Kernel level: zero_reduce_chunks (the local reduction of a reduce-scatter)
bit for bit against the oracle's rank-order sum for every grad dtype, rank
counts 1..8, first pass and accumulate, with and without the fused norm,
sizes spanning several norm tiles with a ragged tail, padded blocks whose
padding is never read, vector and element paths (misaligned accumulator or
block stride), the non-finite flag, and guard bands around every buffer.

Step level: four ZeRO-2 ranks emulated one after another on one GPU.  The
exchange each rank would receive from an all-to-all is built by slicing the
ranks' padded flat grads (torch copies: the data movement only), then every
rank runs its reduction with the fused norm over two micro-batches; the
rank-order vector of the local sums of squares stands in for the 8-byte
all-gather; every rank's combine + AdamW writes its slice of one shared
low-precision FlatParameter, which is what the in-place all-gather would
leave on every rank.  No kernel waits on another rank.  Checked against the
oracle's reduce-scatter, global-norm clip and AdamW, bit for bit.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from _helpers import RTOL_NORM, assert_close_f32, bits_equal_f32, raw

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
GUARD = 40
TDT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fsdp_sharded_mixed_flatparameter_gb300 import build, zero_shard
    build.build()
    zero_shard.lib()


def _guarded(n, dtype, offset, fill=None):
    base = torch.empty(n + offset + GUARD, dtype=dtype, device=DEV)
    base.view(torch.uint8).fill_(0xFF)
    t = base[offset:offset + n]
    if fill is not None:
        t.copy_(fill)
    return base, t, base.clone()


def _guards_intact(base, snap, offset, n):
    es = base.element_size()
    b, s = base.view(torch.uint8), snap.view(torch.uint8)
    return torch.equal(b[:offset * es], s[:offset * es]) and torch.equal(b[(offset + n) * es:], s[(offset + n) * es:])


def _blocks(world, stride, n, dtype, seed):
    """world blocks of `stride` elements: n random grads each, the padding NaN bytes."""
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(world, stride, generator=g) * 1e-3 * torch.exp(torch.randn(world, 1, generator=g)))
    x = x.to(TDT[dtype])
    x.view(torch.uint8).view(world, -1)[:, n * x.element_size():] = 0xFF  # padding: never read
    return x


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
@pytest.mark.parametrize("accumulate", [False, True])
@pytest.mark.parametrize("fused", [False, True])
def test_reduce_chunks_matches_oracle_bit_exact(dtype, world, accumulate, fused):
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    n = 3 * 32768 + 777  # several norm tiles and a ragged tail
    for trial, (acc_off, pad) in enumerate([(0, 16), (0, 5), (3, 16)]):
        # pad 16: every block vector-aligned; pad 5: odd stride (element path); acc_off 3: misaligned accumulator
        stride = n + pad
        host = _blocks(world, stride, n, dtype, 17 * world + trial)
        chunks = host.to(DEV)
        acc0 = (torch.randn(n, generator=torch.Generator().manual_seed(trial)) * 1e-3).float()
        base, acc, _ = _guarded(n, torch.float32, acc_off, acc0.to(DEV))
        snap = base.clone()
        flag = torch.zeros(1, dtype=torch.int32, device=DEV)
        ws = torch.empty(zs.zero_grad_sqnorm_workspace_bytes(n), dtype=torch.uint8, device=DEV) if fused else None
        scale = 1.0 / world
        zs.zero_reduce_chunks(acc, chunks, n, scale, accumulate, flag, ws)
        torch.cuda.synchronize()
        assert _guards_intact(base, snap, acc_off, n), "write outside the accumulator"
        ref = acc0.numpy().copy()
        blocks = raw(host) if dtype == "f32" else host.view(torch.int16).numpy().view(np.uint16)
        assert not oracle.reduce_chunks(ref, np.ascontiguousarray(blocks), dtype, n, scale, accumulate)
        got = raw(acc)
        assert bits_equal_f32(got, ref), f"trial {trial}: reduction not bit-exact"
        assert flag.item() == 0
        if fused:
            # the fused partials equal the separate norm kernel's over the written values
            out_f, out_s = zs.new_norm_result(DEV), zs.new_norm_result(DEV)
            zs.zero_grad_sqnorm_finalize(ws, n, 0.0, 1.0, out_f)
            ws2 = torch.empty_like(ws)
            zs.zero_grad_sqnorm(acc.clone(), 0.0, 1.0, ws2, out_s)
            torch.cuda.synchronize()
            assert bytes(out_f.cpu().numpy()) == bytes(out_s.cpu().numpy())
            r = zs.decode_norm_result(out_f)
            cr = oracle.clip(oracle.sqnorm(ref), 0.0, 1.0)
            assert abs(r.norm - cr.norm) <= RTOL_NORM * cr.norm


def test_reduce_chunks_edge_cases():
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    for n in (0, 1, 7, 8, 9, 32768, 32769):
        for world in (1, 5):
            host = _blocks(world, n + 8, n, "bf16", n + world)
            acc = torch.full((max(n, 1),), 7.0, device=DEV)
            zs.zero_reduce_chunks(acc, host.to(DEV), n, 0.5, False, flag)
            ref = np.full(max(n, 1), 7.0, np.float32)
            oracle.reduce_chunks(ref, np.ascontiguousarray(host.view(torch.int16).numpy().view(np.uint16)),
                                 "bf16", n, 0.5, False)
            torch.cuda.synchronize()
            assert bits_equal_f32(raw(acc), ref), (n, world)
    assert flag.item() == 0
    # a non-finite value in one rank's block raises the flag; argument checks
    host = _blocks(3, 40000, 40000, "f16", 1)
    host[2, 33000] = float("inf")
    acc = torch.zeros(40000, device=DEV)
    zs.zero_reduce_chunks(acc, host.to(DEV), 40000, 1.0 / 3, False, flag)
    torch.cuda.synchronize()
    assert flag.item() == 1 and torch.isinf(acc[33000])
    with pytest.raises(ValueError):  # a block shorter than n
        zs.zero_reduce_chunks(acc, torch.zeros(2, 10, dtype=torch.bfloat16, device=DEV), 11, 1.0, False)
    L = zs.lib()
    dev_chunks = host.to(DEV)  # device addresses, though none of these calls gets past the host checks
    a, c = ctypes.c_void_p(acc.data_ptr()), ctypes.c_void_p(dev_chunks.data_ptr())
    # checked on the host before any launch: no chunks, stride shorter than n, bad dtype, non-finite scale
    assert L.zero_reduce_chunks(a, c, zs.ZERO_F16, 0, 10, 10, 1.0, None, 0, None, None, 0, None) == zs.ZERO_EINVAL
    assert L.zero_reduce_chunks(a, c, zs.ZERO_F16, 2, 5, 10, 1.0, None, 0, None, None, 0, None) == zs.ZERO_EINVAL
    assert L.zero_reduce_chunks(a, c, 7, 2, 10, 10, 1.0, None, 0, None, None, 0, None) == zs.ZERO_EINVAL
    assert L.zero_reduce_chunks(a, c, zs.ZERO_F16, 2, 10, 10, float("nan"), None, 0, None, None, 0, None) == zs.ZERO_EINVAL


def test_four_ranks_zero2_step_through_the_data_plane():
    """Four ZeRO-2 ranks, two micro-batches each reduced as it comes, global norm, AdamW,
    all-gather of the bf16 parameters: bit for bit against the oracle."""
    from fsdp_sharded_mixed_flatparameter_gb300 import FlatShardAdamW, zero_shard as zs
    from fsdp_sharded_mixed_flatparameter_gb300.dataplane import chunk_layout
    import workloads as W
    world, M, steps = 4, 2, 3
    wl = W.small_ragged(n_tensors=700, max_log2=13, world_size=world, rank=0, max_norm=0.2)
    total = wl.total
    chunk, padded = chunk_layout(total, world)
    assert chunk == -(-total // world) and padded % world == 0 and padded - total < world
    flat_param = torch.zeros(padded, dtype=torch.bfloat16, device=DEV)  # the all-gather's result
    opts, states = [], []
    for r in range(world):
        s, e = oracle.shard_range(total, world, r)
        master = W.master_init(wl, s, e)
        opts.append(FlatShardAdamW(wl.numels, world_size=world, rank=r, lr=wl.lr, betas=wl.betas, eps=wl.eps,
                                   weight_decay=wl.weight_decay, max_norm=wl.max_norm, device=DEV,
                                   master=master.to(DEV), lowp_out=flat_param[s:e]))
        states.append(oracle.new_state(raw(master)))
    for t in range(1, steps + 1):
        # every rank's full flat bf16 grad of each micro-batch, padded with zeros
        grads = [[torch.zeros(padded, dtype=torch.bfloat16, device=DEV) for _ in range(M)] for _ in range(world)]
        for r in range(world):
            for j in range(M):
                grads[r][j][:total] = W.flat_grads(wl.with_(seed=100 + r), t, j, 0, total, device=DEV)
        ref_acc = [np.zeros(max(opts[r].n, 1), np.float32) for r in range(world)]
        for j in range(M):
            for q, opt in enumerate(opts):
                # what rank q receives from the all-to-all: block r = rank r's chunk q
                recv = torch.stack([grads[r][j][q * chunk:(q + 1) * chunk] for r in range(world)]).contiguous()
                opt.reduce(recv, accumulate=j > 0, scale=1.0 / (world * M), fuse_norm=j == M - 1)
                oracle.reduce_chunks(ref_acc[q], np.ascontiguousarray(raw(recv)), "bf16", opt.n, 1.0 / (world * M),
                                     j > 0)
        gathered = torch.cat([opt.local_sqnorm() for opt in opts])  # the 8-byte all-gather, rank order
        results = []
        for opt in opts:
            opt.launch_step(gathered_sqnorms=gathered)
            results.append(opt.finish_step())
        assert all(rr == results[0] for rr in results)
        full = np.concatenate([ref_acc[q][:opts[q].n] for q in range(world)])
        cr = oracle.clip(oracle.sqnorm(full), 0.0, wl.max_norm)
        assert abs(results[0].norm - cr.norm) <= 1e-12 * cr.norm and cr.coef < 1.0
        for q, (opt, st) in enumerate(zip(opts, states)):
            assert bits_equal_f32(raw(opt.shard_grad()), ref_acc[q][:opt.n]), f"rank {q} reduced grad"
            st.t += 1
            sc = oracle.adamw_scalars(wl.lr, wl.betas[0], wl.betas[1], wl.eps, wl.weight_decay, st.t)
            oracle.adamw(st.p, st.m, st.v, np.ascontiguousarray(ref_acc[q][:opt.n]), sc, cr.coef, st.lowp)
            for got, ref in ((opt.master, st.p), (opt.exp_avg, st.m), (opt.exp_avg_sq, st.v)):
                assert_close_f32(raw(got), ref)
                if results[0].clip_coef == cr.coef:
                    assert bits_equal_f32(raw(got), ref)
        # the gathered low-precision FlatParameter: every rank's slice, padding untouched
        lowp = raw(flat_param)
        assert np.array_equal(lowp[:total], np.concatenate([st.lowp for st in states]))
        assert not lowp[total:].any()


def test_one_rank_of_eight_full_size_sampled():
    """One rank of an 8-rank ZeRO-2 Llama-7B job at full size, in the launch configuration
    `bench.py --dataplane-ranks 8` times (842,301,952 shard params, 8 received bf16 blocks,
    the reduction with the fused norm, then AdamW), 2 steps: the oracle reduces every element
    for the norm (host threads over disjoint chunks, exact fsum) and the state is compared at
    1M sampled positions (element-wise, so sampling is exact)."""
    import math
    from concurrent.futures import ThreadPoolExecutor
    from fsdp_sharded_mixed_flatparameter_gb300 import FlatShardAdamW, chunk_layout, zero_shard as zs
    import workloads as W
    from _configs import ORACLE_THREADS
    wl = W.llama7b()
    N, r = 8, 3
    total = wl.total
    chunk, _ = chunk_layout(total, N)
    s, e = oracle.shard_range(total, N, r)
    n = e - s
    assert n == chunk == 842301952
    master = W.master_init(wl, s, e, device=DEV)
    opt = FlatShardAdamW(wl.numels, world_size=N, rank=r, lr=wl.lr, betas=wl.betas, eps=wl.eps,
                         weight_decay=wl.weight_decay, max_norm=wl.max_norm, device=DEV, master=master)
    rng = np.random.default_rng(7)
    idx = np.unique(np.concatenate([rng.integers(0, n, size=1_000_000), [0, n - 1]])).astype(np.int64)
    d_idx = torch.from_numpy(idx).to(DEV)
    st = oracle.new_state(raw(master.index_select(0, d_idx)))
    del master
    recv = torch.zeros(N, chunk, dtype=torch.bfloat16, device=DEV)
    step_chunk = 1 << 25
    for t in (1, 2):
        for j in range(N):  # rank j's values of this rank's shard, as the exchange delivers them
            recv[j, :n] = W.flat_grads(wl.with_(seed=wl.seed + j), t, 0, s, e, device=DEV)
        opt.reduce(recv, accumulate=False, scale=1.0 / N, fuse_norm=True)
        opt.launch_step()
        res = opt.finish_step()
        g_sample = np.empty(idx.size, np.float32)

        def oracle_chunk(a):
            b = min(a + step_chunk, n)
            blocks = np.ascontiguousarray(raw(recv[:, a:b]))
            acc = np.empty(b - a, np.float32)
            oracle.reduce_chunks(acc, blocks, "bf16", b - a, 1.0 / N, False)
            sel = (idx >= a) & (idx < b)
            g_sample[sel] = acc[idx[sel] - a]
            return oracle.sqnorm(acc)

        with ThreadPoolExecutor(max_workers=ORACLE_THREADS) as pool:
            sq = math.fsum(pool.map(oracle_chunk, range(0, n, step_chunk)))
        cr = oracle.clip(sq, 0.0, wl.max_norm)
        assert res.finite and cr.finite and cr.coef < 1.0
        assert abs(res.norm - cr.norm) <= RTOL_NORM * cr.norm, (res.norm, cr.norm)
        st.t += 1
        sc = oracle.adamw_scalars(wl.lr, wl.betas[0], wl.betas[1], wl.eps, wl.weight_decay, st.t)
        oracle.adamw(st.p, st.m, st.v, g_sample, sc, cr.coef, st.lowp)
        assert opt.t == st.t
        for got, ref in ((opt.master, st.p), (opt.exp_avg, st.m), (opt.exp_avg_sq, st.v)):
            g = raw(got.index_select(0, d_idx))
            assert_close_f32(g, ref)
            if res.clip_coef == cr.coef:
                assert bits_equal_f32(g, ref)
        if res.clip_coef == cr.coef:
            assert np.array_equal(raw(opt.lowp.index_select(0, d_idx)), st.lowp)
        print(f"rank {r} of {N}, step {t}: norm gpu={res.norm:.17g} oracle={cr.norm:.17g} "
              f"coef equal={res.clip_coef == cr.coef}")


def test_emulated_ranks_captured_in_one_graph():
    """The data plane's device work for three emulated ranks -- each rank's reduction of its
    received blocks with the fused norm, the local sums of squares gathered in rank order,
    the combine, the device step count and AdamW into the shared low-precision FlatParameter
    -- captured once in a CUDA graph and replayed over new received blocks (and a NaN in one
    rank's block at step 2): bit for bit against the oracle after every replay."""
    from fsdp_sharded_mixed_flatparameter_gb300 import FlatShardAdamW, chunk_layout, zero_shard as zs
    import workloads as W
    world, steps = 3, 4
    wl = W.small_ragged(n_tensors=400, max_log2=13, world_size=world, rank=0, max_norm=0.3, grad_dtype="f16")
    total = wl.total
    chunk, padded = chunk_layout(total, world)
    flat_param = torch.zeros(padded, dtype=torch.bfloat16, device=DEV)
    opts, states = [], []
    for r in range(world):
        s, e = oracle.shard_range(total, world, r)
        master = W.master_init(wl, s, e)
        opts.append(FlatShardAdamW(wl.numels, world_size=world, rank=r, lr=wl.lr, betas=wl.betas, eps=wl.eps,
                                   weight_decay=wl.weight_decay, max_norm=wl.max_norm, device=DEV,
                                   master=master.to(DEV), lowp_out=flat_param[s:e], capturable=True))
        states.append(oracle.new_state(raw(master)))
    recv = [torch.zeros(world, chunk, dtype=torch.float16, device=DEV) for _ in range(world)]  # rank q's inbox
    gathered = torch.zeros(world, dtype=torch.float64, device=DEV)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for q, opt in enumerate(opts):
            opt.reduce(recv[q], accumulate=False, scale=1.0 / world, fuse_norm=True)
            gathered[q:q + 1].copy_(opt.local_sqnorm())
        for opt in opts:
            opt.launch_step(gathered_sqnorms=gathered)
    for t in range(1, steps + 1):
        full = [torch.zeros(padded, dtype=torch.float16, device=DEV) for _ in range(world)]
        for r in range(world):
            full[r][:total] = W.flat_grads(wl.with_(seed=200 + r), t, 0, 0, total, device=DEV)
        if t == 2:
            full[2][3] = float("nan")  # in rank 0's chunk: every rank must skip
        for q in range(world):  # what the all-to-all delivers
            recv[q].copy_(torch.stack([full[r][q * chunk:(q + 1) * chunk] for r in range(world)]))
        graph.replay()
        torch.cuda.synchronize()
        accs = []
        for q in range(world):
            n = opts[q].n
            a = np.zeros(max(n, 1), np.float32)
            oracle.reduce_chunks(a, np.ascontiguousarray(raw(recv[q])), "f16", n, 1.0 / world, False)
            accs.append(a[:n])
        cr = oracle.clip(oracle.sqnorm(np.concatenate(accs)), 0.0, wl.max_norm)
        assert cr.finite == (t != 2)
        for q, (opt, st) in enumerate(zip(opts, states)):
            r = opt.finish_step()
            assert r.finite == cr.finite
            if cr.finite:
                st.t += 1
                sc = oracle.adamw_scalars(wl.lr, wl.betas[0], wl.betas[1], wl.eps, wl.weight_decay, st.t)
                oracle.adamw(st.p, st.m, st.v, np.ascontiguousarray(accs[q]), sc, cr.coef, st.lowp)
        for q, (opt, st) in enumerate(zip(opts, states)):
            assert opt.t == st.t == (t if t < 2 else t - 1)
            for got, ref in ((opt.master, st.p), (opt.exp_avg, st.m), (opt.exp_avg_sq, st.v)):
                assert bits_equal_f32(raw(got), ref), (t, q)
        assert np.array_equal(raw(flat_param)[:total], np.concatenate([st.lowp for st in states]))


def _llama_units(numels):
    """Split a Llama tensor list into FSDP units: the embedding, each transformer block
    (9 tensors), and the final norm with the output head."""
    units = [list(numels[:1])]
    i = 1
    while len(numels) - i > 2:
        units.append(list(numels[i:i + 9]))
        i += 9
    units.append(list(numels[i:]))
    assert sum(map(len, units)) == len(numels)
    return units


def test_units_share_one_global_clip():
    """Five FSDP units (embedding, three blocks, head), each its own FlatParameter and data
    plane, stepped with one clip over the whole model: every unit's state bit for bit
    against the oracle's global-norm step, three steps (the second without the norm fused
    into the reductions)."""
    from fsdp_sharded_mixed_flatparameter_gb300 import ZeroUnits
    import workloads as W
    wl = W.small_llama(layers=3, hidden=256, mlp=688, vocab=1000, max_norm=0.05)
    units = _llama_units(wl.numels)
    offs = np.concatenate([[0], np.cumsum([sum(u) for u in units])]).astype(np.int64)
    masters = [W.master_init(wl, int(offs[i]), int(offs[i + 1])) for i in range(len(units))]
    zu = ZeroUnits(units, device=DEV, lr=wl.lr, betas=wl.betas, eps=wl.eps, weight_decay=wl.weight_decay,
                   max_norm=wl.max_norm, masters=[m.to(DEV) for m in masters])
    states = [oracle.new_state(raw(m)) for m in masters]
    for t in range(1, 4):
        grads = []
        for i, u in enumerate(zu.units):
            g = W.flat_grads(wl, t, 0, int(offs[i]), int(offs[i + 1]), device=DEV)
            u.flat_grad[:g.numel()] = g
            grads.append(oracle.to_f32(raw(g), "bf16"))
        zu.reduce_scatter_grads(fuse_norm=t != 2)  # step 2: the norm partials from a separate pass
        res = zu.step()
        cr = oracle.clip(oracle.sqnorm(np.concatenate(grads)), 0.0, wl.max_norm)
        assert res.finite and cr.coef < 1.0
        assert abs(res.norm - cr.norm) <= 1e-12 * cr.norm
        for u, st, g in zip(zu.units, states, grads):
            st.t += 1
            sc = oracle.adamw_scalars(wl.lr, wl.betas[0], wl.betas[1], wl.eps, wl.weight_decay, st.t)
            oracle.adamw(st.p, st.m, st.v, g, sc, cr.coef, st.lowp)
            assert u.opt.t == st.t
            if res.clip_coef == cr.coef:
                for got, ref in ((u.opt.master, st.p), (u.opt.exp_avg, st.m), (u.opt.exp_avg_sq, st.v)):
                    assert bits_equal_f32(raw(got), ref), t
                assert np.array_equal(raw(u.flat_param)[:st.lowp.size], st.lowp)
            else:
                assert_close_f32(raw(u.opt.master), st.p)


def test_units_captured_in_one_graph():
    """The five-unit step captured once (every unit's reduction with the fused norm, the one
    finalize, the combine, the device step count and every unit's AdamW) and replayed over
    new grads -- a NaN in the last unit at step 2 skips every unit -- bit for bit against
    the oracle after every replay."""
    from fsdp_sharded_mixed_flatparameter_gb300 import ZeroUnits
    import workloads as W
    wl = W.small_llama(layers=3, hidden=256, mlp=688, vocab=1000, max_norm=0.05)
    units = _llama_units(wl.numels)
    offs = np.concatenate([[0], np.cumsum([sum(u) for u in units])]).astype(np.int64)
    masters = [W.master_init(wl, int(offs[i]), int(offs[i + 1])) for i in range(len(units))]
    zu = ZeroUnits(units, device=DEV, lr=wl.lr, betas=wl.betas, eps=wl.eps, weight_decay=wl.weight_decay,
                   max_norm=wl.max_norm, masters=[m.to(DEV) for m in masters], capturable=True)
    states = [oracle.new_state(raw(m)) for m in masters]
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        zu.reduce_scatter_grads()
        zu.launch_step()
    for t in range(1, 5):
        grads = []
        for i, u in enumerate(zu.units):
            g = W.flat_grads(wl, t, 0, int(offs[i]), int(offs[i + 1]), device=DEV)
            if t == 2 and i == len(units) - 1:
                g[7] = float("nan")
            u.flat_grad[:g.numel()] = g
            grads.append(oracle.to_f32(raw(g), "bf16"))
        graph.replay()
        res = zu.finish_step()
        cr = oracle.clip(oracle.sqnorm(np.concatenate(grads)), 0.0, wl.max_norm)
        assert res.finite == cr.finite == (t != 2)
        for u, st, g in zip(zu.units, states, grads):
            if cr.finite:
                st.t += 1
                sc = oracle.adamw_scalars(wl.lr, wl.betas[0], wl.betas[1], wl.eps, wl.weight_decay, st.t)
                oracle.adamw(st.p, st.m, st.v, g, sc, cr.coef, st.lowp)
            assert u.opt.t == st.t == (t if t < 2 else t - 1)
            for got, ref in ((u.opt.master, st.p), (u.opt.exp_avg, st.m), (u.opt.exp_avg_sq, st.v)):
                assert bits_equal_f32(raw(got), ref), t
            assert np.array_equal(raw(u.flat_param)[:st.lowp.size], st.lowp)
