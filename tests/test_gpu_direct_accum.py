"""The direct path with micro-batch accumulation: the step's last micro-batch is
never written to the fp32 grad.  The norm pass forms fl(acc + fl(scale * x))
and writes only the norm partials (zero_flatten_cast, accumulate == 2), and
AdamW forms the same values again from the accumulator and the grads
(zero_adamw_step_tensors with d_acc).  Both must be bit-identical to the
accumulating flatten pass followed by the norm and AdamW -- and so to the
oracle -- while leaving the accumulator untouched."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _helpers import bits_equal_f32, norm_result_tensor, raw
from test_gpu_kernels import Guarded, _table_case

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fsdp_sharded_mixed_flatparameter_gb300 import build, zero_shard
    build.build()
    zero_shard.lib()


SHAPES = {
    # tiles across tensor boundaries, tensors without grad, misaligned sources: the staged tiles
    "ragged": (lambda: list(W.ragged_numels(300, seed=17, max_log2=14)), [0, 2, 7], (5,)),
    # whole tiles inside one tensor: the vector tiles, co-aligned (offset 0) and realigned (offset 3)
    "llama": (lambda: list(W.llama_numels(2, 256, 688, 1000)), [0, 0, 3], (5,)),
    # more than 1,024 tensors: AdamW searches the table once per four 2048-element parts
    "ragged_long": (lambda: list(W.ragged_numels(1500, seed=14, max_log2=14)), [0, 1, 3, 8, 5], (3, 700)),
}


def _acc(n, seed, off):
    g = torch.Generator().manual_seed(seed)
    return Guarded(n, torch.float32, off, torch.randn(n, generator=g) * 3e-3)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("shape", list(SHAPES))
def test_norm_of_sum_equals_accumulating_pass(dtype, shape):
    """accumulate == 2 writes the partials the accumulating pass with the fused norm writes,
    raises the same non-finite flag, and leaves the accumulator bit for bit as it was."""
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    numels_fn, offs, nulls = SHAPES[shape]
    numels = numels_fn()
    host, dev = _table_case(numels, dtype, null=nulls, seed=4, elem_offsets=offs)
    table, total = zs.zero_tensor_table(dev, numels)
    d_table = zs.device_table(table, len(numels), DEV)
    tdt = W.torch_dtype(dtype)
    for world, rank, acc_off in ((1, 0, 0), (3, 2, 0), (3, 1, 3)):
        s, e = oracle.shard_range(total, world, rank)
        n = e - s
        A = _acc(n, world + rank, acc_off)  # read only
        B = Guarded(n, torch.float32, 0, A.t.clone())  # updated by the reference pass
        nb = zs.zero_grad_sqnorm_workspace_bytes(n)
        ws_a = torch.full((nb,), 0x11, dtype=torch.uint8, device=DEV)
        ws_b = torch.full((nb,), 0x22, dtype=torch.uint8, device=DEV)
        flags = torch.zeros(2, dtype=torch.int32, device=DEV)
        zs.zero_flatten_cast(d_table, len(numels), total, tdt, s, e, 0.125, zs.NORM_OF_SUM, A.t, flags[0:1], ws_a)
        zs.zero_flatten_cast(d_table, len(numels), total, tdt, s, e, 0.125, True, B.t, flags[1:2], ws_b)
        torch.cuda.synchronize()
        A.check_guards()
        assert torch.equal(A.base.view(torch.uint8), A.snap.view(torch.uint8)), "the accumulator was written"
        assert torch.equal(ws_a, ws_b), (world, rank, acc_off)
        assert flags.tolist() == [0, 0]
    # a non-finite grad raises the flag in both passes, and both partials see it
    if dtype != "f32":
        big = next(d for d in dev if d is not None and d.numel() >= 2)
        big[1] = float("inf")
        s, e = 0, total
        A = _acc(total, 9, 0)
        B = Guarded(total, torch.float32, 0, A.t.clone())
        nb = zs.zero_grad_sqnorm_workspace_bytes(total)
        ws_a = torch.zeros(nb, dtype=torch.uint8, device=DEV)
        ws_b = torch.ones(nb, dtype=torch.uint8, device=DEV)
        flags = torch.zeros(2, dtype=torch.int32, device=DEV)
        zs.zero_flatten_cast(d_table, len(numels), total, tdt, s, e, 0.5, zs.NORM_OF_SUM, A.t, flags[0:1], ws_a)
        zs.zero_flatten_cast(d_table, len(numels), total, tdt, s, e, 0.5, True, B.t, flags[1:2], ws_b)
        torch.cuda.synchronize()
        assert flags.tolist() == [1, 1] and torch.equal(ws_a, ws_b)
        assert not math.isfinite(float(ws_a.view(torch.float64).sum()))


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("shape", list(SHAPES))
def test_adamw_tensors_with_acc_equals_accumulate_then_adamw(dtype, shape):
    """AdamW with d_acc equals the accumulating flatten pass + AdamW bit for bit: shards that
    start anywhere, state, accumulator and low-precision copy at their own alignments."""
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    numels_fn, offs, nulls = SHAPES[shape]
    numels = numels_fn()
    host, dev = _table_case(numels, dtype, null=nulls, seed=21, elem_offsets=offs)
    table, total = zs.zero_tensor_table(dev, numels)
    d_table = zs.device_table(table, len(numels), DEV)
    tdt = W.torch_dtype(dtype)
    for world, rank, state_off, acc_off, lowp_dt, lowp_off in ((1, 0, 0, 0, torch.bfloat16, 0),
                                                              (4, 2, 0, 5, torch.float16, 3),
                                                              (5, 1, 3, 3, torch.bfloat16, 1),
                                                              (7, 6, 0, 0, None, 0)):
        s, e = oracle.shard_range(total, world, rank)
        n = e - s
        gen = torch.Generator().manual_seed(world * 10 + rank)
        p0 = torch.randn(n, generator=gen) * 0.02
        A = [Guarded(n, torch.float32, state_off, x) for x in (p0, torch.zeros(n), torch.zeros(n))]
        B = [Guarded(n, torch.float32, 0, x) for x in (p0, torch.zeros(n), torch.zeros(n))]
        LA = Guarded(n, lowp_dt, lowp_off) if lowp_dt is not None else None
        LB = Guarded(n, lowp_dt, 0) if lowp_dt is not None else None
        for t in range(1, 4):
            acc = _acc(n, 100 * t + world, acc_off)
            grad = acc.t.clone()
            coef = float(np.float32(0.25 + 0.2 * t))
            clip = norm_result_tensor(DEV, norm=1.0 / coef, coef=coef)
            scale = 0.125 if t == 2 else 0.5
            zs.zero_adamw_step_tensors(A[0].t, A[1].t, A[2].t, d_table, len(numels), total, tdt, s, scale,
                                       None if LA is None else LA.t, 1e-3, 0.9, 0.95, 1e-8, 0.1, t, clip, acc=acc.t)
            zs.zero_flatten_cast(d_table, len(numels), total, tdt, s, e, scale, True, grad)
            zs.zero_adamw_step(B[0].t, B[1].t, B[2].t, grad, None if LB is None else LB.t, 1e-3, 0.9, 0.95,
                               1e-8, 0.1, t, clip)
            torch.cuda.synchronize()
            assert torch.equal(acc.base.view(torch.uint8), acc.snap.view(torch.uint8)), "the accumulator was written"
        for a, b in zip(A, B):
            a.check_guards()
            assert bits_equal_f32(raw(a.t), raw(b.t)), (world, rank, state_off, acc_off)
        if LA is not None:
            LA.check_guards()
            assert np.array_equal(raw(LA.t), raw(LB.t))


@pytest.mark.parametrize("grad_range", ["shard", "full"])
def test_step_tensors_accumulated_matches_oracle_and_materialized_step(grad_range):
    """Three micro-batches of per-tensor grads: two flattened, the last read in place.  The
    optimizer's state equals the materialized path's bit for bit, and the oracle's whenever
    the binary32 clip coefficients agree (ZeRO-1 full-range norm and a shard-only one)."""
    from fsdp_sharded_mixed_flatparameter_gb300 import FlatShardAdamW
    wl = W.small_llama(layers=2, hidden=256, mlp=688, vocab=1000, world_size=3, rank=1, max_norm=0.02,
                       micro_batches=3)
    s, e = oracle.shard_range(wl.total, wl.world_size, wl.rank)
    glo, ghi = (0, wl.total) if grad_range == "full" else (s, e)
    M = wl.micro_batches
    master = W.master_init(wl, s, e)
    kw = dict(world_size=wl.world_size, rank=wl.rank, lr=wl.lr, betas=wl.betas, eps=wl.eps,
              weight_decay=wl.weight_decay, max_norm=wl.max_norm, device=DEV, grad_range=grad_range)
    direct = FlatShardAdamW(wl.numels, master=master.to(DEV), **kw)
    mat = FlatShardAdamW(wl.numels, master=master.to(DEV), **kw)
    st = oracle.new_state(raw(master))
    for t in range(1, 5):
        tgs = [W.tensor_grads(wl, t, j, device="cpu") for j in range(M)]
        dgrads = [[x.to(DEV) for x in tg.tensors] for tg in tgs]
        for j in range(M - 1):
            direct.flatten(dgrads[j], accumulate=j > 0, scale=1.0 / M)
        r1 = direct.step_tensors(dgrads[-1], scale=1.0 / M, accumulated=True)
        for j in range(M):
            mat.flatten(dgrads[j], accumulate=j > 0, scale=1.0 / M, fuse_norm=j == M - 1)
        r2 = mat.step()
        g = np.zeros(ghi - glo, np.float32)
        for j in range(M):
            oracle.flatten([raw(x) for x in tgs[j].tensors], wl.numels, "bf16", glo, ghi, 1.0 / M, g,
                           accumulate=j > 0)
        cr = oracle.clip(oracle.sqnorm(g), 0.0, wl.max_norm)
        st.t += 1
        sc = oracle.adamw_scalars(wl.lr, wl.betas[0], wl.betas[1], wl.eps, wl.weight_decay, st.t)
        oracle.adamw(st.p, st.m, st.v, np.ascontiguousarray(g[s - glo:e - glo]), sc, cr.coef, st.lowp, "bf16")
        assert r1 == r2 and abs(r1.norm - cr.norm) <= 1e-12 * cr.norm and cr.coef < 1.0
        for a, b, ref in ((direct.master, mat.master, st.p), (direct.exp_avg, mat.exp_avg, st.m),
                          (direct.exp_avg_sq, mat.exp_avg_sq, st.v)):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))
            if r1.clip_coef == cr.coef:
                assert bits_equal_f32(raw(a), ref)
        assert torch.equal(direct.lowp.view(torch.int16), mat.lowp.view(torch.int16))
        if r1.clip_coef == cr.coef:
            assert np.array_equal(raw(direct.lowp), st.lowp)
        assert direct.t == mat.t == st.t


@pytest.mark.parametrize("M", [1, 3])
@pytest.mark.parametrize("graph", [False, True])
def test_step_flat_matches_accum_path(M, graph):
    """Flat fp16 shard grads (ZeRO-3): step_flat with the last micro-batch read in place
    equals accum + step bit for bit, eager and replayed from a CUDA graph, and a
    non-finite last micro-batch skips the step on both."""
    from fsdp_sharded_mixed_flatparameter_gb300 import FlatShardAdamW
    wl = W.llama13b_zero3().with_(numels=tuple(W.llama_numels(2, 320, 864, 1500)), max_norm=0.05,
                                  micro_batches=M)
    s, e = oracle.shard_range(wl.total, wl.world_size, wl.rank)
    master = W.master_init(wl, s, e, device=DEV)
    kw = dict(world_size=wl.world_size, rank=wl.rank, lr=wl.lr, betas=wl.betas, eps=wl.eps,
              weight_decay=wl.weight_decay, max_norm=wl.max_norm, device=DEV, lowp_dtype=torch.float16)
    direct = FlatShardAdamW(wl.numels, master=master.clone(), capturable=graph, grad_buffer=M > 1, **kw)
    mat = FlatShardAdamW(wl.numels, master=master.clone(), capturable=graph, **kw)
    srcs = [torch.empty(e - s, dtype=torch.float16, device=DEV) for _ in range(M)]

    def run_direct():
        for j in range(M - 1):
            direct.accum(srcs[j], accumulate=j > 0, scale=1.0 / M)
        direct.launch_step_flat(srcs[-1], scale=1.0 / M, accumulated=M > 1)

    def run_mat():
        for j in range(M):
            mat.accum(srcs[j], accumulate=j > 0, scale=1.0 / M, fuse_norm=j == M - 1)
        mat.launch_step()

    graphs = None
    for t in range(1, 6):
        for j in range(M):
            W.flat_grads(wl, t, j, s, e, device=DEV, out=srcs[j])
        if t == 4:
            srcs[-1][777] = float("nan")  # the step is skipped on both paths
        if graph:
            if graphs is None:
                direct.device_flat_table(srcs[-1])
                torch.cuda.synchronize()
                graphs = (torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph())
                with torch.cuda.graph(graphs[0]):
                    run_direct()
                with torch.cuda.graph(graphs[1]):
                    run_mat()
            graphs[0].replay()
            graphs[1].replay()
        else:
            run_direct()
            run_mat()
        r1, r2 = direct.finish_step(), mat.finish_step()
        assert repr(r1) == repr(r2) and r1.finite == (t != 4)
        for a, b in ((direct.master, mat.master), (direct.exp_avg, mat.exp_avg), (direct.exp_avg_sq, mat.exp_avg_sq),
                     (direct.lowp, mat.lowp)):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), t
        assert direct.t == mat.t == (t if t < 4 else t - 1)
    if M == 1:
        assert direct.grad.numel() == 0


def test_accumulated_needs_the_grad_buffer():
    from fsdp_sharded_mixed_flatparameter_gb300 import FlatShardAdamW
    opt = FlatShardAdamW([100, 28], device=DEV, grad_buffer=False)
    grads = [torch.zeros(100, dtype=torch.bfloat16, device=DEV), torch.zeros(28, dtype=torch.bfloat16, device=DEV)]
    with pytest.raises(ValueError):
        opt.step_tensors(grads, accumulated=True)
    with pytest.raises(ValueError):
        opt.step_flat(torch.zeros(127, dtype=torch.bfloat16, device=DEV))  # not the grad range's size
