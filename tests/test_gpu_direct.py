"""The direct path of a step without micro-batch accumulation: a norm-only
pass and an AdamW that both read the per-tensor grads through the
FlatParameter table (no fp32 flat grad written).  It must be bit-identical to
flatten + norm + AdamW, and therefore to the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _helpers import assert_lowp_ulp, bits_equal_f32, norm_result_tensor, raw
from test_gpu_kernels import Guarded, _table_case

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fsdp_sharded_mixed_flatparameter_gb300 import build, zero_shard
    build.build()
    zero_shard.lib()


CASES = [
    ("ragged", lambda: list(W.ragged_numels(250, seed=13, max_log2=13)), [0, 1, 3, 8, 5], (3,)),
    # more than 1,024 tensors: AdamW searches the table once per four 2048-element parts
    ("ragged_long", lambda: list(W.ragged_numels(1500, seed=14, max_log2=14)), [0, 1, 3, 8, 5], (3, 700)),
    ("llama", lambda: list(W.llama_numels(1, 256, 688, 1000)), [0], ()),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_adamw_tensors_equals_flatten_then_adamw(case, dtype):
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    _, numels_fn, offs, nulls = case
    numels = numels_fn()
    host, dev = _table_case(numels, dtype, null=nulls, seed=21, elem_offsets=offs)
    table, total = zs.zero_tensor_table(dev, numels)
    d_table = zs.device_table(table, len(numels), DEV)
    tdt = W.torch_dtype(dtype)
    for world, rank, state_off, lowp_dt, lowp_off in ((1, 0, 0, torch.bfloat16, 0), (4, 2, 0, torch.float16, 3),
                                                      (5, 1, 3, torch.bfloat16, 1), (7, 6, 0, None, 0)):
        s, e = oracle.shard_range(total, world, rank)
        n = e - s
        gen = torch.Generator().manual_seed(world * 10 + rank)
        p0 = torch.randn(n, generator=gen) * 0.02
        A = [Guarded(n, torch.float32, state_off, x) for x in (p0, torch.zeros(n), torch.zeros(n))]
        B = [Guarded(n, torch.float32, 0, x) for x in (p0, torch.zeros(n), torch.zeros(n))]
        LA = Guarded(n, lowp_dt, lowp_off) if lowp_dt is not None else None
        LB = Guarded(n, lowp_dt, 0) if lowp_dt is not None else None
        grad = torch.empty(n, device=DEV)
        for t in range(1, 4):
            coef = float(np.float32(0.25 + 0.2 * t))
            clip = norm_result_tensor(DEV, norm=1.0 / coef, coef=coef)
            scale = 0.5 if t == 2 else 1.0
            zs.zero_adamw_step_tensors(A[0].t, A[1].t, A[2].t, d_table, len(numels), total, tdt, s, scale,
                                       None if LA is None else LA.t, 1e-3, 0.9, 0.95, 1e-8, 0.1, t, clip)
            zs.zero_flatten_cast(d_table, len(numels), total, tdt, s, e, scale, False, grad)
            zs.zero_adamw_step(B[0].t, B[1].t, B[2].t, grad, None if LB is None else LB.t, 1e-3, 0.9, 0.95,
                               1e-8, 0.1, t, clip)
        torch.cuda.synchronize()
        for a, b in zip(A, B):
            a.check_guards()
            assert bits_equal_f32(raw(a.t), raw(b.t)), (world, rank, state_off)
        if LA is not None:
            LA.check_guards()
            assert np.array_equal(raw(LA.t), raw(LB.t))


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("shape", ["ragged", "llama", "llama_large"])
def test_norm_only_flatten_equals_fused_flatten(dtype, shape):
    """The norm-only pass's partials equal the writing pass's, on both of its kernels: lists of
    small tensors (ragged, and a small Llama list: the tiled kernel without stores, staged and
    vector tiles) and of large ones (a Llama list with tensors of millions of elements: K1n,
    whole 32768-element tiles inside one tensor on the vector path, tensor boundaries element
    by element), every grad dtype, a misaligned start or not."""
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    if shape == "ragged":
        numels = list(W.ragged_numels(300, seed=17, max_log2=14))
        host, dev = _table_case(numels, dtype, null=(5,), seed=4, elem_offsets=[0, 2, 7])
    elif shape == "llama":
        numels = list(W.llama_numels(2, 256, 688, 1000))
        host, dev = _table_case(numels, dtype, null=(5,), seed=4, elem_offsets=[0, 0, 3])
    else:
        numels = list(W.llama_numels(1, 1024, 2752, 2000))
        assert sum(numels) // len(numels) > 16 * 32768  # the K1n side of the kernel choice
        host, dev = _table_case(numels, dtype, null=(5,), seed=4, elem_offsets=[0, 0, 3])
    table, total = zs.zero_tensor_table(dev, numels)
    d_table = zs.device_table(table, len(numels), DEV)
    for world, rank in ((1, 0), (3, 2)):
        s, e = oracle.shard_range(total, world, rank)
        nb = zs.zero_grad_sqnorm_workspace_bytes(e - s)
        ws_a = torch.full((nb,), 0x11, dtype=torch.uint8, device=DEV)
        ws_b = torch.full((nb,), 0x22, dtype=torch.uint8, device=DEV)
        dst = torch.empty(e - s, device=DEV)
        zs.zero_flatten_cast(d_table, len(numels), total, W.torch_dtype(dtype), s, e, 0.25, False, None, norm_ws=ws_a)
        zs.zero_flatten_cast(d_table, len(numels), total, W.torch_dtype(dtype), s, e, 0.25, False, dst, norm_ws=ws_b)
        assert torch.equal(ws_a, ws_b)
    with pytest.raises(zs.ZeroError):  # norm-only cannot accumulate
        zs.zero_flatten_cast(d_table, len(numels), total, W.torch_dtype(dtype), s, e, 0.25, True, None, norm_ws=ws_a)


def test_step_tensors_matches_oracle_and_materialized_step():
    from fsdp_sharded_mixed_flatparameter_gb300 import FlatShardAdamW
    wl = W.small_llama(layers=2, hidden=256, mlp=688, vocab=1000, world_size=3, rank=1, max_norm=0.02)
    s, e = oracle.shard_range(wl.total, wl.world_size, wl.rank)
    master = W.master_init(wl, s, e)
    kw = dict(world_size=wl.world_size, rank=wl.rank, lr=wl.lr, betas=wl.betas, eps=wl.eps,
              weight_decay=wl.weight_decay, max_norm=wl.max_norm, device=DEV)
    direct = FlatShardAdamW(wl.numels, master=master.to(DEV), grad_buffer=False, **kw)
    mat = FlatShardAdamW(wl.numels, master=master.to(DEV), **kw)
    st = oracle.new_state(raw(master))
    for t in range(1, 5):
        tg = W.tensor_grads(wl, t, 0, device="cpu")
        dgrads = [x.to(DEV) for x in tg.tensors]
        r1 = direct.step_tensors(dgrads)
        mat.flatten(dgrads, accumulate=False, fuse_norm=True)
        r2 = mat.step()
        g = np.zeros(e - s, np.float32)
        oracle.flatten([raw(x) for x in tg.tensors], wl.numels, "bf16", s, e, 1.0, g, accumulate=False)
        cr = oracle.step_reference(st, g, lr=wl.lr, betas=wl.betas, eps=wl.eps, wd=wl.weight_decay,
                                   max_norm=wl.max_norm)
        assert r1 == r2 and abs(r1.norm - cr.norm) <= 1e-12 * cr.norm and cr.coef < 1.0
        for a, b, ref in ((direct.master, mat.master, st.p), (direct.exp_avg, mat.exp_avg, st.m),
                          (direct.exp_avg_sq, mat.exp_avg_sq, st.v)):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))
            if r1.clip_coef == cr.coef:
                assert bits_equal_f32(raw(a), ref)
        assert direct.t == mat.t == st.t
    assert direct.grad.numel() == 0
