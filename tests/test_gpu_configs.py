"""The five workload configurations end to end on the GPU against the oracle.

tiny, GPT-2 ZeRO-1 and the ragged stress run at full size with the whole
shard compared after every step; Llama-7B and the Llama-13B ZeRO-3 shard run
at full size for their full step counts (5 and 20) with every grad in the
norm and a seeded sample of shard positions compared after every step, and
again on shape-preserving smaller lists with the whole shard compared.
"""
import math

import numpy as np
import pytest
import torch

import workloads as W
from _configs import run_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fsdp_sharded_mixed_flatparameter_gb300 import build, zero_shard
    build.build()
    zero_shard.lib()


def _summary(rep):
    exact = sum(s.exact for s in rep.steps)
    worst = max(abs(s.gpu_norm - s.ref_norm) / s.ref_norm for s in rep.steps)
    print(f"{rep.name}: n={rep.n} steps={len(rep.steps)} bit-exact steps={exact} worst norm rel err={worst:.2e}")
    for s in rep.steps:
        print(f"  step {s.t}: norm gpu={s.gpu_norm:.17g} oracle={s.ref_norm:.17g} "
              f"rel err={abs(s.gpu_norm - s.ref_norm) / s.ref_norm:.2e} coef gpu={s.gpu_coef!r} "
              f"oracle={s.ref_coef!r} bit-exact={s.exact}")


def test_tiny_full():
    rep = run_workload(W.tiny(), steps=3)
    assert len(rep.steps) == 3 and all(s.gpu_coef == 1.0 for s in rep.steps)
    _summary(rep)


def test_tiny_short_tail_shard():
    """tiny list, 8 ranks, rank 7: the short last shard [1,104,159, 1,261,891)."""
    wl = W.tiny().with_(world_size=8, rank=7, max_norm=0.5)
    rep = run_workload(wl, steps=3, fused=False)
    assert rep.n == 157732
    _summary(rep)


def test_gpt2_zero1_rank3_full():
    rep = run_workload(W.gpt2_zero1(), steps=10)
    assert all(s.ref_coef < 1.0 for s in rep.steps), "clipping expected to trigger"
    _summary(rep)


def test_ragged_rank2_full():
    rep = run_workload(W.ragged(), steps=5)
    assert all(s.ref_coef < 1.0 for s in rep.steps)
    _summary(rep)


def test_llama7b_full_size_all_steps_sampled():
    """The configuration as stated: 6,738,415,616 params, all 5 steps, every grad in the
    oracle's norm, a seeded sample of 1M shard positions compared after every step."""
    wl = W.llama7b()
    rep = run_workload(wl, steps=wl.steps, sample=1_000_000)
    assert rep.n == 6738415616 and len(rep.steps) == 5
    assert all(s.ref_coef < 1.0 for s in rep.steps), "clipping expected to trigger"
    _summary(rep)


def test_llama7b_full_size_direct_path_sampled():
    """The benchmark's direct path (norm pass + AdamW through the tensor table, no fp32 grad) at
    full size, for the configuration's 5 steps."""
    rep = run_workload(W.llama7b(), steps=W.llama7b().steps, sample=1_000_000, direct=True)
    assert rep.n == 6738415616 and len(rep.steps) == 5
    _summary(rep)


def test_ragged_direct_path_full():
    rep = run_workload(W.ragged(), steps=2, direct=True)
    _summary(rep)


def test_gpt2_zero1_rank3_direct_accum_full():
    """GPT-2 ZeRO-1 with the last of the 8 micro-batches never written: the norm over the whole
    124M buffer and AdamW both add it to the other seven's sum on the fly."""
    rep = run_workload(W.gpt2_zero1(), steps=10, direct=True)
    assert all(s.ref_coef < 1.0 for s in rep.steps)
    _summary(rep)


def test_llama13b_zero3_rank7_direct_accum_full_size_all_steps_sampled():
    """The 13B ZeRO-3 rank at full size, all 20 steps, the last fp16 micro-batch read in place
    by the norm pass and AdamW (step_flat)."""
    wl = W.llama13b_zero3()
    rep = run_workload(wl, steps=wl.steps, sample=1_000_000, direct=True)
    assert rep.n == 1626983040 and len(rep.steps) == 20
    assert all(s.ref_coef < 1.0 for s in rep.steps)
    _summary(rep)


def test_llama13b_zero3_shape_direct_accum_graph_all_steps():
    """The same path captured once in a CUDA graph and replayed for every step, whole shard
    compared."""
    wl = W.llama13b_zero3().with_(numels=tuple(W.llama_numels(5, 640, 1728, 4000)), max_norm=0.1)
    rep = run_workload(wl, steps=W.llama13b_zero3().steps, direct=True, graph=True)
    assert all(s.ref_coef < 1.0 for s in rep.steps)
    _summary(rep)


def test_llama7b_shape_all_steps():
    wl = W.small_llama(layers=4, hidden=512, mlp=1376, vocab=3200)
    rep = run_workload(wl, steps=W.llama7b().steps, fused=False)
    _summary(rep)


def test_llama13b_zero3_rank7_full_size_all_steps_sampled():
    """The configuration as stated: rank 7's 1,626,983,040 params, 8 fp16 micro-batches per
    step, all 20 steps, every grad in the oracle's norm, 1M shard positions compared."""
    wl = W.llama13b_zero3()
    rep = run_workload(wl, steps=wl.steps, sample=1_000_000)
    assert rep.n == 1626983040 and len(rep.steps) == 20
    assert all(s.ref_coef < 1.0 for s in rep.steps), "clipping expected to trigger"
    _summary(rep)


def test_llama13b_zero3_shape_all_steps():
    wl = W.llama13b_zero3().with_(numels=tuple(W.llama_numels(5, 640, 1728, 4000)), max_norm=0.1)
    rep = run_workload(wl, steps=W.llama13b_zero3().steps, fused=False)
    assert all(s.ref_coef < 1.0 for s in rep.steps)
    _summary(rep)


def test_llama13b_zero3_f16_chunk_full_size_sampled():
    """The ZeRO page's ZeRO-3 update at the 13B rank's full size: fp16 local parameter chunk,
    Adam without weight decay (section "ZeRO-3: 切分参数"), 8 fp16 micro-batches, 2 steps."""
    wl = W.llama13b_zero3_f16chunk()
    assert wl.lowp_dtype == "f16" and wl.weight_decay == 0.0
    rep = run_workload(wl, steps=2, sample=1_000_000)
    assert rep.n == 1626983040 and all(s.ref_coef < 1.0 for s in rep.steps)
    _summary(rep)


def test_llama13b_zero3_f16_chunk_shape_all_steps():
    wl = W.llama13b_zero3_f16chunk().with_(numels=tuple(W.llama_numels(5, 640, 1728, 4000)), max_norm=0.1)
    rep = run_workload(wl, steps=W.llama13b_zero3().steps, fused=False)
    _summary(rep)


def test_null_grads_and_fp16_writeback():
    """Tensors without grad read as zeros; the ZeRO-3 fp16 local chunk as the low-precision copy."""
    wl = W.small_ragged(n_tensors=400, null_grads=(0, 5, 399), lowp_dtype="f16", world_size=3, rank=1)
    rep = run_workload(wl, steps=3)
    _summary(rep)


def test_nonfinite_grad_skips_step():
    """An inf grad makes the norm non-finite: the step is skipped on both sides, t does not move."""
    from fsdp_sharded_mixed_flatparameter_gb300 import FlatShardAdamW
    dev = torch.device("cuda:0")
    opt = FlatShardAdamW([1000, 24], lr=1e-3, max_norm=1.0, device=dev,
                         master=torch.linspace(-1, 1, 1024, device=dev))
    g = [torch.full((1000,), 1e-3, device=dev, dtype=torch.bfloat16), torch.zeros(24, device=dev, dtype=torch.bfloat16)]
    opt.flatten(g, accumulate=False)
    assert opt.step().finite and opt.t == 1
    snap = [x.clone() for x in (opt.master, opt.exp_avg, opt.exp_avg_sq, opt.lowp)]
    g[1][3] = math.inf
    opt.found_nonfinite.zero_()
    opt.flatten(g, accumulate=False)
    r = opt.step()
    assert not r.finite and opt.t == 1 and opt.found_nonfinite.item() == 1
    for a, b in zip(snap, (opt.master, opt.exp_avg, opt.exp_avg_sq, opt.lowp)):
        assert torch.equal(a, b)


def test_resume_and_determinism_bit_identical():
    """Run 4 steps straight; run 2, save the state, restore it into a fresh optimizer and run 2 more:
    the two end states are bit-identical (and a repeated run reproduces the first bit for bit)."""
    from fsdp_sharded_mixed_flatparameter_gb300 import FlatShardAdamW
    dev = torch.device("cuda:0")
    wl = W.small_ragged(n_tensors=300, world_size=2, rank=1, max_norm=0.5)
    s, e = __import__("oracle").shard_range(wl.total, wl.world_size, wl.rank)
    master = W.master_init(wl, s, e)

    def make():
        return FlatShardAdamW(wl.numels, world_size=wl.world_size, rank=wl.rank, lr=wl.lr, betas=wl.betas,
                              eps=wl.eps, weight_decay=wl.weight_decay, max_norm=wl.max_norm, device=dev,
                              master=master.to(dev))

    def run(opt, steps):
        for t in steps:
            tg = W.tensor_grads(wl, t, 0, device="cpu")
            opt.flatten([None if x is None else x.to(dev) for x in tg.tensors], accumulate=False, fuse_norm=True)
            assert opt.step().finite

    a = make()
    run(a, range(1, 5))
    b = make()
    run(b, range(1, 3))
    sd = b.state_dict()
    c = make()
    c.load_state_dict(sd)
    run(c, range(3, 5))
    d = make()
    run(d, range(1, 5))
    for name in ("master", "exp_avg", "exp_avg_sq", "lowp"):
        x, y, z = getattr(a, name), getattr(c, name), getattr(d, name)
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8)), name
        assert torch.equal(x.view(torch.uint8), z.view(torch.uint8)), name
    assert a.t == c.t == d.t == 4


def test_empty_and_single_element_shards():
    """More ranks than elements: empty shards step as no-ops (t still advances: the
    norm of nothing is 0), one-element shards update like the oracle -- through the
    materialized step, the direct path, and the direct path with accumulation over
    per-tensor and flat grads (two halves: the same grad exactly)."""
    from fsdp_sharded_mixed_flatparameter_gb300 import FlatShardAdamW
    import oracle
    dev = torch.device("cuda:0")
    numels = [3, 2]
    g = [torch.tensor([1e-3, -2e-3, 3e-3], dtype=torch.bfloat16), torch.tensor([4e-3, 0.0], dtype=torch.bfloat16)]
    full = np.zeros(5, np.float32)
    oracle.flatten([x.view(torch.int16).numpy().view(np.uint16) for x in g], numels, "bf16", 0, 5, 1.0, full, False)
    modes = ("materialized", "direct", "direct_accumulated", "flat_accumulated")
    for rank in range(8):
        s, e = oracle.shard_range(5, 8, rank)
        p0 = torch.linspace(-1, 1, 5)[s:e].contiguous()
        opt = FlatShardAdamW(numels, world_size=8, rank=rank, lr=1e-2, max_norm=1.0, device=dev, master=p0.to(dev))
        dg = [x.to(dev) for x in g]
        flat = torch.cat(g)[s:e].contiguous().to(dev)
        for mode in modes:
            if mode == "direct":
                r = opt.step_tensors(dg)
            elif mode == "direct_accumulated":
                opt.flatten(dg, accumulate=False, scale=0.5)
                r = opt.step_tensors(dg, scale=0.5, accumulated=True)
            elif mode == "flat_accumulated":
                opt.accum(flat, accumulate=False, scale=0.5)
                r = opt.step_flat(flat, scale=0.5, accumulated=True)
            else:
                opt.flatten(dg, accumulate=False, fuse_norm=True)
                r = opt.step()
            assert r.finite
        st = oracle.new_state(p0.numpy())
        for _ in modes:
            oracle.step_reference(st, np.ascontiguousarray(full[s:e]), lr=1e-2, betas=(0.9, 0.999), eps=1e-8, wd=0.0,
                                  max_norm=1.0)
        assert opt.t == st.t == len(modes) and opt.n == e - s
        assert np.array_equal(opt.master.cpu().numpy(), st.p)


def test_registered_grads_match_passed_grads():
    """register_grads() once, then flatten()/step_tensors() without grads: same bits as passing them."""
    from fsdp_sharded_mixed_flatparameter_gb300 import FlatShardAdamW
    dev = torch.device("cuda:0")
    wl = W.small_ragged(n_tensors=800, world_size=2, rank=0, max_norm=0.5)
    s, e = __import__("oracle").shard_range(wl.total, 2, 0)
    master = W.master_init(wl, s, e)
    kw = dict(world_size=2, rank=0, lr=wl.lr, max_norm=wl.max_norm, device=dev)
    a = FlatShardAdamW(wl.numels, master=master.to(dev), **kw)
    b = FlatShardAdamW(wl.numels, master=master.to(dev), **kw)
    tg = W.tensor_grads(wl, 1, 0, device=dev)
    b.register_grads(tg.tensors)
    for t in range(2):
        a.flatten(tg.tensors, accumulate=False, fuse_norm=True)
        b.flatten(accumulate=False, fuse_norm=True)
        assert a.step() == b.step()
    assert a.step_tensors(tg.tensors) == b.step_tensors()
    for name in ("master", "exp_avg", "exp_avg_sq", "lowp"):
        assert torch.equal(getattr(a, name).view(torch.uint8), getattr(b, name).view(torch.uint8))


def test_cached_table_is_not_reused_for_other_sizes():
    """The optimizer's device tables are cached by grad address; a later list with a
    tensor at the same address but a different size or layout is checked again (and
    refused) instead of hitting the cache."""
    from fsdp_sharded_mixed_flatparameter_gb300 import FlatShardAdamW
    dev = torch.device("cuda:0")
    numels = [1000, 3000, 24]
    opt = FlatShardAdamW(numels, device=dev)
    grads = [torch.randn(n, device=dev).to(torch.bfloat16) for n in numels]
    opt.flatten(grads, accumulate=False)
    short = list(grads)
    short[1] = grads[1][:2999]            # same address, one element short
    with pytest.raises(ValueError):
        opt.flatten(short, accumulate=False)
    square = torch.randn(40, 25, device=dev).to(torch.bfloat16)
    opt2 = FlatShardAdamW([1000], device=dev)
    opt2.flatten([square.view(-1)], accumulate=False)
    with pytest.raises(ValueError):        # same address and size, not contiguous
        opt2.flatten([square.t()], accumulate=False)
