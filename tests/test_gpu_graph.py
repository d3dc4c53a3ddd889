"""Graph-capturable steps: the step count and the skip decision on the device.

The device step state must give exactly the host path's scalars and skip
policy, and a whole step captured once in a CUDA graph and replayed over
grads rewritten in place must match the oracle step by step like the
host-driven steps do.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _configs import run_workload
from _helpers import bits_equal_f32, raw

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fsdp_sharded_mixed_flatparameter_gb300 import build, zero_shard
    build.build()
    zero_shard.lib()
    torch.cuda.init()


def _norm_result(finite: bool, coef: float = 0.5) -> torch.Tensor:
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    r = zs.zero_norm_result(4.0, 2.0, coef, 1 if finite else 0)
    return torch.frombuffer(bytearray(bytes(memoryview(r))), dtype=torch.uint8).to(DEV)


def test_prepare_device_scalars_equal_host_scalars():
    """zero_adamw_prepare_device: step += 1 and the host path's scalar bits for a finite
    norm; nothing for a non-finite norm; ZERO_EINVAL status for bad hyper-parameters."""
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    hps = [(3e-4, 0.9, 0.95, 1e-8, 0.1), (1e-4, 0.9, 0.999, 1e-8, 0.0), (6e-4, 0.0, 0.98, 1e-6, 0.05)]
    ok, bad = _norm_result(True), _norm_result(False)
    for hp in hps:
        d_hp = zs.device_hparams(*hp, DEV)
        st = zs.new_adamw_device_state(DEV)
        for t in list(range(1, 301)) + [10 ** 6, 2 ** 40]:
            if t > 300:
                st = zs.new_adamw_device_state(DEV, t - 1)
            zs.zero_adamw_prepare_device(d_hp, ok if t % 2 else None, st)
            d = zs.decode_adamw_device_state(st)
            assert d.step == t and d.apply and d.status == 0
            want = zs.zero_adamw_scalars(*hp, t)
            assert np.array_equal(d.scalars.view(np.uint32), want.view(np.uint32)), (hp, t)
            assert np.array_equal(want.view(np.uint32), oracle.adamw_scalars(*hp, t).view(np.uint32)), (hp, t)
        zs.zero_adamw_prepare_device(d_hp, bad, st)
        d = zs.decode_adamw_device_state(st)
        assert d.step == 2 ** 40 and not d.apply and d.status == 0
    st = zs.new_adamw_device_state(DEV, 5)
    for badhp in [(1e-3, 1.0, 0.999, 1e-8, 0.0), (-1.0, 0.9, 0.999, 1e-8, 0.0), (1e-3, 0.9, 0.999, 0.0, 0.0),
                  (math.nan, 0.9, 0.999, 1e-8, 0.0)]:
        zs.zero_adamw_prepare_device(zs.device_hparams(*badhp, DEV), ok, st)
        d = zs.decode_adamw_device_state(st)
        assert d.step == 5 and not d.apply and d.status == zs.ZERO_EINVAL, badhp


def test_device_state_step_skips_and_matches_host_step():
    """zero_adamw_step_device / _tensors_device against zero_adamw_step / _tensors with
    the host counter: bit-identical state, including a skipped (non-finite) step that
    changes nothing and does not advance the device count."""
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    n = 100_003
    g = torch.Generator().manual_seed(5)
    grad = (torch.randn(n, generator=g) * 1e-3).to(DEV)
    init = (torch.randn(n, generator=g) * 0.02).to(DEV)
    hp = (1e-3, 0.9, 0.95, 1e-8, 0.1)
    A = [init.clone(), torch.zeros(n, device=DEV), torch.zeros(n, device=DEV)]
    B = [init.clone(), torch.zeros(n, device=DEV), torch.zeros(n, device=DEV)]
    LA, LB = torch.empty(n, dtype=torch.bfloat16, device=DEV), torch.empty(n, dtype=torch.bfloat16, device=DEV)
    d_hp, st = zs.device_hparams(*hp, DEV), zs.new_adamw_device_state(DEV)
    ok, bad = _norm_result(True, 0.75), _norm_result(False)
    t = 0
    for k, clip in enumerate([ok, ok, bad, ok, None]):
        finite = clip is not bad
        if finite:
            t += 1
            zs.zero_adamw_step(*A, grad, LA, *hp, t, clip)
        zs.zero_adamw_prepare_device(d_hp, clip, st)
        zs.zero_adamw_step_device(*B, grad, LB, st, clip)
        torch.cuda.synchronize()
        for a, b in zip(A, B):
            assert bits_equal_f32(raw(a), raw(b)), k
        assert torch.equal(LA.view(torch.int16), LB.view(torch.int16))
        assert zs.decode_adamw_device_state(st).step == t
    # the table-reading variant, misaligned state buffers (staged path) included
    numels = [5000, 0, 70001, 25002]
    gt = [None if m == 0 else (torch.randn(m, generator=g) * 1e-3).to(torch.bfloat16).to(DEV) for m in numels]
    table, total = zs.zero_tensor_table(gt, numels)
    d_table = zs.device_table(table, len(numels), DEV)
    for lo, off in ((0, 0), (3, 1)):  # off 1: state 4 bytes past a 32-byte boundary (staged path)
        m = total - lo

        def fresh():
            bufs = [torch.zeros(m + off, device=DEV) for _ in range(3)]
            bufs[0][off:].copy_(init[:m])
            return [b[off:] for b in bufs]
        A2, B2 = fresh(), fresh()
        st2 = zs.new_adamw_device_state(DEV, 7)
        for clip in (ok, bad, ok):
            if clip is not bad:
                zs.zero_adamw_step_tensors(*A2, d_table, len(numels), total, torch.bfloat16, lo, 0.5, None, *hp,
                                           zs.decode_adamw_device_state(st2).step + 1, clip)
            zs.zero_adamw_prepare_device(d_hp, clip, st2)
            zs.zero_adamw_step_tensors_device(*B2, d_table, len(numels), total, torch.bfloat16, lo, 0.5, None, st2,
                                              clip)
            torch.cuda.synchronize()
            for a, b in zip(A2, B2):
                assert bits_equal_f32(raw(a), raw(b)), lo


@pytest.mark.parametrize("name,kw", [
    ("tiny", dict(steps=3)),
    ("gpt2", dict(steps=4)),
    ("ragged_small", dict(steps=3)),
    ("llama13b_small", dict(steps=3)),
    ("llama_direct", dict(steps=3, direct=True)),
    # the last of 8 micro-batches read in place (per-tensor grads, ZeRO-1 full-buffer norm)
    ("gpt2_direct", dict(steps=3, direct=True)),
    # a table of more than 1,024 tensors (AdamW searches it once per four parts), 2 micro-batches
    ("ragged_long_direct", dict(steps=3, direct=True)),
])
def test_graph_replayed_steps_match_oracle(name, kw):
    """Whole steps (all micro-batches' grad passes with the fused norm, finalize, prepare,
    AdamW) captured once in a CUDA graph and replayed every step: the oracle's state
    after every step, and the device step count equals the oracle's."""
    wl = {"tiny": W.tiny(),
          "gpt2": W.gpt2_zero1(),
          "ragged_small": W.small_ragged(n_tensors=800, world_size=4, rank=2),
          "llama13b_small": W.llama13b_zero3().with_(numels=tuple(W.llama_numels(2, 512, 1376, 3200))),
          "llama_direct": W.small_llama(layers=2, hidden=256, mlp=688, vocab=1000, world_size=3, rank=1,
                                        max_norm=0.02),
          "gpt2_direct": W.gpt2_zero1(),
          "ragged_long_direct": W.small_ragged(n_tensors=1500, max_log2=13, world_size=4, rank=2,
                                               micro_batches=2)}[name]
    rep = run_workload(wl, graph=True, **kw)
    assert len(rep.steps) == kw["steps"]


def test_graph_replay_skips_a_nonfinite_step():
    """A NaN grad written into the captured grads' storage before one replay: that
    replay changes no state and does not advance the device step count; the next
    replays continue exactly like host-driven steps that skip the same step."""
    from fsdp_sharded_mixed_flatparameter_gb300 import FlatShardAdamW
    wl = W.small_llama(layers=2, hidden=256, mlp=688, vocab=1000, world_size=2, rank=1, max_norm=0.05)
    s, e = oracle.shard_range(wl.total, wl.world_size, wl.rank)
    master = W.master_init(wl, s, e, device=DEV)
    kw = dict(world_size=wl.world_size, rank=wl.rank, lr=wl.lr, betas=wl.betas, eps=wl.eps,
              weight_decay=wl.weight_decay, max_norm=wl.max_norm, device=DEV)
    A = FlatShardAdamW(wl.numels, master=master.clone(), **kw)
    B = FlatShardAdamW(wl.numels, master=master.clone(), capturable=True, **kw)
    tg = W.tensor_grads(wl, 1, 0, device=DEV)
    B.register_grads(tg.tensors)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        B.flatten(accumulate=False, scale=0.5, fuse_norm=True)
        B.launch_step()
    for t in range(1, 6):
        W.tensor_grads(wl, t, 0, device=DEV, storage=tg.storage)
        if t == 3:
            tg.tensors[-1][17] = math.nan  # lm_head: inside rank 1's shard
        A.flatten(tg.tensors, accumulate=False, scale=0.5, fuse_norm=True)
        ra = A.step()
        graph.replay()
        rb = B.finish_step()
        assert ra.finite == rb.finite == (t != 3)
        assert A.t == B.t == (t if t < 3 else t - 1)
        for nm in ("master", "exp_avg", "exp_avg_sq"):
            assert bits_equal_f32(raw(getattr(A, nm)), raw(getattr(B, nm))), (t, nm)
        assert torch.equal(A.lowp.view(torch.int16), B.lowp.view(torch.int16))


def test_capturable_state_dict_round_trip_and_lr_change():
    """t lives on the device: state_dict reads it, load_state_dict writes it; changing lr
    (set_hparams or plain assignment) rewrites the device hyper-parameters that an already
    captured graph reads."""
    from fsdp_sharded_mixed_flatparameter_gb300 import FlatShardAdamW
    wl = W.small_llama(layers=1, hidden=128, mlp=344, vocab=301, max_norm=math.inf)
    kw = dict(lr=1e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1, device=DEV)
    master = W.master_init(wl, 0, wl.total, device=DEV)
    A = FlatShardAdamW(wl.numels, master=master.clone(), **kw)
    B = FlatShardAdamW(wl.numels, master=master.clone(), capturable=True, **kw)
    tg = W.tensor_grads(wl, 1, 0, device=DEV)
    B.register_grads(tg.tensors)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        B.launch_step_tensors()
    for t in range(1, 4):
        if t == 3:
            A.set_hparams(lr=2e-4)
            B.lr = 2e-4  # plain assignment reaches the device copy the graph reads
        A.step_tensors(tg.tensors)
        graph.replay()
        B.finish_step()
        assert bits_equal_f32(raw(A.master), raw(B.master)), t
    sd = B.state_dict()
    assert sd["t"] == 3
    C = FlatShardAdamW(wl.numels, capturable=True, **kw)
    C.set_hparams(lr=2e-4)
    C.load_state_dict(sd)
    assert C.t == 3
    A.step_tensors(tg.tensors)
    C.step_tensors(tg.tensors)
    assert A.t == C.t == 4 and bits_equal_f32(raw(A.master), raw(C.master))
