"""Four ZeRO-2/3 ranks emulated one after another on one GPU (no concurrent
ranks, no collective): phase 1 runs every rank's flatten with the fused norm
and its local sum of squares, the rank-order vector of those values stands in
for the all-gather, phase 2 runs every rank's combine + AdamW.  The result is
checked against the oracle's global-norm step over the whole flat buffer."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _helpers import RTOL_NORM, assert_close_f32, bits_equal_f32, raw

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fsdp_sharded_mixed_flatparameter_gb300 import build, zero_shard
    build.build()
    zero_shard.lib()


def test_combine_matches_rank_order_sum():
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    vals = [3.25, 1e-3, 7.0, 0.0, 2.5e2]
    out = zs.new_norm_result(DEV)
    zs.zero_grad_sqnorm_combine(torch.tensor(vals, dtype=torch.float64, device=DEV), 1.0, out)
    r = zs.decode_norm_result(out)
    total = 0.0
    for v in vals:
        total += v
    cr = oracle.clip(total, 0.0, 1.0)
    assert r.sqnorm == total and r.norm == cr.norm and r.clip_coef == cr.coef and r.finite
    zs.zero_grad_sqnorm_combine(torch.tensor([1.0, float("inf")], dtype=torch.float64, device=DEV), 1.0, out)
    assert not zs.decode_norm_result(out).finite


def test_four_ranks_global_norm_step():
    from fsdp_sharded_mixed_flatparameter_gb300 import FlatShardAdamW
    world = 4
    base = W.small_ragged(n_tensors=500, max_log2=13, world_size=world, rank=0, max_norm=0.5)
    steps = 3
    opts, states = [], []
    for r in range(world):
        s, e = oracle.shard_range(base.total, world, r)
        master = W.master_init(base, s, e)  # drawn once (CPU), copied to the GPU side
        opts.append(FlatShardAdamW(base.numels, world_size=world, rank=r, lr=base.lr, betas=base.betas, eps=base.eps,
                                   weight_decay=base.weight_decay, max_norm=base.max_norm, device=DEV,
                                   master=master.to(DEV)))
        states.append(oracle.new_state(raw(master)))
    for t in range(1, steps + 1):
        tg = W.tensor_grads(base, t, 0, device=DEV)
        # phase 1: every rank's flatten (fused norm) and local sum of squares
        locals_ = []
        for opt in opts:
            opt.flatten(tg.tensors, accumulate=False, fuse_norm=True)
            locals_.append(opt.local_sqnorm())
        gathered = torch.cat(locals_)  # rank order: the all-gather's result
        # phase 2: combine + AdamW on every rank
        results = []
        for opt in opts:
            opt.launch_step(gathered_sqnorms=gathered)
            results.append(opt.finish_step())
        assert all(rr == results[0] for rr in results), "ranks disagree on the global norm"
        # oracle: global norm over the whole flat buffer, each rank's update on its shard
        full = np.zeros(base.total, np.float32)
        oracle.flatten([raw(x) for x in tg.tensors], base.numels, "bf16", 0, base.total, 1.0, full, False)
        cr = oracle.clip(oracle.sqnorm(full), 0.0, base.max_norm)
        assert abs(results[0].norm - cr.norm) <= 1e-12 * cr.norm
        assert cr.coef < 1.0
        for r, (opt, st) in enumerate(zip(opts, states)):
            s, e = oracle.shard_range(base.total, world, r)
            st.t += 1
            sc = oracle.adamw_scalars(base.lr, base.betas[0], base.betas[1], base.eps, base.weight_decay, st.t)
            oracle.adamw(st.p, st.m, st.v, np.ascontiguousarray(full[s:e]), sc, cr.coef, st.lowp)
            for got, ref in ((opt.master, st.p), (opt.exp_avg, st.m), (opt.exp_avg_sq, st.v)):
                assert_close_f32(raw(got), ref)
                if results[0].clip_coef == cr.coef:
                    assert bits_equal_f32(raw(got), ref)
            assert opt.t == st.t
