"""FlatShardAdamW's host logic without a GPU: shard bookkeeping, argument checks,
checkpoint validation, hyper-parameter properties, and no CPU fallback."""
import math

import pytest
import torch

import oracle
import workloads as W


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fsdp_sharded_mixed_flatparameter_gb300 import build
    build.build()


def _opt(**kw):
    from fsdp_sharded_mixed_flatparameter_gb300 import FlatShardAdamW
    numels = list(W.llama_numels(1, 128, 344, 301))
    base = dict(world_size=3, rank=1, lr=1e-3, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1, max_norm=1.0,
                device="cpu")
    base.update(kw)
    return FlatShardAdamW(numels, **base), numels


def test_shard_bookkeeping_matches_the_oracle():
    for grad_range in ("shard", "full"):
        opt, numels = _opt(grad_range=grad_range)
        total = sum(numels)
        assert opt.total == total
        assert (opt.start, opt.end) == oracle.shard_range(total, 3, 1)
        assert opt.n == opt.end - opt.start == opt.master.numel() == opt.exp_avg.numel() == opt.lowp.numel()
        want = (0, total) if grad_range == "full" else (opt.start, opt.end)
        assert (opt.glo, opt.ghi) == want and opt.grad.numel() == want[1] - want[0]
        assert opt.shard_grad().numel() == opt.n
        assert opt.resident_bytes() == 4 * (opt.grad.numel() + 3 * opt.n) + 2 * opt.n


def test_argument_checks():
    from fsdp_sharded_mixed_flatparameter_gb300 import FlatShardAdamW
    with pytest.raises(ValueError):
        _opt(grad_range="half")
    with pytest.raises(ValueError):
        _opt(master=torch.zeros(5))
    with pytest.raises(Exception):
        FlatShardAdamW([10, 20], world_size=2, rank=2, device="cpu")  # rank outside [0, world)


def test_state_dict_round_trip_and_shard_check():
    a, numels = _opt()
    a.master.normal_()
    a.exp_avg.uniform_()
    a.t = 7
    sd = a.state_dict()
    b, _ = _opt()
    b.load_state_dict(sd)
    assert b.t == 7 and torch.equal(b.master, a.master) and torch.equal(b.exp_avg, a.exp_avg)
    c, _ = _opt(rank=2)
    with pytest.raises(ValueError):
        c.load_state_dict(sd)  # another rank's shard


def test_hyper_parameter_properties():
    opt, _ = _opt()
    assert (opt.lr, opt.betas, opt.eps, opt.weight_decay) == (1e-3, (0.9, 0.95), 1e-8, 0.1)
    opt.lr = 2e-4
    opt.set_hparams(weight_decay=0.0)
    opt.betas = (0.8, 0.99)
    assert (opt.lr, opt.betas, opt.weight_decay) == (2e-4, (0.8, 0.99), 0.0)


def test_no_cpu_fallback():
    """The optimizer's buffers may live on the host, but nothing computes there: every
    kernel call refuses host tensors before anything runs."""
    opt, numels = _opt()
    grads = [torch.zeros(n, dtype=torch.bfloat16) for n in numels]
    with pytest.raises(ValueError):
        opt.flatten(grads, accumulate=False)
    with pytest.raises(ValueError):
        opt.step()
    with pytest.raises(ValueError):  # the direct path (last micro-batch read in place) likewise
        opt.step_tensors(grads, accumulated=True)
    with pytest.raises(ValueError):
        opt.step_flat(torch.zeros(opt.ghi - opt.glo, dtype=torch.bfloat16), accumulated=True)
    assert opt.t == 0 and math.isfinite(opt.lr)


def test_direct_path_argument_checks():
    """step_flat wants a 1-D grad over the grad range; the accumulated direct path wants the
    grad buffer; the binding's accumulate argument takes False / True / NORM_OF_SUM only."""
    from fsdp_sharded_mixed_flatparameter_gb300 import FlatShardAdamW
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    opt, numels = _opt()
    with pytest.raises(ValueError):
        opt.device_flat_table(torch.zeros(opt.ghi - opt.glo + 1, dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        opt.device_flat_table(torch.zeros(1, opt.ghi - opt.glo, dtype=torch.bfloat16))
    nobuf = FlatShardAdamW(numels, device="cpu", grad_buffer=False)
    with pytest.raises(ValueError, match="grad buffer"):
        nobuf._launch_direct(None, 0, nobuf.total, torch.bfloat16, 0, nobuf.total, 0, 1.0, True, None, None)
    assert [zs._accum_mode(a) for a in (False, True, 0, 1, zs.NORM_OF_SUM)] == [0, 1, 0, 1, 2]
    for bad in (3, -1, 2.5):
        with pytest.raises(ValueError):
            zs._accum_mode(bad)
