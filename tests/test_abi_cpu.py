"""The C-ABI library without a GPU: it builds, loads, exports every symbol the
header declares, its host-only calls agree with the oracle bit for bit, and
invalid arguments are rejected on the host before anything is launched."""
import ctypes
import math
import os
import re

import numpy as np
import pytest

import oracle
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from fsdp_sharded_mixed_flatparameter_gb300 import build, zero_shard
    build.build()
    return zero_shard.lib()


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(zero_[a-z0-9_]+)\s*\(", src))
    return names


def test_header_declares_the_boundary():
    want = {"zero_shard_range", "zero_tensor_table", "zero_flatten_cast", "zero_accum",
            "zero_grad_sqnorm_workspace_bytes", "zero_grad_sqnorm", "zero_adamw_step", "zero_status_string",
            "zero_last_error"}
    assert want <= declared_symbols()


def test_library_exports_every_declared_symbol(L):
    for name in sorted(declared_symbols()):
        assert hasattr(L, name), name


def test_shard_range_matches_oracle(L):
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    for total in list(range(0, 70)) + [1261891, 124439808, 6738415616, 13015864320, 2**62]:
        for world in (1, 2, 3, 4, 7, 8, 17, 64):
            for rank in {0, 1 % world, world // 2, world - 1}:
                assert zs.zero_shard_range(total, world, rank) == oracle.shard_range(total, world, rank), \
                    (total, world, rank)


def test_shard_range_rejects(L):
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    for args in [(-1, 2, 0), (10, 0, 0), (10, 2, 2), (10, 2, -1)]:
        with pytest.raises(zs.ZeroError) as ei:
            zs.zero_shard_range(*args)
        assert ei.value.status == zs.ZERO_EINVAL
    s = ctypes.c_int64()
    assert L.zero_shard_range(10, 2, 0, ctypes.byref(s), None) == 1
    assert b"NULL" in L.zero_last_error()


def test_tensor_table_matches_oracle_offsets(L):
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    for numels in (W.small_ragged().numels, W.gpt2_zero1().numels, W.llama7b().numels, (0, 0, 5, 0), ()):
        table, total = zs.zero_tensor_table(numels=numels)
        off = oracle.flat_offsets(numels)
        assert total == off[-1]
        got = [table[i].flat_offset for i in range(len(numels))]
        assert got == list(off[:-1])
        assert all(table[i].ptr is None for i in range(len(numels)))


def test_tensor_table_rejects(L):
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    with pytest.raises(zs.ZeroError):
        zs.zero_tensor_table(numels=[3, -1])
    with pytest.raises(zs.ZeroError):
        zs.zero_tensor_table(numels=[2**62, 2**62, 2**62])


def test_workspace_bytes(L):
    assert L.zero_grad_sqnorm_workspace_bytes(0) == 0
    assert L.zero_grad_sqnorm_workspace_bytes(-5) == 0
    assert L.zero_grad_sqnorm_workspace_bytes(1) == 8
    assert L.zero_grad_sqnorm_workspace_bytes(32768) == 8
    assert L.zero_grad_sqnorm_workspace_bytes(32769) == 16
    assert L.zero_grad_sqnorm_workspace_bytes(6738415616) == 8 * 205641


def test_invalid_arguments_return_einval_before_any_launch(L):
    """Every check below happens on the host; no CUDA call is made (there is no GPU here)."""
    from fsdp_sharded_mixed_flatparameter_gb300.zero_shard import zero_adamw_hparams
    FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: each call fails validation first
    hp = zero_adamw_hparams(1e-3, 0.9, 0.999, 1e-8, 0.0)
    cases = [
        L.zero_flatten_cast(None, 2, 10, 1, 0, 5, 1.0, None, 0, FAKE, None, None, 0, None),          # NULL table
        L.zero_flatten_cast(FAKE, -1, 10, 1, 0, 5, 1.0, None, 0, FAKE, None, None, 0, None),         # n_tensors < 0
        L.zero_flatten_cast(FAKE, 2, 10, 1, 6, 5, 1.0, None, 0, FAKE, None, None, 0, None),          # start > end
        L.zero_flatten_cast(FAKE, 2, 10, 1, 0, 11, 1.0, None, 0, FAKE, None, None, 0, None),         # end > total
        L.zero_flatten_cast(FAKE, 2, 10, 7, 0, 5, 1.0, None, 0, FAKE, None, None, 0, None),          # bad dtype
        L.zero_flatten_cast(FAKE, 2, 10, 1, 0, 5, 1.0, None, 2, FAKE, None, None, 0, None),          # 2 without norm ws
        L.zero_flatten_cast(FAKE, 2, 10, 1, 0, 5, 1.0, None, 2, None, None, FAKE, 8, None),          # 2 with NULL dst
        L.zero_flatten_cast(FAKE, 2, 10, 1, 0, 5, 1.0, None, 3, FAKE, None, FAKE, 8, None),          # accumulate 3
        L.zero_flatten_cast(FAKE, 2, 10, 1, 0, 5, 1.0, None, -1, FAKE, None, FAKE, 8, None),         # accumulate -1
        L.zero_accum(FAKE, FAKE, 1, 10, 1.0, None, 2, None, FAKE, 8, None),                          # accumulate 2
        L.zero_flatten_cast(FAKE, 2, 10, 1, 0, 5, math.nan, None, 0, FAKE, None, None, 0, None),     # NaN scale
        L.zero_flatten_cast(FAKE, 2, 10, 1, 0, 5, 1.0, None, 0, None, None, None, 0, None),          # NULL dst
        L.zero_flatten_cast(FAKE, 0, 10, 1, 0, 5, 1.0, None, 0, FAKE, None, None, 0, None),          # total without tensors
        L.zero_accum(None, FAKE, 1, 10, 1.0, None, 0, None, None, 0, None),
        L.zero_accum(FAKE, FAKE, 1, -1, 1.0, None, 0, None, None, 0, None),
        L.zero_accum(FAKE, FAKE, 9, 10, 1.0, None, 0, None, None, 0, None),
        L.zero_accum(FAKE, FAKE, 1, 10, math.inf, None, 0, None, None, 0, None),
        L.zero_flatten_cast(FAKE, 2, 10, 1, 0, 5, 1.0, None, 0, FAKE, None, FAKE, 0, None),   # norm ws too small
        L.zero_flatten_cast(FAKE, 2, 10, 1, 0, 5, 1.0, None, 0, FAKE, None, ctypes.c_void_p(0x1003), 8, None),  # misaligned
        L.zero_accum(FAKE, FAKE, 1, 40000, 1.0, None, 0, None, FAKE, 8, None),              # norm ws too small
        L.zero_grad_sqnorm_finalize(None, 10, 0.0, 1.0, FAKE, None),                   # NULL ws
        L.zero_grad_sqnorm_finalize(FAKE, 10, 0.0, 1.0, None, None),                   # NULL out
        L.zero_grad_sqnorm_finalize(FAKE, -1, 0.0, 1.0, FAKE, None),                   # n < 0
        L.zero_grad_sqnorm_finalize(FAKE, 10, math.inf, 1.0, FAKE, None),              # bad extra
        L.zero_grad_sqnorm(None, 10, 0.0, 1.0, FAKE, 8, FAKE, None),                  # NULL grad
        L.zero_grad_sqnorm(FAKE, 10, 0.0, 1.0, FAKE, 8, None, None),                  # NULL out
        L.zero_grad_sqnorm(FAKE, 40000, 0.0, 1.0, FAKE, 8, FAKE, None),               # workspace too small
        L.zero_grad_sqnorm(FAKE, 10, 0.0, 1.0, None, 8, FAKE, None),                  # NULL workspace
        L.zero_grad_sqnorm(FAKE, 10, 0.0, 1.0, ctypes.c_void_p(0x1004), 8, FAKE, None),  # misaligned ws
        L.zero_grad_sqnorm(FAKE, 10, -1.0, 1.0, FAKE, 8, FAKE, None),                 # negative extra
        L.zero_grad_sqnorm(FAKE, 10, 0.0, math.nan, FAKE, 8, FAKE, None),             # NaN max_norm
        L.zero_grad_sqnorm(FAKE, 10, 0.0, -1.0, FAKE, 8, FAKE, None),                 # negative max_norm
        L.zero_adamw_step(FAKE, FAKE, FAKE, FAKE, None, 1, 10, ctypes.byref(hp), 0, None, None),   # step 0
        L.zero_adamw_step(FAKE, FAKE, FAKE, FAKE, None, 1, 10, None, 1, None, None),               # NULL hp
        L.zero_adamw_step(FAKE, None, FAKE, FAKE, None, 1, 10, ctypes.byref(hp), 1, None, None),   # NULL m
        L.zero_adamw_step(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 10, ctypes.byref(hp), 1, None, None),   # F32 lowp
        L.zero_adamw_step(FAKE, FAKE, FAKE, FAKE, None, 1, -3, ctypes.byref(hp), 1, None, None),   # n < 0
    ]
    for i, bad in enumerate([zero_adamw_hparams(-1, .9, .999, 1e-8, 0), zero_adamw_hparams(1e-3, 1.0, .999, 1e-8, 0),
                             zero_adamw_hparams(1e-3, .9, .999, 0.0, 0), zero_adamw_hparams(1e-3, .9, .999, 1e-8, -1),
                             zero_adamw_hparams(math.nan, .9, .999, 1e-8, 0)]):
        cases.append(L.zero_adamw_step(FAKE, FAKE, FAKE, FAKE, None, 1, 10, ctypes.byref(bad), 1, None, None))
    # AdamW through the tensor table (d_acc is nullable and never the reason for a refusal)
    cases += [
        L.zero_adamw_step_tensors(FAKE, FAKE, FAKE, None, 2, 10, 1, 0, 1.0, None, FAKE, None, 1, 5, ctypes.byref(hp), 1,
                                  None, None),                                                   # NULL table
        L.zero_adamw_step_tensors(FAKE, FAKE, FAKE, FAKE, 2, 10, 1, 6, 1.0, None, FAKE, None, 1, 5, ctypes.byref(hp), 1,
                                  None, None),                                                   # past total
        L.zero_adamw_step_tensors(FAKE, FAKE, FAKE, FAKE, 2, 10, 9, 0, 1.0, None, FAKE, None, 1, 5, ctypes.byref(hp), 1,
                                  None, None),                                                   # bad grad dtype
        L.zero_adamw_step_tensors(FAKE, FAKE, FAKE, FAKE, 2, 10, 1, 0, math.inf, None, FAKE, None, 1, 5,
                                  ctypes.byref(hp), 1, None, None),                              # inf grad_scale
        L.zero_adamw_step_tensors(FAKE, FAKE, FAKE, FAKE, 2, 10, 1, 0, 1.0, None, FAKE, None, 1, 5, ctypes.byref(hp), 0,
                                  None, None),                                                   # step 0
        L.zero_adamw_step_tensors(FAKE, None, FAKE, FAKE, 2, 10, 1, 0, 1.0, None, FAKE, None, 1, 5, ctypes.byref(hp), 1,
                                  None, None),                                                   # NULL m
    ]
    # graph-capturable calls (device step state)
    cases += [
        L.zero_adamw_prepare_device(None, None, FAKE, None),                                   # NULL hp
        L.zero_adamw_prepare_device(FAKE, None, None, None),                                   # NULL state
        L.zero_adamw_prepare_device(FAKE, None, ctypes.c_void_p(0x1004), None),                # misaligned state
        L.zero_adamw_step_device(FAKE, FAKE, FAKE, FAKE, None, 1, 10, None, None, None),       # NULL state
        L.zero_adamw_step_device(FAKE, FAKE, FAKE, None, None, 1, 10, FAKE, None, None),       # NULL grad
        L.zero_adamw_step_device(FAKE, FAKE, FAKE, FAKE, FAKE, 0, 10, FAKE, None, None),       # F32 lowp
        L.zero_adamw_step_device(FAKE, FAKE, FAKE, FAKE, None, 1, -1, FAKE, None, None),       # n < 0
        L.zero_adamw_step_tensors_device(FAKE, FAKE, FAKE, None, 2, 10, 1, 0, 1.0, None, None, None, 1, 5, FAKE, None,
                                         None),                                                  # NULL table
        L.zero_adamw_step_tensors_device(FAKE, FAKE, FAKE, FAKE, 2, 10, 1, 6, 1.0, None, FAKE, None, 1, 5, FAKE, None,
                                         None),                                                  # past total
        L.zero_adamw_step_tensors_device(FAKE, FAKE, FAKE, FAKE, 2, 10, 1, 0, 1.0, None, FAKE, None, 1, 5, None, None,
                                         None),                                                  # NULL state
        L.zero_loss_scale_update_device(None, 1, 2.0, 0.5, 10, None, None),                     # NULL state
        L.zero_loss_scale_update_device(FAKE, 0, 2.0, 0.5, 10, None, None),                     # accum_steps 0
        L.zero_loss_scale_update_device(FAKE, 1, 1.0, 0.5, 10, None, None),                     # growth 1
        L.zero_loss_scale_update_device(FAKE, 1, 2.0, 1.0, 10, None, None),                     # backoff 1
        L.zero_loss_scale_update_device(FAKE, 1, 2.0, 0.5, 0, None, None),                      # interval 0
        L.zero_adamw_scalars(ctypes.byref(hp), 0, FAKE),                                       # step 0
        L.zero_adamw_scalars(None, 1, FAKE),                                                   # NULL hp
        L.zero_adamw_scalars(ctypes.byref(hp), 1, None),                                       # NULL out
    ]
    assert cases == [1] * len(cases), [i for i, c in enumerate(cases) if c != 1]
    assert len(L.zero_last_error()) > 0


def test_empty_calls_are_noops_without_a_gpu(L):
    from fsdp_sharded_mixed_flatparameter_gb300.zero_shard import zero_adamw_hparams
    hp = zero_adamw_hparams(1e-3, 0.9, 0.999, 1e-8, 0.0)
    assert L.zero_flatten_cast(None, 0, 0, 1, 0, 0, 1.0, None, 0, None, None, None, 0, None) == 0
    assert L.zero_flatten_cast(None, 0, 0, 1, 0, 0, 1.0, None, 2, None, None, None, 0, None) == 0  # norm of the sum
    assert L.zero_adamw_step_tensors(None, None, None, None, 0, 0, 1, 0, 1.0, None, None, None, 1, 0,
                                     ctypes.byref(hp), 1, None, None) == 0
    assert L.zero_accum(None, None, 1, 0, 1.0, None, 0, None, None, 0, None) == 0
    assert L.zero_adamw_step(None, None, None, None, None, 1, 0, ctypes.byref(hp), 1, None, None) == 0


def test_adamw_scalars_match_oracle(L):
    """The per-step scalars (bias corrections by double-double binary powering, shared with
    the device step state) equal the oracle's pow-based ones bit for bit over the first
    100,000 steps and a sparse sweep to 10^7 steps, for every configuration's hyper-parameters
    and a few more betas."""
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    hps = {(w.lr, w.betas[0], w.betas[1], w.eps, w.weight_decay) for w in (f() for f in W.ALL.values())}
    hps |= {(1e-3, 0.8, 0.99, 1e-6, 0.01), (6e-4, 0.0, 0.98, 1e-8, 0.0), (2e-5, 0.99, 0.9999, 1e-12, 0.3)}
    steps = list(range(1, 100_001)) + list(range(100_001, 10_000_000, 9973))
    for hp in sorted(hps):
        for t in steps:
            got, ref = zs.zero_adamw_scalars(*hp, t), oracle.adamw_scalars(*hp, t)
            if not np.array_equal(got.view(np.uint32), ref.view(np.uint32)):
                raise AssertionError((hp, t, got, ref))


def test_status_strings(L):
    assert L.zero_status_string(0) == b"ZERO_OK"
    assert b"EINVAL" in L.zero_status_string(1)
    assert b"ECUDA" in L.zero_status_string(2)


def test_binding_refuses_host_tensors(L):
    import torch
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    cpu = torch.zeros(16)
    with pytest.raises(ValueError):
        zs.zero_adamw_step(cpu, cpu, cpu, cpu, None, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1)
    with pytest.raises(ValueError):  # pageable host grads never reach the table
        zs.zero_tensor_table([cpu], [16])
    with pytest.raises(ValueError):
        zs.zero_accum(cpu, cpu, 1.0, False)


def test_loss_scale_update_matches_oracle(L):
    """The library's host policy against the oracle's, including growth capped at float max."""
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    rng = np.random.default_rng(3)
    for interval, init in ((1, 2.0 ** 16), (4, 2.0 ** 16), (7, 2.0 ** 120), (2000, 1.0)):
        found = [bool(x) for x in rng.random(500) < 0.2]
        sc = zs.DynamicLossScale(init, 2.0, 0.5, interval)
        got = []
        for f in found:
            sc.update(f)
            got.append(sc.scale)
        assert got == oracle.loss_scale_trajectory(found, init, 2.0, 0.5, interval)
    bad = zs.DynamicLossScale(2.0, 1.0, 0.5, 10)
    with pytest.raises(zs.ZeroError):
        bad.update(False)
