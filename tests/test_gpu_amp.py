"""Mixed precision with dynamic loss scaling on the GPU vs the oracle.

fp16 shard grads of a scaled loss (S * g, S = 2^16 at start) accumulate over
4 micro-batches with the unscale folded into the accumulate scale
1/(S * 4); an overflow injected in one micro-batch of step 3 must raise the
non-finite flag, skip the step on both sides (state and t untouched) and back
the scale off; the scale then grows again after `growth_interval` good steps.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _helpers import bits_equal_f32, raw

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fsdp_sharded_mixed_flatparameter_gb300 import build, zero_shard
    build.build()
    zero_shard.lib()


def test_loss_scaled_fp16_accumulation_with_overflow_skip():
    from fsdp_sharded_mixed_flatparameter_gb300 import DynamicLossScale, FlatShardAdamW
    wl = W.llama13b_zero3().with_(numels=tuple(W.llama_numels(2, 256, 688, 1000)), max_norm=0.05)
    s, e = oracle.shard_range(wl.total, wl.world_size, wl.rank)
    n, M, interval = e - s, 4, 2
    master = W.master_init(wl, s, e)
    opt = FlatShardAdamW(wl.numels, world_size=wl.world_size, rank=wl.rank, lr=wl.lr, betas=wl.betas, eps=wl.eps,
                         weight_decay=wl.weight_decay, max_norm=wl.max_norm, device=DEV, master=master.to(DEV))
    scaler = DynamicLossScale(2.0 ** 16, 2.0, 0.5, interval)
    st = oracle.new_state(master.numpy())
    ref_scales, found_hist = [], []
    ref_scale = 2.0 ** 16
    for t in range(1, 8):
        S = ref_scale  # the oracle side's scale decides the inputs
        assert scaler.scale == S
        unscale = 1.0 / (S * M)
        acc = np.zeros(n, np.float32)
        ref_flag = False
        for j in range(M):
            g = W.flat_grads(wl.with_(grad_dtype="f32", grad_std=1e-5), t, j, s, e)
            x = (g * S).to(torch.float16)
            if t == 3 and j == 2:
                x[n // 3] = math.inf  # overflow in one micro-batch
            opt.accum(x.to(DEV), accumulate=j > 0, scale=unscale, fuse_norm=j == M - 1)
            ref_flag |= oracle.accum(acc, raw(x), "f16", unscale, accumulate=j > 0)
        res = opt.step()
        found = bool(opt.found_nonfinite.item())
        opt.found_nonfinite.zero_()
        scaler.update(found or not res.finite)
        cr = oracle.step_reference(st, acc, lr=wl.lr, betas=wl.betas, eps=wl.eps, wd=wl.weight_decay,
                                   max_norm=wl.max_norm)
        assert found == ref_flag == (t == 3)
        assert res.finite == cr.finite == (t != 3)
        found_hist.append(ref_flag or not cr.finite)
        ref_scale = oracle.loss_scale_trajectory(found_hist, 2.0 ** 16, 2.0, 0.5, interval)[-1]
        assert scaler.scale == ref_scale, (t, scaler.scale, ref_scale)
        assert opt.t == st.t == (t if t < 3 else t - 1)
        for got, ref in ((opt.master, st.p), (opt.exp_avg, st.m), (opt.exp_avg_sq, st.v)):
            assert bits_equal_f32(raw(got), ref), t
        assert np.array_equal(raw(opt.lowp), st.lowp)
    # backed off once at step 3, grew at steps 2, 5, 7
    assert scaler.scale == 2.0 ** 16 * 2 * 0.5 * 2 * 2


@pytest.mark.parametrize("direct,inf_micro", [(False, 2), (True, 2), (True, 3)],
                         ids=["materialized", "direct", "direct-overflow-in-last"])
def test_graph_captured_loss_scaled_steps_with_device_scale(direct, inf_micro):
    """The same loss-scaled fp16 accumulation, captured once in a CUDA graph with the loss
    scale on the device (DeviceLossScale): the accumulate passes read the unscale factor
    from device memory, the overflow flag and the non-finite norm drive the device-side
    update, the step count and skip decision stay on the device.  Replayed for 7 steps
    (an overflow at step 3) and checked after every step against the oracle: the state bit
    for bit, the step count, and the scale trajectory of the GradScaler policy.  direct:
    the last micro-batch is read in place (step_flat, accumulated) by the norm pass and
    AdamW, both reading the unscale factor on the device; the overflow lands in an earlier
    micro-batch or in that last one."""
    from fsdp_sharded_mixed_flatparameter_gb300 import DeviceLossScale, FlatShardAdamW
    wl = W.llama13b_zero3().with_(numels=tuple(W.llama_numels(2, 256, 688, 1000)), max_norm=0.05)
    s, e = oracle.shard_range(wl.total, wl.world_size, wl.rank)
    n, M, interval = e - s, 4, 2
    master = W.master_init(wl, s, e)
    opt = FlatShardAdamW(wl.numels, world_size=wl.world_size, rank=wl.rank, lr=wl.lr, betas=wl.betas, eps=wl.eps,
                         weight_decay=wl.weight_decay, max_norm=wl.max_norm, device=DEV, master=master.to(DEV),
                         capturable=True)
    scaler = DeviceLossScale(DEV, 2.0 ** 16, 2.0, 0.5, interval, accum_steps=M)
    micro = [torch.zeros(n, dtype=torch.float16, device=DEV) for _ in range(M)]
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    if direct:
        opt.device_flat_table(micro[-1])  # built before the capture
    with torch.cuda.graph(graph):
        if direct:
            for j in range(M - 1):
                opt.accum(micro[j], accumulate=j > 0, loss_scale=scaler)
            opt.launch_step_flat(micro[-1], accumulated=True, loss_scale=scaler)
        else:
            for j in range(M):
                opt.accum(micro[j], accumulate=j > 0, fuse_norm=j == M - 1, loss_scale=scaler)
            opt.launch_step()
        scaler.launch_update(opt.norm_buf)
    st = oracle.new_state(master.numpy())
    found_hist = []
    ref_scale = 2.0 ** 16
    for t in range(1, 8):
        S = scaler.scale  # what a backward would multiply the loss by (read here only to build inputs)
        assert S == ref_scale, (t, S, ref_scale)
        unscale = float(np.float32(1.0 / (S * M)))
        acc = np.zeros(n, np.float32)
        ref_flag = False
        for j in range(M):
            g = W.flat_grads(wl.with_(grad_dtype="f32", grad_std=1e-5), t, j, s, e)
            x = (g * S).to(torch.float16)
            if t == 3 and j == inf_micro:
                x[n // 3] = math.inf
            micro[j].copy_(x.to(DEV))
            ref_flag |= oracle.accum(acc, raw(x), "f16", unscale, accumulate=j > 0)
        graph.replay()
        cr = oracle.step_reference(st, acc, lr=wl.lr, betas=wl.betas, eps=wl.eps, wd=wl.weight_decay,
                                   max_norm=wl.max_norm)
        assert ref_flag == (t == 3) and cr.finite == (t != 3)
        found_hist.append(ref_flag or not cr.finite)
        ref_scale = oracle.loss_scale_trajectory(found_hist, 2.0 ** 16, 2.0, 0.5, interval)[-1]
        state = scaler.read()
        assert state.scale == ref_scale and state.found_inf == 0, (t, state.scale, ref_scale)
        assert state.unscale == np.float32(1.0 / (ref_scale * M))
        assert opt.t == st.t == (t if t < 3 else t - 1)
        for got, ref in ((opt.master, st.p), (opt.exp_avg, st.m), (opt.exp_avg_sq, st.v)):
            assert bits_equal_f32(raw(got), ref), t
        assert np.array_equal(raw(opt.lowp), st.lowp)
    assert ref_scale == 2.0 ** 16 * 2 * 0.5 * 2 * 2


def test_device_scale_matches_host_scale_in_every_grad_pass():
    """A scale read from device memory (d_scale) gives the bits of the same scale passed from
    the host, in the flatten (writing, norm-only and norm of the accumulated sum), the
    accumulation, the reduction and AdamW through the table (with and without the sum), with
    their fused norm partials and the non-finite flag."""
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    from test_gpu_kernels import _table_case
    numels = list(W.llama_numels(1, 256, 688, 1000)) + list(W.ragged_numels(50, seed=2, max_log2=12))
    host, dev = _table_case(numels, "f16", seed=5, elem_offsets=[0, 3])
    table, total = zs.zero_tensor_table(dev, numels)
    d_table = zs.device_table(table, len(numels), DEV)
    nb = zs.zero_grad_sqnorm_workspace_bytes(total)
    for scale in (2.0 ** -16 / 4, 0.3):
        dsc = torch.tensor([scale], dtype=torch.float32, device=DEV)
        outs = []
        for d_scale in (None, dsc):
            hs = scale if d_scale is None else 7.0  # the host value is ignored when d_scale is given
            flag = torch.zeros(1, dtype=torch.int32, device=DEV)
            dst = torch.empty(total, device=DEV)
            ws1 = torch.zeros(nb, dtype=torch.uint8, device=DEV)
            zs.zero_flatten_cast(d_table, len(numels), total, torch.float16, 0, total, hs, False, dst, flag, ws1,
                                 d_scale=d_scale)
            ws2 = torch.zeros(nb, dtype=torch.uint8, device=DEV)
            zs.zero_flatten_cast(d_table, len(numels), total, torch.float16, 0, total, hs, False, None, flag, ws2,
                                 d_scale=d_scale)
            src = torch.cat([x.view(-1) for x in dev])
            acc = torch.full((total,), 0.5, device=DEV)
            ws3 = torch.zeros(nb, dtype=torch.uint8, device=DEV)
            zs.zero_accum(acc, src, hs, True, flag, ws3, d_scale=d_scale)
            red = torch.zeros(total, device=DEV)
            ws4 = torch.zeros(nb, dtype=torch.uint8, device=DEV)
            zs.zero_reduce_chunks(red, torch.stack([src, src.flip(0)]), total, hs, False, flag, ws4, d_scale=d_scale)
            # the direct path: the norm of the accumulated sum, and AdamW through the table with the sum
            ws5 = torch.zeros(nb, dtype=torch.uint8, device=DEV)
            zs.zero_flatten_cast(d_table, len(numels), total, torch.float16, 0, total, hs, zs.NORM_OF_SUM, acc, flag,
                                 ws5, d_scale=d_scale)
            state = [torch.linspace(-0.1, 0.1, total, device=DEV), torch.zeros(total, device=DEV),
                     torch.zeros(total, device=DEV)]
            lowp = torch.empty(total, dtype=torch.bfloat16, device=DEV)
            for t in (1, 2):
                zs.zero_adamw_step_tensors(*state, d_table, len(numels), total, torch.float16, 0, hs, lowp, 1e-3, 0.9,
                                           0.95, 1e-8, 0.1, t, None, acc=acc if t == 2 else None, d_scale=d_scale)
            torch.cuda.synchronize()
            outs.append(([t.cpu().view(torch.uint8).numpy() for t in (dst, ws1, ws2, acc, ws3, red, ws4, ws5,
                                                                      *state, lowp)],
                         flag.item()))
        (host_bufs, host_flag), (dev_bufs, dev_flag) = outs
        assert host_flag == dev_flag
        for a, b in zip(host_bufs, dev_bufs):
            assert np.array_equal(a, b), scale
