"""Run one workload through the CUDA path (FlatShardAdamW over the C ABI) and
through the CPU oracle, step by step, comparing after every step.

Inputs come from ``workloads`` (seeded, drawn once on the GPU and copied to
the host for the oracle).  Each side computes its own grad norm and clip
coefficient.  The oracle either tracks the whole shard or, for the
multi-billion-parameter configurations, a seeded sample of shard positions;
its grad norm always covers every element (the grads are streamed to the
host in chunks).  Sampling is exact because the update is element-wise once
the coefficient is known (pinned by the shard-slice equivalence test).
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np
import torch

import oracle
import workloads as W
from _helpers import (RTOL_NORM, assert_close_f32, assert_lowp_ulp, assert_lowp_ulp_f16, bits_equal_f32, raw)

DEV = torch.device("cuda:0")
# host threads for the oracle's chunks of the multi-billion-parameter configurations
ORACLE_THREADS = max(1, min(16, os.cpu_count() or 1))


@dataclass
class StepReport:
    t: int
    gpu_norm: float
    ref_norm: float
    gpu_coef: float
    ref_coef: float
    exact: bool


@dataclass
class RunReport:
    name: str
    n: int
    steps: List[StepReport] = field(default_factory=list)


def _host_parts(tg: W.TensorGrads, numels, offsets, a: int, b: int, nulls):
    """Host arrays whose concatenation is the flat range [a, b) of the per-tensor grads."""
    i0 = int(np.searchsorted(offsets, a, side="right") - 1)
    parts, pn = [], []
    first = None
    i = i0
    spans = []
    while i < len(numels) and offsets[i] < b:
        lo, hi = max(a, offsets[i]), min(b, offsets[i] + numels[i])
        if hi > lo:
            spans.append((i, lo, hi))
        i += 1
    # one device->host copy of the storage region that holds these spans
    live = [(i, lo, hi) for (i, lo, hi) in spans if i not in nulls]
    if live:
        s0 = tg.starts[live[0][0]] + (live[0][1] - offsets[live[0][0]])
        s1 = tg.starts[live[-1][0]] + (live[-1][2] - offsets[live[-1][0]])
        host = raw(tg.storage[s0:s1])
    for i, lo, hi in spans:
        pn.append(hi - lo)
        if i in nulls:
            parts.append(None)
        else:
            st = tg.starts[i] + (lo - offsets[i]) - s0
            parts.append(np.ascontiguousarray(host[st:st + (hi - lo)]))
    return parts, pn


def _adamw_parts(st, g, sc, coef, lowp_dtype, threads: int, part: int = 1 << 24) -> None:
    """The oracle's AdamW over the state, in contiguous parts on host threads when it is
    large: the update is element-wise, so the parts give the single call's values."""
    n = st.p.size
    if threads <= 1 or n <= 2 * part:
        oracle.adamw(st.p, st.m, st.v, g, sc, coef, st.lowp, lowp_dtype)
        return

    def one(a):
        b = min(a + part, n)
        oracle.adamw(st.p[a:b], st.m[a:b], st.v[a:b], g[a:b], sc, coef, st.lowp[a:b], lowp_dtype)

    with ThreadPoolExecutor(max_workers=threads) as pool:
        list(pool.map(one, range(0, n, part)))


def run_workload(wl: W.Workload, steps: int, sample: Optional[int] = None, chunk: int = 1 << 26,
                 seed: int = 0, fused: bool = True, direct: bool = False, graph: bool = False,
                 oracle_threads: int = ORACLE_THREADS) -> RunReport:
    """fused: the last micro-batch's flatten/accumulate also computes the grad
    norm's partials (the norm is then only finalized); otherwise the norm is a
    separate pass over the flat grad.  direct: the last micro-batch is never
    written to the fp32 grad: step_tensors() (per-tensor grads) or step_flat()
    (flat ZeRO-3 grads) read it in the norm pass and in AdamW, added to the
    earlier micro-batches' sum when there are any (without them there is no
    fp32 grad buffer at all).  graph: a
    capturable optimizer (step count and skip decision on the device); the
    first step's grad passes and step are captured in one CUDA graph and every
    step replays it over grads rewritten in place."""
    from fsdp_sharded_mixed_flatparameter_gb300 import FlatShardAdamW

    s, e = oracle.shard_range(wl.total, wl.world_size, wl.rank)
    n = e - s
    glo, ghi = (0, wl.total) if wl.mode == "zero1" else (s, e)
    lowp_dt = W.torch_dtype(wl.lowp_dtype)
    master = W.master_init(wl, s, e, device=DEV)
    opt = FlatShardAdamW(wl.numels, world_size=wl.world_size, rank=wl.rank, lr=wl.lr, betas=wl.betas, eps=wl.eps,
                         weight_decay=wl.weight_decay, max_norm=wl.max_norm, lowp_dtype=lowp_dt,
                         grad_range="full" if wl.mode == "zero1" else "shard", device=DEV, master=master.clone(),
                         grad_buffer=not direct or wl.micro_batches > 1, capturable=graph)
    assert (opt.start, opt.end) == (s, e)
    if sample is None or sample >= n:
        idx = None
        st = oracle.new_state(raw(master))
    else:
        rng = np.random.default_rng(seed)
        idx = np.unique(np.concatenate([rng.integers(0, n, size=sample), [0, n - 1]])).astype(np.int64)
        st = oracle.new_state(raw(master)[idx])
        d_idx = torch.from_numpy(idx).to(DEV)
    del master
    offsets = oracle.flat_offsets(wl.numels)
    nulls = set(wl.null_grads)
    M = wl.micro_batches
    scale = 1.0 / M
    report = RunReport(wl.name, n)
    storages = [None] * M
    captured = None

    def enqueue(micro):
        for j in range(M - 1 if direct else M):
            if wl.mode == "zero3":
                opt.accum(micro[j], accumulate=j > 0, scale=scale, fuse_norm=fused and j == M - 1)
            else:
                opt.flatten(micro[j].tensors, accumulate=j > 0, scale=scale, fuse_norm=fused and j == M - 1)
        if direct and wl.mode == "zero3":
            opt.launch_step_flat(micro[-1], scale=scale, accumulated=M > 1)
        elif direct:
            opt.launch_step_tensors(micro[-1].tensors, scale=scale, accumulated=M > 1)
        else:
            opt.launch_step()

    for t in range(1, steps + 1):
        micro = []
        for j in range(M):
            if wl.mode == "zero3":
                src = W.flat_grads(wl, t, j, s, e, device=DEV, out=storages[j])
                storages[j] = src
                micro.append(src)
            else:
                tg = W.tensor_grads(wl, t, j, device=DEV, storage=storages[j])
                storages[j] = tg.storage
                micro.append(tg)
        if graph:
            if captured is None:
                for src in micro:  # device tables built before capture (no copies inside it)
                    if wl.mode != "zero3":
                        opt.device_table(src.tensors)
                    elif direct:
                        opt.device_flat_table(src)
                torch.cuda.synchronize()
                captured = torch.cuda.CUDAGraph()
                with torch.cuda.graph(captured):
                    enqueue(micro)
            captured.replay()
        else:
            enqueue(micro)
        res = opt.finish_step()

        # ---- oracle side: accumulate every element (chunked) for the norm.  The
        # chunks are independent (the oracle's calls on disjoint ranges), so large
        # configurations run them on a pool of host threads (ctypes and the
        # device-to-host copies release the GIL); math.fsum of the chunk sums is
        # exact whatever the order, so the result is the single-threaded one.
        g_shard = np.empty(n if idx is None else idx.size, np.float32)

        def oracle_chunk(a):
            b = min(a + chunk, ghi)
            acc = np.empty(b - a, np.float32)
            for j in range(M):
                if wl.mode == "zero3":
                    oracle.accum(acc, raw(micro[j][a - s:b - s]), wl.grad_dtype, scale, accumulate=j > 0)
                else:
                    parts, pn = _host_parts(micro[j], wl.numels, offsets, a, b, nulls)
                    oracle.flatten(parts, pn, wl.grad_dtype, 0, b - a, scale, acc, accumulate=j > 0)
            # the shard's grad values the update needs (disjoint per chunk)
            lo, hi = max(a, s), min(b, e)
            if hi > lo:
                if idx is None:
                    g_shard[lo - s:hi - s] = acc[lo - a:hi - a]
                else:
                    sel = (idx >= lo - s) & (idx < hi - s)
                    g_shard[sel] = acc[idx[sel] + s - a]
            return oracle.sqnorm(acc)

        starts = list(range(glo, ghi, chunk))
        if len(starts) > 2 and oracle_threads > 1:
            with ThreadPoolExecutor(max_workers=min(oracle_threads, len(starts))) as pool:
                sq_parts = list(pool.map(oracle_chunk, starts))
        else:
            sq_parts = [oracle_chunk(a) for a in starts]
        sq = math.fsum(sq_parts)
        cr = oracle.clip(sq, 0.0, wl.max_norm)
        assert res.finite == cr.finite
        assert abs(res.norm - cr.norm) <= RTOL_NORM * cr.norm, (t, res.norm, cr.norm)
        assert abs(res.clip_coef - cr.coef) <= RTOL_NORM * cr.coef, (t, res.clip_coef, cr.coef)
        if cr.finite:
            st.t += 1
            sc = oracle.adamw_scalars(wl.lr, wl.betas[0], wl.betas[1], wl.eps, wl.weight_decay, st.t)
            _adamw_parts(st, g_shard, sc, cr.coef, wl.lowp_dtype, oracle_threads)
        assert opt.t == st.t

        # ---- compare
        if idx is None:
            got = {k: raw(getattr(opt, a)) for k, a in (("p", "master"), ("m", "exp_avg"), ("v", "exp_avg_sq"),
                                                         ("lowp", "lowp"))}
        else:
            got = {k: raw(getattr(opt, a).index_select(0, d_idx))
                   for k, a in (("p", "master"), ("m", "exp_avg"), ("v", "exp_avg_sq"), ("lowp", "lowp"))}
        exact = True
        for k, ref in (("p", st.p), ("m", st.m), ("v", st.v)):
            assert_close_f32(got[k], ref, name=f"{wl.name} step {t} {k}")
            exact &= bits_equal_f32(got[k], ref)
        (assert_lowp_ulp_f16 if wl.lowp_dtype == "f16" else assert_lowp_ulp)(got["lowp"], st.lowp,
                                                                                name=f"{wl.name} step {t} lowp")
        exact &= bool(np.array_equal(got["lowp"], st.lowp))
        # both sides follow the same rounding sequence: with the same binary32
        # clip coefficient the whole state must agree bit for bit
        if res.clip_coef == cr.coef:
            assert exact, f"{wl.name} step {t}: same coefficient but state not bit-exact"
        report.steps.append(StepReport(t, res.norm, cr.norm, res.clip_coef, cr.coef, exact))
    return report
