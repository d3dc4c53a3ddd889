"""Benchmark of the flat-shard optimizer step on the Llama-7B-shaped flat buffer.

One step = the whole hot path over one batch of synthetic grads:
  flatten/cast of the 291 bf16 per-tensor grads into the fp32 flat grad, the
  same pass computing the grad norm's tile partials (K1 with the fused norm)
  -> norm finalize + clip coefficient (K3b)
  -> fused AdamW on fp32 master/exp_avg/exp_avg_sq with the bf16 write-back (K4)
  -> device->host read of the step's grad norm (the skip-policy decision).
Inputs are resident in HBM (135 GB, far larger than the 129 MB L2, so no
flush is needed between steps).  Prints one JSON line.

With N > 1 ranks (torchrun, one per GPU) the step is the ZeRO-2 data plane
over Llama-7B (strong scaling): all-to-all of the flat bf16 grads, rank-order
fp32 reduction with the fused norm, global norm, AdamW on the shard, all-gather
of the bf16 parameters.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
  python bench.py --workload NAME         another configuration's step
  python bench.py --dataplane-ranks N     one rank of an N-rank ZeRO-2 job

--impl reference times the CPU oracle (plain single-threaded C) on a bounded
sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "fused AdamW shard step: params/s and HBM GB/s as % of GB300 peak (Llama-7B flat)"
UNIT = "params/s"
ADAMW_BYTES_PER_PARAM = 30      # read g,p,m,v fp32; write p,m,v fp32 + bf16 copy
FLATTEN_BYTES_PER_PARAM = 6     # read bf16 grad, write fp32 flat grad
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "adamw_llama7b_traffic.txt")


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def adamw_source_hash():
    import hashlib
    h = hashlib.sha256()
    for f in ("adamw.cu", "adam.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "fsdp_sharded_mixed_flatparameter_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def adamw_traffic_per_param():
    """DRAM bytes per parameter of the AdamW kernel from the committed ncu summary,
    or None when the kernel sources have changed since those counters were taken."""
    vals = {}
    try:
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    vals[k.strip()] = v.strip()
    except OSError:
        return None
    if vals.get("adamw_source_sha256") != adamw_source_hash():
        return None
    return float(vals["dram_bytes_per_param"]) if "dram_bytes_per_param" in vals else None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------- oracle
def oracle_step_rate(wl: W.Workload, sample_params: int, min_seconds: float, max_passes: int):
    """Time the oracle's whole step (flatten/cast, sum of squares, clip, AdamW) on
    the first `sample_params` params of the workload, single-threaded."""
    import oracle
    numels, tot = [], 0
    for n in wl.numels:
        take = min(n, sample_params - tot)
        if take <= 0:
            break
        numels.append(take)
        tot += take
    g = torch.Generator().manual_seed(wl.seed)
    grads = [(torch.randn(n, generator=g) * wl.grad_std).to(torch.bfloat16).view(torch.int16).numpy()
             .view(np.uint16) for n in numels]
    p = (torch.randn(tot, generator=g) * wl.init_std).numpy()
    st = oracle.new_state(p)
    flat = np.empty(tot, np.float32)
    passes, t0 = 0, time.perf_counter()
    stage = [0.0, 0.0, 0.0]
    while True:
        ta = time.perf_counter()
        oracle.flatten(grads, numels, "bf16", 0, tot, 1.0, flat, accumulate=False)
        tb = time.perf_counter()
        sq = oracle.sqnorm(flat)
        cr = oracle.clip(sq, 0.0, wl.max_norm)
        tc = time.perf_counter()
        st.t += 1
        sc = oracle.adamw_scalars(wl.lr, wl.betas[0], wl.betas[1], wl.eps, wl.weight_decay, st.t)
        oracle.adamw(st.p, st.m, st.v, flat, sc, cr.coef, st.lowp)
        td = time.perf_counter()
        stage[0] += tb - ta
        stage[1] += tc - tb
        stage[2] += td - tc
        passes += 1
        el = time.perf_counter() - t0
        # min_seconds <= 0: exactly max_passes passes; else stop once min_seconds have passed
        if passes >= max_passes or (min_seconds > 0.0 and el >= min_seconds):
            break
    oracle_step_rate.last_stages = {k: tot * passes / v for k, v in zip(("flatten", "sqnorm", "adamw"), stage)}
    return tot * passes / el, tot, passes, el


def oracle_step_rate_threads(wl: W.Workload, sample_params: int, threads: int, passes: int):
    """The oracle's whole step on the same sample as oracle_step_rate, with the element
    range split into `threads` contiguous parts run by that many host threads (the
    oracle's C functions release the GIL): flatten/cast of each part, each part's sum
    of squares (added exactly with math.fsum, so the norm is the single-threaded one's
    to the last bit or two), clip, AdamW of each part.  A second CPU baseline using all
    the host's cores; the single-threaded oracle stays the parity reference."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor
    numels, tot = [], 0
    for n in wl.numels:
        take = min(n, sample_params - tot)
        if take <= 0:
            break
        numels.append(take)
        tot += take
    g = torch.Generator().manual_seed(wl.seed)
    grads = [(torch.randn(n, generator=g) * wl.grad_std).to(torch.bfloat16).view(torch.int16).numpy()
             .view(np.uint16) for n in numels]
    p = (torch.randn(tot, generator=g) * wl.init_std).numpy()
    st = oracle.new_state(p)
    flat = np.empty(tot, np.float32)
    bounds = [tot * i // threads for i in range(threads + 1)]
    parts = [(a, b) for a, b in zip(bounds[:-1], bounds[1:]) if b > a]

    def flatten_part(ab):
        a, b = ab
        oracle.flatten(grads, numels, "bf16", a, b, 1.0, flat[a:b], accumulate=False)

    def sq_part(ab):
        return oracle.sqnorm(flat[ab[0]:ab[1]])

    with ThreadPoolExecutor(max_workers=len(parts)) as pool:
        def one_pass():
            list(pool.map(flatten_part, parts))
            cr = oracle.clip(math.fsum(pool.map(sq_part, parts)), 0.0, wl.max_norm)
            st.t += 1
            sc = oracle.adamw_scalars(wl.lr, wl.betas[0], wl.betas[1], wl.eps, wl.weight_decay, st.t)
            list(pool.map(lambda ab: oracle.adamw(st.p[ab[0]:ab[1]], st.m[ab[0]:ab[1]], st.v[ab[0]:ab[1]],
                                                  flat[ab[0]:ab[1]], sc, cr.coef, st.lowp[ab[0]:ab[1]]), parts))
        one_pass()  # warm-up: page in the buffers
        t0 = time.perf_counter()
        for _ in range(passes):
            one_pass()
        el = time.perf_counter() - t0
    return tot * passes / el, tot, passes, el


def _sample_list(numels, lo: int, count: int):
    """Sizes of the pieces of the tensor list that cover flat positions [lo, lo + count)."""
    out, pos = [], 0
    for n in numels:
        a, b = max(pos, lo), min(pos + n, lo + count)
        if b > a:
            out.append(b - a)
        pos += n
        if pos >= lo + count:
            break
    return out


def oracle_config_rates(wl: W.Workload, sample_params: int = 1 << 23, min_seconds: float = 2.0, max_reps: int = 5):
    """Time the oracle's stages for one configuration on a bounded sample, single-threaded:
    the grad pass of every micro-batch (per-tensor flatten/cast, or the flat accumulation of
    ZeRO-3 shard grads), the sum of squares and clip, and AdamW.  Returns the per-stage
    rates (elements/s) and the whole step's params/s extrapolated to the configuration's
    sizes (M grad passes and one norm over the grad range, AdamW over the shard)."""
    import oracle
    s, e = oracle.shard_range(wl.total, wl.world_size, wl.rank)
    n = e - s
    glo, ghi = (0, wl.total) if wl.mode == "zero1" else (s, e)
    S = min(sample_params, ghi - glo)
    A = min(sample_params, n)
    rng = np.random.default_rng(wl.seed)
    lowp = {"bf16": torch.bfloat16, "f16": torch.float16}

    def raw16(x):
        return torch.from_numpy(x).to(lowp[wl.grad_dtype]).view(torch.int16).numpy().view(np.uint16)

    def draw(k):
        x = (rng.standard_normal(k) * wl.grad_std).astype(np.float32)
        return x if wl.grad_dtype == "f32" else raw16(x)

    pieces = _sample_list(wl.numels, glo, S)
    srcs = [draw(k) for k in pieces]
    flat_src = draw(S)
    acc = np.empty(S, np.float32)
    st = oracle.new_state((rng.standard_normal(A) * wl.init_std).astype(np.float32))
    gA = (rng.standard_normal(A) * wl.grad_std).astype(np.float32)
    M = wl.micro_batches
    t_grad = t_norm = t_adam = 0.0
    reps = 0
    while reps < max_reps and (reps == 0 or t_grad + t_norm + t_adam < min_seconds):
        t0 = time.perf_counter()
        for j in range(M):
            if wl.mode == "zero3":
                oracle.accum(acc, flat_src, wl.grad_dtype, 1.0 / M, accumulate=j > 0)
            else:
                oracle.flatten(srcs, pieces, wl.grad_dtype, 0, S, 1.0 / M, acc, accumulate=j > 0)
        t1 = time.perf_counter()
        cr = oracle.clip(oracle.sqnorm(acc), 0.0, wl.max_norm)
        t2 = time.perf_counter()
        st.t += 1
        sc = oracle.adamw_scalars(wl.lr, wl.betas[0], wl.betas[1], wl.eps, wl.weight_decay, st.t)
        oracle.adamw(st.p, st.m, st.v, gA, sc, cr.coef, st.lowp)
        t3 = time.perf_counter()
        t_grad += t1 - t0
        t_norm += t2 - t1
        t_adam += t3 - t2
        reps += 1
    r_grad, r_norm, r_adam = M * S * reps / t_grad, S * reps / t_norm, A * reps / t_adam
    step_s = M * (ghi - glo) / r_grad + (ghi - glo) / r_norm + n / r_adam
    return {"value": n / step_s, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"each stage timed on a sample ({S} grad elements x {M} micro-batches, {A} AdamW params, "
                      f"{reps} reps in {t_grad + t_norm + t_adam:.1f} s); value = shard params / "
                      f"(the step's time extrapolated from the stage rates)",
            "stages_elems_per_s": {"grad_pass": r_grad, "sqnorm": r_norm, "adamw": r_adam}}


REFERENCE_SAMPLE = 1 << 24  # params of one reference-arm step (one oracle step over this sample)


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    wl = W.llama7b()
    sample = REFERENCE_SAMPLE
    # exactly --warmup untimed passes, then exactly --steps timed passes, each one whole
    # oracle step over the sample
    if args.warmup > 0:
        oracle_step_rate(wl, sample, 0.0, args.warmup)
    rate, tot, passes, el = oracle_step_rate(wl, sample, 0.0, args.steps)
    assert passes == args.steps
    cores = 1
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / passes,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "params_per_rank": tot, "sample_params": tot,
                   "workload_params": wl.total, "tensors": wl.n_tensors, "world_size": 1,
                   "grad_dtype": "bf16", "lowp_dtype": "bf16", "max_norm": wl.max_norm},
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"each step: the oracle's whole step (flatten/cast, norm, clip, AdamW) on the "
                                   f"first {tot} params of the Llama-7B flat list; value in params/s"},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------------ GPU
def run_gpu(args):
    """The headline line: Llama-7B as one rank (N = 1)."""
    from fsdp_sharded_mixed_flatparameter_gb300 import FlatShardAdamW
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs

    world, rank = 1, 0
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    base = W.llama7b()
    if args.small:
        # profiling case: same tensor shapes per layer, 1 layer, smaller vocab (268M params,
        # ~5 GB on the device, still far larger than L2)
        base = base.with_(name="llama7b_1layer_v8000", numels=tuple(W.llama_numels(1, 4096, 11008, 8000)))
    wl = base
    s, e = zs.zero_shard_range(wl.total, world, rank)
    n = e - s
    shard_numels = list(base.numels)
    torch.manual_seed(0)

    # per-tensor bf16 grads of this rank's shard, one padded storage buffer
    tg = W.tensor_grads(base.with_(seed=base.seed + rank), step=1, micro=0, device=dev)
    master = W.master_init(wl, s, e, device=dev)
    opt = FlatShardAdamW(shard_numels, lr=wl.lr, betas=wl.betas, eps=wl.eps, weight_decay=wl.weight_decay,
                         max_norm=wl.max_norm, device=dev, master=master)
    del master
    grads = tg.tensors
    d_table, _, _ = opt.device_table(grads)
    stream = torch.cuda.current_stream(dev)
    grad_bytes = sum(t.numel() * t.element_size() for t in grads)

    def norm_stage():
        """Norm + clip coefficient from the partials the flatten pass fused in."""
        zs.zero_grad_sqnorm_finalize(opt.ws, n, 0.0, opt.max_norm, opt.norm_buf, stream)

    def one_step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        zs.zero_flatten_cast(d_table, len(grads), opt.total, torch.bfloat16, 0, n, 1.0, False, opt.grad, None,
                             opt.ws, stream)
        if ev is not None:
            ev[1].record(stream)
        norm_stage()
        if ev is not None:
            ev[2].record(stream)
        zs.zero_adamw_step(opt.master, opt.exp_avg, opt.exp_avg_sq, opt.grad, opt.lowp, opt.lr, opt.betas[0],
                           opt.betas[1], opt.eps, opt.weight_decay, opt.t + 1, opt.norm_buf, stream)
        if ev is not None:
            ev[3].record(stream)
        r = opt.finish_step()  # device->host read of the step's result
        if not r.finite:
            raise RuntimeError("non-finite grad norm in the benchmark")
        return r

    def barrier():
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        one_step()
    kernel_events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    with ClockSampler(local) as clk:
        t_start.record(stream)
        for k in range(args.steps):
            one_step(kernel_events[k])
        t_end.record(stream)
        barrier()
    elapsed_ms = t_start.elapsed_time(t_end)

    # ---- the direct path of a step without micro-batch accumulation: a norm-only
    # pass and an AdamW that both read the bf16 grads through the tensor table;
    # no fp32 flat grad is written (30 instead of 36 bytes per parameter).  Same
    # results bit for bit; timed the same way on the same state.
    def one_step_direct(ev=None):
        if ev is not None:
            ev[0].record(stream)
        zs.zero_flatten_cast(d_table, len(grads), opt.total, torch.bfloat16, 0, n, 1.0, False, None, None, opt.ws,
                             stream)
        if ev is not None:
            ev[1].record(stream)
        norm_stage()
        if ev is not None:
            ev[2].record(stream)
        zs.zero_adamw_step_tensors(opt.master, opt.exp_avg, opt.exp_avg_sq, d_table, len(grads), opt.total,
                                   torch.bfloat16, 0, 1.0, opt.lowp, opt.lr, opt.betas[0], opt.betas[1], opt.eps,
                                   opt.weight_decay, opt.t + 1, opt.norm_buf, stream)
        if ev is not None:
            ev[3].record(stream)
        r = opt.finish_step()
        if not r.finite:
            raise RuntimeError("non-finite grad norm in the benchmark")

    for _ in range(args.warmup):
        one_step_direct()
    direct_events = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    d_start, d_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    d_start.record(stream)
    for k in range(args.steps):
        one_step_direct(direct_events[k])
    d_end.record(stream)
    barrier()
    direct_ms = d_start.elapsed_time(d_end)
    dk1 = [ev[0].elapsed_time(ev[1]) for ev in direct_events]
    dk4 = [ev[2].elapsed_time(ev[3]) for ev in direct_events]

    k1 = [ev[0].elapsed_time(ev[1]) for ev in kernel_events]
    k3 = [ev[1].elapsed_time(ev[2]) for ev in kernel_events]
    k4 = [ev[2].elapsed_time(ev[3]) for ev in kernel_events]

    # ---- end to end through the public API (FlatShardAdamW) with host buffers.  The
    # step's bf16 grads live in pinned host memory; the flatten kernel reads them directly
    # over the host link (UVA-mapped pinned memory), so the host-to-device
    # transfer and the flatten/cast are one pass.  For comparison the same is
    # timed with an explicit copy-engine copy into device memory first.
    host = torch.empty(tg.storage.numel(), dtype=tg.storage.dtype, pin_memory=True)
    host.copy_(tg.storage)
    host_grads = [host[st:st + nn] for st, nn in zip(tg.starts, shard_numels)]
    def user_step(step_grads):
        """The calls a user makes: FlatShardAdamW.flatten (fused norm) + step()."""
        opt.flatten(step_grads, accumulate=False, fuse_norm=True, stream=stream)
        r = opt.step(stream=stream)
        if not r.finite:
            raise RuntimeError("non-finite grad norm in the benchmark")

    def one_step_host():
        user_step(host_grads)

    def one_step_copy_engine():
        tg.storage.copy_(host, non_blocking=True)
        user_step(grads)

    def timed(fn):
        for _ in range(max(1, args.warmup // 2)):
            fn()
        barrier()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(args.steps):
            fn()
        b.record(stream)
        barrier()
        return a.elapsed_time(b)

    e2e_ms = timed(one_step_host)
    e2e_copy_ms = timed(one_step_copy_engine)

    peaks, peak_src = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    t_k4 = statistics.mean(k4) / 1e3
    achieved = ADAMW_BYTES_PER_PARAM * n / t_k4 / 1e9
    tpp = adamw_traffic_per_param()
    value = n * world * args.steps / (elapsed_ms / 1e3)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": base.name, "params_per_rank": n, "tensors": len(grads), "world_size": world,
                   "grad_dtype": "bf16", "lowp_dtype": "bf16", "max_norm": wl.max_norm,
                   "l2": "inputs larger than L2 (135 GB resident per GPU); no flush"},
        "roofline": {"bound": "hbm", "kernel": "adamw_v8_kernel", "achieved": achieved, "peak": hbm,
                     "unit": "GB/s", "frac": achieved / hbm, "peak_source": peak_src,
                     "traffic": None if tpp is None else tpp * n,
                     "algorithmic_bytes_per_launch": ADAMW_BYTES_PER_PARAM * n},
        "kernels_ms": {"flatten_norm": statistics.mean(k1), "norm_finalize": statistics.mean(k3),
                       "adamw": statistics.mean(k4)},
        "kernels_gbs": {"flatten_norm": FLATTEN_BYTES_PER_PARAM * n / (statistics.mean(k1) / 1e3) / 1e9,
                        "adamw": achieved},
        "bytes_per_param_step": FLATTEN_BYTES_PER_PARAM + ADAMW_BYTES_PER_PARAM,
        "direct_path": {"value": n * world * args.steps / (direct_ms / 1e3), "unit": UNIT,
                        "ms_per_step": direct_ms / args.steps, "bytes_per_param_step": 2 + 28,
                        "kernels_ms": {"norm_pass": statistics.mean(dk1), "adamw_tensors": statistics.mean(dk4)},
                        "kernels_gbs": {"norm_pass": 2 * n / (statistics.mean(dk1) / 1e3) / 1e9,
                                        "adamw_tensors": 28 * n / (statistics.mean(dk4) / 1e3) / 1e9},
                        "what": "no micro-batch accumulation: norm and AdamW read the bf16 grads through the "
                                "tensor table, the fp32 flat grad is never written; bit-identical results"},
        "gpu_launches": 3 * args.steps,
        "clocks": clk.summary(),
        "e2e": {"value": n * world * args.steps / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": grad_bytes,
                "d2h_bytes_per_step": zs.NORM_RESULT_BYTES, "ms_per_step": e2e_ms / args.steps,
                "how": "bf16 grads in pinned host memory read by the flatten kernel over the host link",
                "copy_engine_ms_per_step": e2e_copy_ms / args.steps},
    }
    if not args.no_cpu_baseline:
        rate, tot, passes, el = oracle_step_rate(base, 1 << 25, 10.0, 50)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": f"first {tot} params of the Llama-7B flat list, {passes} whole-step "
                                          f"passes in {el:.1f} s",
                                "stages_elems_per_s": oracle_step_rate.last_stages}
        threads = max(1, os.cpu_count() or 1)
        trate, ttot, tpasses, tel = oracle_step_rate_threads(base, 1 << 25, threads, 10)
        line["cpu_baseline_all_cores"] = {
            "value": trate, "unit": UNIT, "cores": threads, "kind": "oracle, element ranges on host threads",
            "sample": f"first {ttot} params of the Llama-7B flat list split into {threads} ranges, {tpasses} "
                      f"whole-step passes in {tel:.1f} s"}
    print(json.dumps(line))
    return 0


# ------------------------------------------------------- ZeRO-2/3 data plane
def run_dataplane(args):
    """Llama-7B trained by N ranks with the ZeRO-2 data plane (strong scaling: the
    model is fixed and each rank owns 1/N of it, the ZeRO page's Llama-7B-on-8-cards
    setting).  One step per rank:
      exchange   all-to-all of the padded flat bf16 grad (NCCL): each rank receives
                 every rank's chunk of its shard
      reduce     zero_reduce_chunks: rank-order fp32 sum, x 1/N, fused norm partials
      norm       local finalize, 8-byte all-gather of the ranks' sums, combine
      adamw      fused AdamW on the shard, bf16 write-back into the rank's slice
      all-gather the ranks' bf16 slices into every rank's full FlatParameter
      read       the 24-byte norm result (skip decision)
    With one process and --dataplane-ranks N it times one rank of an N-rank job on
    this GPU: the received blocks are synthetic (every rank's grads as they would
    arrive), the exchange and both all-gathers are left out (nothing to exchange
    with) and the other ranks' sums of squares are stood in by copies of this
    rank's; the line says so.  When ranks share GPUs (fewer devices than ranks)
    they exchange through gloo on host memory: a check of the code path, marked
    as such, not a bench number."""
    import torch.distributed as dist
    from fsdp_sharded_mixed_flatparameter_gb300 import (ZeroDataPlane, exchange_chunks, gather_shards,
                                                        gather_sqnorms, zero_shard as zs)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    ndev = torch.cuda.device_count()
    shared = world > 1 and ndev < world
    dev = torch.device("cuda", local % ndev)
    torch.cuda.set_device(dev)
    group = None
    if world > 1:
        if shared:
            dist.init_process_group("gloo")
        else:
            dist.init_process_group("nccl", device_id=dev)
        group = dist.group.WORLD
    N = world if world > 1 else args.dataplane_ranks
    r = rank if world > 1 else 0
    wl = W.llama7b()
    if args.small:
        wl = wl.with_(name="llama7b_1layer_v8000", numels=tuple(W.llama_numels(1, 4096, 11008, 8000)))
    total = wl.total
    s, e = zs.zero_shard_range(total, N, r)
    n = e - s
    stream = torch.cuda.current_stream(dev)
    master = W.master_init(wl, s, e, device=dev)
    if world > 1:
        dp = ZeroDataPlane(wl.numels, group=group, device=dev, lr=wl.lr, betas=wl.betas, eps=wl.eps,
                           weight_decay=wl.weight_decay, max_norm=wl.max_norm, master=master)
        opt, chunk = dp.opt, dp.chunk
        dp.flat_grad[:total] = W.flat_grads(wl.with_(seed=wl.seed + rank), 1, 0, 0, total, device=dev)
        recv2d = dp.recv.view(N, chunk)
    else:
        from fsdp_sharded_mixed_flatparameter_gb300 import FlatShardAdamW, chunk_layout
        dp = None
        chunk, _ = chunk_layout(total, N)
        opt = FlatShardAdamW(wl.numels, world_size=N, rank=r, lr=wl.lr, betas=wl.betas, eps=wl.eps,
                             weight_decay=wl.weight_decay, max_norm=wl.max_norm, device=dev, master=master)
        recv2d = torch.zeros(N, chunk, dtype=torch.bfloat16, device=dev)
        for j in range(N):  # rank j's values of this rank's shard
            recv2d[j, :n] = W.flat_grads(wl.with_(seed=wl.seed + j), 1, 0, s, e, device=dev)
    del master
    local_buf = zs.new_norm_result(dev)
    NEV = 6

    def one_step(ev=None):
        def mark(i):
            if ev is not None:
                ev[i].record(stream)
        mark(0)
        if dp is not None:
            exchange_chunks(dp.flat_grad, dp.recv, group)
        mark(1)
        zs.zero_reduce_chunks(opt.grad, recv2d, n, 1.0 / N, False, None, opt.ws, stream)
        mark(2)
        zs.zero_grad_sqnorm_finalize(opt.ws, n, 0.0, math.inf, local_buf, stream)
        local_sq = zs.sqnorm_view(local_buf)
        gathered = gather_sqnorms(local_sq, group) if dp is not None else local_sq.repeat(N)
        zs.zero_grad_sqnorm_combine(gathered, opt.max_norm, opt.norm_buf, stream)
        mark(3)
        zs.zero_adamw_step(opt.master, opt.exp_avg, opt.exp_avg_sq, opt.grad, opt.lowp, opt.lr, opt.betas[0],
                           opt.betas[1], opt.eps, opt.weight_decay, opt.t + 1, opt.norm_buf, stream)
        mark(4)
        if dp is not None:
            gather_shards(dp.flat_param, group)
        mark(5)
        res = opt.finish_step(stream)
        if not res.finite:
            raise RuntimeError("non-finite grad norm in the benchmark")

    def barrier():
        torch.cuda.synchronize(dev)
        if group is not None:
            dist.barrier()

    for _ in range(args.warmup):
        one_step()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(NEV)] for _ in range(args.steps)]
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    with ClockSampler(dev.index) as clk:
        a.record(stream)
        for k in range(args.steps):
            one_step(evs[k])
        b.record(stream)
        barrier()
    elapsed_ms = a.elapsed_time(b)
    parts = {name: statistics.mean(ev[i].elapsed_time(ev[i + 1]) for ev in evs)
             for i, name in enumerate(("exchange", "reduce", "norm", "adamw", "all_gather"))}

    e2e_ms, h2d = None, 0
    if dp is not None:
        # end to end through the public API: the step's grads come from pinned host memory
        host = torch.empty(dp.flat_grad.numel(), dtype=dp.flat_grad.dtype, pin_memory=True)
        host.copy_(dp.flat_grad)
        h2d = host.numel() * host.element_size()

        def user_step():
            dp.flat_grad.copy_(host, non_blocking=True)
            dp.reduce_scatter_grads()
            if not dp.step().finite:
                raise RuntimeError("non-finite grad norm in the benchmark")
        user_step()
        barrier()
        a.record(stream)
        for _ in range(args.steps):
            user_step()
        b.record(stream)
        barrier()
        e2e_ms = a.elapsed_time(b)
    if group is not None:
        t = torch.tensor([elapsed_ms, e2e_ms or 0.0] + list(parts.values()), dtype=torch.float64)
        if not shared:
            t = t.to(dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        vals = t.tolist()
        elapsed_ms, e2e_ms = vals[0], vals[1]
        parts = dict(zip(parts, vals[2:]))
        if rank != 0:
            dist.destroy_process_group()
            return 0
    peaks, peak_src = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    adamw_gbs = ADAMW_BYTES_PER_PARAM * n / (parts["adamw"] / 1e3) / 1e9
    reduce_bytes = (2 * N + 4) * n  # N bf16 blocks read, the fp32 shard grad written
    line = {
        "metric": METRIC, "value": total * args.steps / (elapsed_ms / 1e3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True, "scaling": "strong", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{wl.name} ZeRO-2 over {N} ranks", "params_total": total, "params_per_rank": n,
                   "ranks": N, "grad_dtype": "bf16", "lowp_dtype": "bf16", "max_norm": wl.max_norm,
                   "l2": "inputs larger than L2; no flush"},
        "roofline": {"bound": "hbm", "kernel": "adamw_v8_kernel", "achieved": adamw_gbs, "peak": hbm, "unit": "GB/s",
                     "frac": adamw_gbs / hbm, "peak_source": peak_src, "traffic": None,
                     "algorithmic_bytes_per_launch": ADAMW_BYTES_PER_PARAM * n},
        "kernels_ms": parts,
        "kernels_gbs": {"reduce": reduce_bytes / (parts["reduce"] / 1e3) / 1e9, "adamw": adamw_gbs},
        "gpu_launches": 4 * args.steps,
        "clocks": clk.summary(),
    }
    if dp is None:
        line["value"] = n * args.steps / (elapsed_ms / 1e3)
        line["emulated"] = (f"one rank of a {N}-rank job on one GPU: the {N} received blocks are synthetic, the "
                            f"exchange and all-gathers are not run, the other ranks' sums of squares are copies of "
                            f"this rank's; value = this rank's params/s")
        line["scaling"] = "weak"
    else:
        line["e2e"] = {"value": total * args.steps / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": zs.NORM_RESULT_BYTES, "ms_per_step": e2e_ms / args.steps,
                       "how": "ZeroDataPlane.reduce_scatter_grads + step, grads copied from pinned host memory"}
        if shared:
            line["emulated"] = "ranks share one GPU and exchange through gloo on host memory: a code-path check"
    print(json.dumps(line))
    if group is not None:
        dist.destroy_process_group()
    return 0


def llama_unit_numels(numels):
    """A Llama tensor list as FSDP units: the embedding, each transformer block (9 tensors),
    the final norm with the output head."""
    units, i = [list(numels[:1])], 1
    while len(numels) - i > 2:
        units.append(list(numels[i:i + 9]))
        i += 9
    units.append(list(numels[i:]))
    return units


def run_units(args):
    """Llama-7B wrapped as 34 FSDP units (embedding, 32 blocks, head), one FlatParameter and
    data plane each, stepped under one global clip on one GPU (one rank): every unit's
    reduction with the fused norm, the units' local sums combined, AdamW per unit.  The same
    bytes as one FlatParameter; the line shows what the 34-way split costs in launches."""
    from fsdp_sharded_mixed_flatparameter_gb300 import ZeroUnits
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = W.llama7b()
    units = llama_unit_numels(wl.numels)
    offs = [0]
    for u in units:
        offs.append(offs[-1] + sum(u))
    zu = ZeroUnits(units, device=dev, lr=wl.lr, betas=wl.betas, eps=wl.eps, weight_decay=wl.weight_decay,
                   max_norm=wl.max_norm, masters=[W.master_init(wl, offs[i], offs[i + 1], device=dev)
                                                  for i in range(len(units))])
    for i, u in enumerate(zu.units):
        u.flat_grad[:offs[i + 1] - offs[i]] = W.flat_grads(wl, 1, 0, offs[i], offs[i + 1], device=dev)
    stream = torch.cuda.current_stream(dev)

    def one_step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        zu.reduce_scatter_grads()
        if ev is not None:
            ev[1].record(stream)
        if not zu.step().finite:
            raise RuntimeError("non-finite grad norm in the benchmark")
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        one_step()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    with ClockSampler(dev.index) as clk:
        a.record(stream)
        for k in range(args.steps):
            one_step(evs[k])
        b.record(stream)
        torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / args.steps
    t_reduce = statistics.mean(ev[0].elapsed_time(ev[1]) for ev in evs)
    t_step = statistics.mean(ev[1].elapsed_time(ev[2]) for ev in evs)
    line = {
        "metric": METRIC, "value": wl.total / (ms / 1e3), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"{wl.name} as {len(units)} FSDP units", "params_per_rank": wl.total,
                   "units": len(units), "grad_dtype": "bf16", "lowp_dtype": "bf16", "max_norm": wl.max_norm,
                   "l2": "inputs larger than L2; no flush"},
        "bytes_per_param_step": 6 + 30,
        "phases_ms": {"reductions": t_reduce, "norm_adamw_read": t_step},
        "phases_gbs": {"reductions": 6 * wl.total / (t_reduce / 1e3) / 1e9,
                       "adamw": 30 * wl.total / (t_step / 1e3) / 1e9},
        "gpu_launches": (2 * len(units) + 2) * args.steps,  # per unit reduce + AdamW; one finalize, one combine
        "clocks": clk.summary(),
    }
    print(json.dumps(line))
    return 0


L2_BYTES = 129 << 20


def l2_flusher(dev, step_bytes: int):
    """A writer of 512 MB (4x the 129 MB L2) to run between timed steps when a step's
    working set is small enough to stay L2-resident, else None."""
    if step_bytes >= 4 * L2_BYTES:
        return None
    buf = torch.empty(512 << 18, dtype=torch.float32, device=dev)
    return lambda: buf.fill_(1.0)


def graph_step_ms(args, wl, s, e, dev, micro, stream, flush=None):
    """ms per step of the configuration's whole step replayed from a CUDA graph: a
    capturable optimizer (device step count), all micro-batches' grad passes with the
    fused norm on the last, finalize, prepare and AdamW captured once.  Returns (per
    replay after an L2 flush when `flush` is given, else back to back; back to back)."""
    from fsdp_sharded_mixed_flatparameter_gb300 import FlatShardAdamW
    opt = FlatShardAdamW(wl.numels, world_size=wl.world_size, rank=wl.rank, lr=wl.lr, betas=wl.betas, eps=wl.eps,
                         weight_decay=wl.weight_decay, max_norm=wl.max_norm,
                         grad_range="full" if wl.mode == "zero1" else "shard", device=dev,
                         lowp_dtype=W.torch_dtype(wl.lowp_dtype), master=W.master_init(wl, s, e, device=dev),
                         capturable=True)
    M = wl.micro_batches
    if wl.mode != "zero3":
        for m in micro:
            opt.device_table(m)  # device tables built before capture
    torch.cuda.synchronize(dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for j in range(M):
            if wl.mode == "zero3":
                opt.accum(micro[j], accumulate=j > 0, scale=1.0 / M, fuse_norm=j == M - 1)
            else:
                opt.flatten(micro[j], accumulate=j > 0, scale=1.0 / M, fuse_norm=j == M - 1)
        opt.launch_step()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):  # back to back
        graph.replay()
    b.record(stream)
    torch.cuda.synchronize(dev)
    b2b = a.elapsed_time(b) / args.steps
    ms = b2b
    if flush is not None:  # each replay timed alone, after an L2 flush outside its events
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for a, b in evs:
            flush()
            a.record(stream)
            graph.replay()
            b.record(stream)
        torch.cuda.synchronize(dev)
        ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    if not opt.finish_step().finite:
        raise RuntimeError("non-finite grad norm in the benchmark")
    return ms, b2b


def direct_step_ms(args, wl, opt, micro, tables, stream, flush=None) -> dict:
    """The same step with its last micro-batch never written to the fp32 grad: the
    earlier micro-batches' passes, then a norm pass over the last one (added on the fly
    to their sum, or alone without accumulation) that writes only the norm partials, and
    AdamW reading the last micro-batch through the tensor table (plus the sum).  Timed
    like the materialized step (per-step events after an L2 flush when `flush` is given)."""
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    M = wl.micro_batches
    span = opt.ghi - opt.glo
    if wl.mode == "zero3":
        last = (opt.device_flat_table(micro[-1]), 1, span, micro[-1].dtype, 0, span, opt.start - opt.glo)
    else:
        table, count, dt = tables[-1]
        last = (table, count, opt.total, dt, opt.glo, opt.ghi, opt.start)
    esize = W.torch_dtype(wl.grad_dtype).itemsize

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        for j in range(M - 1):
            if wl.mode == "zero3":
                opt.accum(micro[j], accumulate=j > 0, scale=1.0 / M, stream=stream)
            else:
                table, count, dt = tables[j]
                zs.zero_flatten_cast(table, count, opt.total, dt, opt.glo, opt.ghi, 1.0 / M, j > 0, opt.grad, None,
                                     None, stream)
        table, count, total, dt, lo, hi, sstart = last
        zs.zero_flatten_cast(table, count, total, dt, lo, hi, 1.0 / M, zs.NORM_OF_SUM if M > 1 else False,
                             opt.grad if M > 1 else None, None, opt.ws, stream)
        if ev is not None:
            ev[1].record(stream)
        zs.zero_grad_sqnorm_finalize(opt.ws, span, 0.0, opt.max_norm, opt.norm_buf, stream)
        if ev is not None:
            ev[2].record(stream)
        zs.zero_adamw_step_tensors(opt.master, opt.exp_avg, opt.exp_avg_sq, table, count, total, dt, sstart, 1.0 / M,
                                   opt.lowp, opt.lr, opt.betas[0], opt.betas[1], opt.eps, opt.weight_decay, opt.t + 1,
                                   opt.norm_buf, stream, acc=opt.shard_grad() if M > 1 else None)
        if ev is not None:
            ev[3].record(stream)
        if not opt.finish_step().finite:
            raise RuntimeError("non-finite grad norm in the benchmark")

    for _ in range(args.warmup):
        step()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for k in range(args.steps):
        if flush is not None:
            flush()
        step(evs[k])
    b.record(stream)
    torch.cuda.synchronize()
    ms = (a.elapsed_time(b) / args.steps if flush is None
          else statistics.mean(ev[0].elapsed_time(ev[3]) for ev in evs))
    t_grad = statistics.mean(ev[0].elapsed_time(ev[1]) for ev in evs)
    t_k4 = statistics.mean(ev[2].elapsed_time(ev[3]) for ev in evs)
    n = opt.n
    acc = 4 if M > 1 else 0
    # earlier passes: source read, fp32 sum written (first) or read and written (later); the norm pass
    # reads the last source and the sum; AdamW reads p, m, v, the grad (and the sum), writes p, m, v, lowp
    grad_bytes = (M - 1) * span * esize + 4 * span * max(0, 1 + 2 * (M - 2)) + span * (esize + acc)
    k4_bytes = n * (12 + esize + acc + 12 + 2)
    return {"ms_per_step": ms, "value": n / (ms / 1e3), "unit": UNIT,
            "kernels_ms": {"grad_passes_and_norm_pass": t_grad, "adamw_from_table": t_k4},
            "kernels_gbs": {"grad_passes_and_norm_pass": grad_bytes / (t_grad / 1e3) / 1e9,
                            "adamw_from_table": k4_bytes / (t_k4 / 1e3) / 1e9},
            "adamw_bytes_per_param": 12 + esize + acc + 12 + 2,
            "what": "the last micro-batch is never written to the fp32 grad: a norm pass "
                    + ("adds it to the earlier micro-batches' sum on the fly" if M > 1 else "reads it")
                    + " and writes only the norm partials, and AdamW reads it through the tensor table"
                    + (" and adds it to the sum" if M > 1 else "") + "; bit-identical to the materialized step"}


def run_config(args):
    """One configuration's whole step on one GPU (its micro-batches, fused norm on the
    last one, AdamW), inputs resident; prints one JSON line with the per-kernel split."""
    from fsdp_sharded_mixed_flatparameter_gb300 import FlatShardAdamW
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    wl = {**W.ALL, **W.VARIANTS}[args.workload]()
    if args.small:
        # profiling case: the same distribution on ~10x fewer parameters
        if wl.name.startswith("ragged"):
            wl = wl.with_(name=wl.name + "_2000", numels=tuple(W.ragged_numels(2000, seed=0)))
        elif wl.name.startswith("llama13b"):
            wl = wl.with_(name=wl.name + "_5l", numels=tuple(W.llama_numels(5, 5120, 13824, 32000)))
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    s, e = zs.zero_shard_range(wl.total, wl.world_size, wl.rank)
    n = e - s
    opt = FlatShardAdamW(wl.numels, world_size=wl.world_size, rank=wl.rank, lr=wl.lr, betas=wl.betas, eps=wl.eps,
                         weight_decay=wl.weight_decay, max_norm=wl.max_norm,
                         grad_range="full" if wl.mode == "zero1" else "shard", device=dev,
                         lowp_dtype=W.torch_dtype(wl.lowp_dtype), master=W.master_init(wl, s, e, device=dev))
    M = wl.micro_batches
    esize = W.torch_dtype(wl.grad_dtype).itemsize
    if wl.mode == "zero3":
        micro = [W.flat_grads(wl, 1, j, s, e, device=dev) for j in range(M)]
    else:
        micro = [W.tensor_grads(wl, 1, j, device=dev).tensors for j in range(M)]
    src_bytes = M * opt.grad.numel() * esize  # each pass reads the grad range's elements once
    stream = torch.cuda.current_stream(dev)

    tables = [] if wl.mode == "zero3" else [opt.device_table(m) for m in micro]  # built once, like registered grads

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        for j in range(M):
            if wl.mode == "zero3":
                opt.accum(micro[j], accumulate=j > 0, scale=1.0 / M, fuse_norm=j == M - 1, stream=stream)
            else:
                table, count, dt = tables[j]
                zs.zero_flatten_cast(table, count, opt.total, dt, opt.glo, opt.ghi, 1.0 / M, j > 0, opt.grad, None,
                                     opt.ws if j == M - 1 else None, stream)
        if ev is not None:
            ev[1].record(stream)
        zs.zero_grad_sqnorm_finalize(opt.ws, opt.grad.numel(), 0.0, opt.max_norm, opt.norm_buf, stream)
        if ev is not None:
            ev[2].record(stream)
        zs.zero_adamw_step(opt.master, opt.exp_avg, opt.exp_avg_sq, opt.shard_grad(), opt.lowp, opt.lr,
                           opt.betas[0], opt.betas[1], opt.eps, opt.weight_decay, opt.t + 1, opt.norm_buf, stream)
        if ev is not None:
            ev[3].record(stream)
        if not opt.finish_step().finite:
            raise RuntimeError("non-finite grad norm in the benchmark")

    # bytes one step touches: every grad pass and AdamW (the fp32 grad buffer is re-read by each pass)
    step_bytes = src_bytes + 4 * opt.grad.numel() * (2 * M) + ADAMW_BYTES_PER_PARAM * n
    flush = l2_flusher(dev, step_bytes)
    for _ in range(args.warmup):
        step()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    a.record(stream)
    for k in range(args.steps):
        if flush is not None:
            flush()
        step(evs[k])
    b.record(stream)
    torch.cuda.synchronize(dev)
    if flush is None:
        ms = a.elapsed_time(b) / args.steps
        eager_b2b = ms
    else:  # the step's own events (first grad pass to the end of AdamW), the flush outside them
        ms = statistics.mean(ev[0].elapsed_time(ev[3]) for ev in evs)
        a.record(stream)
        for k in range(args.steps):  # and back to back, host read of the norm after every step
            step()
        b.record(stream)
        torch.cuda.synchronize(dev)
        eager_b2b = a.elapsed_time(b) / args.steps
    t_grad = statistics.mean(ev[0].elapsed_time(ev[1]) for ev in evs)
    t_k4 = statistics.mean(ev[2].elapsed_time(ev[3]) for ev in evs)
    direct = direct_step_ms(args, wl, opt, micro, tables, stream, flush)
    graph_ms = graph_step_ms(args, wl, s, e, dev, micro, stream, flush) if n <= (1 << 31) else None
    peaks, _ = measured_peaks()
    grad_elems = opt.grad.numel()
    # grad passes: every micro-batch reads its source; the first writes the fp32 grad, later ones read+write it
    grad_bytes = src_bytes + 4 * grad_elems * (1 + 2 * (M - 1))
    line = {
        "metric": METRIC, "value": n / (ms / 1e3), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "params_per_rank": n, "tensors": wl.n_tensors, "world_size": wl.world_size,
                   "rank": wl.rank, "micro_batches": M, "grad_dtype": wl.grad_dtype, "mode": wl.mode,
                   "lowp_dtype": wl.lowp_dtype, "weight_decay": wl.weight_decay, "grad_buffer_elems": grad_elems,
                   "l2": (f"step touches {step_bytes / 1e6:.0f} MB < 4x L2: 512 MB written between timed steps, "
                          f"each step timed by its own events (first grad pass to the end of AdamW)"
                          if flush is not None else "inputs larger than L2; no flush")},
        "kernels_ms": {"flatten_or_accum_with_norm": t_grad, "adamw": t_k4},
        "kernels_gbs": {"flatten_or_accum_with_norm": grad_bytes / (t_grad / 1e3) / 1e9,
                        "adamw": ADAMW_BYTES_PER_PARAM * n / (t_k4 / 1e3) / 1e9},
        "adamw_frac_of_measured_hbm": ADAMW_BYTES_PER_PARAM * n / (t_k4 / 1e3) / 1e9 / float(peaks["hbm_gbs"]),
    }
    line["back_to_back_ms_per_step"] = eager_b2b  # steps launched one after another, norm read on the host each
    if graph_ms is not None:
        line["graph"] = {"ms_per_step": graph_ms[0], "value": n / (graph_ms[0] / 1e3), "unit": UNIT,
                         "back_to_back_ms_per_step": graph_ms[1],
                         "what": "the same step captured once in a CUDA graph (step count and skip decision on the "
                                 "device), no host work or device-to-host read per step; ms_per_step timed like the "
                                 "eager step, back_to_back_ms_per_step = replays one after another"}
    line["direct"] = direct
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_config_rates(wl)
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", default="llama7b_flat", choices=sorted({**W.ALL, **W.VARIANTS}),
                    help="another configuration's step (a table row, not the headline line)")
    ap.add_argument("--small", action="store_true",
                    help="profiling case for ncu (a smaller list of the same shape), not a bench line")
    ap.add_argument("--units", action="store_true",
                    help="Llama-7B as 34 FSDP units (one FlatParameter each) under one clip, one GPU")
    ap.add_argument("--dataplane-ranks", type=int, default=0,
                    help="with one process: time one rank of an N-rank ZeRO-2 Llama-7B job (reduce, norm, AdamW)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.workload != "llama7b_flat":
        return run_config(args)
    if args.units:
        return run_units(args)
    if args.gpus > 1 or args.dataplane_ranks > 1:
        return run_dataplane(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
