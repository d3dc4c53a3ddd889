"""bench.py's CPU legs without a GPU: the reference arm times exactly the passes it
reports, and the all-core oracle baseline computes the same step as the single-core one."""
import io
import json
import types
from contextlib import redirect_stdout

import numpy as np

import workloads as W


def test_oracle_step_rate_runs_exactly_the_requested_passes():
    import bench
    rate, tot, passes, el = bench.oracle_step_rate(W.llama7b(), 1 << 16, 0.0, 3)
    assert passes == 3 and tot == 1 << 16 and rate > 0 and el > 0


def test_reference_arm_reports_what_it_timed(monkeypatch):
    import bench
    monkeypatch.setattr(bench, "REFERENCE_SAMPLE", 1 << 16)
    args = types.SimpleNamespace(steps=4, warmup=2, gpus=1)
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(args) == 0
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 4 and line["warmup"] == 2
    assert line["config"]["sample_params"] == line["config"]["params_per_rank"] == 1 << 16
    assert line["config"]["workload_params"] == W.llama7b().total
    assert abs(line["value"] - (1 << 16) / (line["ms_per_step"] / 1e3)) <= 1e-6 * line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["cores"] == 1


def test_all_core_baseline_computes_the_single_core_step():
    """Same sample, same oracle functions on thread ranges: the state after one pass equals
    the single-threaded pass bit for bit (the norm's range sums are added exactly)."""
    import bench
    import oracle
    wl = W.llama7b()
    n = 1 << 15
    bench.oracle_step_rate_threads(wl, n, 4, 1)  # warms up and runs; no state exposed, so recompute here
    # recompute both ways on the same inputs
    numels, tot = [], 0
    for k in wl.numels:
        take = min(k, n - tot)
        if take <= 0:
            break
        numels.append(take)
        tot += take
    import torch
    g = torch.Generator().manual_seed(wl.seed)
    grads = [(torch.randn(k, generator=g) * wl.grad_std).to(torch.bfloat16).view(torch.int16).numpy()
             .view(np.uint16) for k in numels]
    flat1 = np.empty(tot, np.float32)
    oracle.flatten(grads, numels, "bf16", 0, tot, 1.0, flat1, accumulate=False)
    flat4 = np.empty(tot, np.float32)
    bounds = [tot * i // 4 for i in range(5)]
    for a, b in zip(bounds[:-1], bounds[1:]):
        oracle.flatten(grads, numels, "bf16", a, b, 1.0, flat4[a:b], accumulate=False)
    assert np.array_equal(flat1, flat4)
    import math
    sq1 = oracle.sqnorm(flat1)
    sq4 = math.fsum(oracle.sqnorm(flat4[a:b]) for a, b in zip(bounds[:-1], bounds[1:]))
    assert abs(sq1 - sq4) <= 1e-15 * sq1
