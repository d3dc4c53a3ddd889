"""bench.py's N > 1 code path (the ZeRO-2 data-plane step) run as two ranks under
torchrun on one GPU: with fewer GPUs than ranks the ranks exchange through gloo on host
memory, so no kernel waits on another rank.  A check that the path runs and prints its
line, not a measurement (the line says so)."""
import json
import os
import socket
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_bench_two_ranks_on_one_gpu_runs_the_data_plane():
    from fsdp_sharded_mixed_flatparameter_gb300 import build
    build.build()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--gpus", "2", "--small",
           "--steps", "2", "--warmup", "3"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert p.returncode == 0, p.stdout[-3000:] + p.stderr[-3000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout  # rank 0 alone prints
    line = json.loads(lines[0])
    assert line["n_gpus"] == 2 and line["scaling"] == "strong" and "emulated" in line
    assert line["config"]["ranks"] == 2 and line["value"] > 0
    assert set(line["kernels_ms"]) == {"exchange", "reduce", "norm", "adamw", "all_gather"}
    assert line["e2e"]["h2d_bytes_per_step"] > 0
