"""The self-checking debug library (built with -DZERO_DEBUG).

Each kernel checks every global-memory access site's index against its
extent and its address against its vector alignment, recording violations
instead of faulting.  Its reporting path is exercised by a self-test that
records a violation without touching memory, and the kernel, direct-path,
graph, AMP, multi-rank and data-plane suites run under it with a check after
every test that nothing was recorded.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _env():
    env = dict(os.environ)
    env["ZERO_SHARD_DEBUG"] = "1"
    return env


@pytest.fixture(scope="module", autouse=True)
def _libs():
    from fsdp_sharded_mixed_flatparameter_gb300 import build
    build.build(debug=True)


def test_release_library_has_no_debug_record():
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    if zs.debug_build_selected():
        pytest.skip("this process runs the debug library")
    with pytest.raises(zs.ZeroError):
        zs.zero_debug_errors()


def test_debug_selftest_is_reported():
    code = (
        "import torch\n"
        "from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs\n"
        "assert zs.library_path().endswith('libzeroshard_debug.so')\n"
        "zs.zero_debug_errors(reset=True)\n"
        "zs.zero_debug_selftest(4242); torch.cuda.synchronize()\n"
        "r = zs.zero_debug_errors(reset=True)\n"
        "assert (r.count, r.site, r.index, r.block) == (1, 999, 4242, 0), r\n"
        "assert zs.zero_debug_errors().count == 0\n"
        "print('ok')\n")
    p = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=_env(), capture_output=True, text=True,
                       timeout=600)
    assert p.returncode == 0 and "ok" in p.stdout, p.stdout + p.stderr


def test_kernel_suites_record_no_violation_under_the_debug_build():
    suites = ["tests/test_gpu_kernels.py", "tests/test_gpu_direct.py", "tests/test_gpu_graph.py",
              "tests/test_gpu_amp.py", "tests/test_gpu_multirank.py", "tests/test_gpu_dataplane.py",
              "tests/test_gpu_direct_accum.py"]
    # (the 2^32-pattern write-back check and the full-size data-plane rank run once, under the
    # release build: here they would only repeat the same kernel sites for a minute)
    p = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
                        "-k", "not exhaustive_through_adamw and not full_size"] + suites,
                       cwd=ROOT, env=_env(), capture_output=True, text=True, timeout=1800)
    assert p.returncode == 0, p.stdout[-4000:] + p.stderr[-2000:]
