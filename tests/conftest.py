import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size configuration, minutes of runtime")


def pytest_collection_modifyitems(config, items):
    # GPU tests without a GPU are skipped, never silently run on a CPU fallback
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


@pytest.fixture(autouse=True)
def _no_debug_violations(request):
    """Under the self-checking debug library (ZERO_SHARD_DEBUG=1) every GPU test must
    leave no recorded access violation (index out of its extent or misaligned vector)."""
    yield
    if os.environ.get("ZERO_SHARD_DEBUG") == "1" and "gpu" in request.keywords:
        from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
        rec = zs.zero_debug_errors(reset=True)
        assert rec.count == 0, f"debug build recorded access violations: {rec}"
