"""zero_grad_sqnorm_noalloc: the grad norm for callers that cannot allocate.

Some callers cannot call cudaMalloc: their framework's pool owns all device
memory, or they run where the implicit synchronisation of an allocation is
not allowed.  For them the library keeps the norm's tile partials in its own
fixed device array.  This file checks, through the C ABI, that the entry
point gives exactly what the workspace version gives (the same kernels in
the same tile order, so the same bytes), and the oracle's norm within the
norm bar, on two calls in a row: a large call first, then a smaller one
that finds the large call's partials still in the shared array beyond its
own tile range and must not read them.  Sizes beyond the limit are refused.
It is collected last so that a run stopping at its first failure has
already run every other test; it passes alone in a fresh process as well.
"""
import ctypes

import numpy as np
import pytest
import torch

from _helpers import RTOL_NORM

LIMIT = (1 << 19) * 32768


def _lib():
    from fsdp_sharded_mixed_flatparameter_gb300 import build, zero_shard
    build.build()
    return zero_shard


def test_noalloc_rejects_sizes_beyond_the_limit():
    """Checked on the host before any CUDA call, so this runs without a GPU too."""
    zs = _lib()
    L = zs.lib()
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: the size check fails first
    assert L.zero_grad_sqnorm_noalloc(fake, LIMIT + 1, 0.0, 1.0, fake, None) == zs.ZERO_EINVAL
    assert b"limit" in L.zero_last_error()
    assert L.zero_grad_sqnorm_noalloc(fake, -1, 0.0, 1.0, fake, None) == zs.ZERO_EINVAL
    assert L.zero_grad_sqnorm_noalloc(fake, 10, 0.0, 1.0, None, None) == zs.ZERO_EINVAL


@pytest.mark.gpu
def test_noalloc_matches_workspace_version_two_calls_in_a_row():
    import oracle
    zs = _lib()
    L = zs.lib()
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev)
    # a large call first (92 tiles), then a smaller one (2 tiles) with other data and settings
    for n, seed, extra, max_norm in ((3_000_017, 1, 0.0, 1.0), (40_001, 2, 0.25, 0.5)):
        gen = torch.Generator().manual_seed(seed)
        host = (torch.randn(n, generator=gen) * 1e-3 * torch.exp(torch.linspace(-4, 4, n))).float()
        g = host.to(dev)
        # the workspace version's partials beyond this call's tiles are NaN bytes: reading them would show
        ws = torch.full((zs.zero_grad_sqnorm_workspace_bytes(4 * n),), 0xFF, dtype=torch.uint8, device=dev)
        ref_out = zs.new_norm_result(dev)
        zs.zero_grad_sqnorm(g, extra, max_norm, ws, ref_out, stream)
        out = zs.new_norm_result(dev)
        st = L.zero_grad_sqnorm_noalloc(ctypes.c_void_p(g.data_ptr()), n, extra, max_norm,
                                        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(stream.cuda_stream))
        assert st == zs.ZERO_OK, L.zero_last_error()
        torch.cuda.synchronize(dev)
        # same kernels, same tile order: the same bytes
        assert bytes(out.cpu().numpy()) == bytes(ref_out.cpu().numpy()), (n, zs.decode_norm_result(out),
                                                                          zs.decode_norm_result(ref_out))
        got = zs.decode_norm_result(out)
        assert got.finite
        ref = oracle.clip(oracle.sqnorm(np.ascontiguousarray(host.numpy())), extra, max_norm)
        assert abs(got.norm - ref.norm) <= RTOL_NORM * ref.norm, (n, got.norm, ref.norm)
        assert abs(got.clip_coef - ref.coef) <= RTOL_NORM * ref.coef, (n, got.clip_coef, ref.coef)
