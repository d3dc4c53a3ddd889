"""Index arithmetic past 2^31 elements: a single bf16 tensor of 2^31 + 1000 elements
behind a 7-element tensor (so flat offsets are not multiples of 8 and its tiles take the
register-realigned path), shard ranges around element 2^31 of the tensor through the
flatten, the norm-only pass and AdamW through the table; and the reduction of two ranks'
blocks longer than 2^31 elements.  Every value is checked against the oracle over the
windows computed (the operations are element-wise; the norm windows are whole tiles)."""
import numpy as np
import pytest
import torch

import oracle
from _helpers import RTOL_NORM, bits_equal_f32, raw

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
BIG = (1 << 31) + 1000


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fsdp_sharded_mixed_flatparameter_gb300 import build, zero_shard
    build.build()
    zero_shard.lib()


def _fill_bf16(t: torch.Tensor, seed: int) -> None:
    g = torch.Generator(device=DEV)
    step = 1 << 28
    for a in range(0, t.numel(), step):
        g.manual_seed(seed + a)
        b = min(a + step, t.numel())
        t[a:b] = (torch.randn(b - a, generator=g, device=DEV) * 1e-3).to(torch.bfloat16)


def test_flatten_norm_and_table_adamw_past_2_31():
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    small = torch.arange(7, dtype=torch.float32, device=DEV).to(torch.bfloat16) * 1e-3
    big = torch.empty(BIG + 8, dtype=torch.bfloat16, device=DEV)[1:BIG + 1]  # element-, not 16-byte-aligned
    _fill_bf16(big, 11)
    numels = [7, BIG]
    table, total = zs.zero_tensor_table([small, big], numels)
    d_table = zs.device_table(table, 2, DEV)
    # shard ranges in flat coordinates: around big's element 2^31, and its end
    for s, e in ((7 + (1 << 31) - 40000, 7 + (1 << 31) + 900), (total - 70001, total)):
        n = e - s
        host_big = raw(big[s - 7:e - 7])
        ref = np.empty(n, np.float32)
        oracle.flatten([None, host_big], [0, n], "bf16", 0, n, 0.5, ref, accumulate=False)
        dst = torch.empty(n, device=DEV)
        ws = torch.empty(zs.zero_grad_sqnorm_workspace_bytes(n), dtype=torch.uint8, device=DEV)
        zs.zero_flatten_cast(d_table, 2, total, torch.bfloat16, s, e, 0.5, False, dst, None, ws)
        out_f = zs.new_norm_result(DEV)
        zs.zero_grad_sqnorm_finalize(ws, n, 0.0, 1.0, out_f)
        ws2 = torch.empty_like(ws)
        zs.zero_flatten_cast(d_table, 2, total, torch.bfloat16, s, e, 0.5, False, None, None, ws2)  # norm only
        out_n = zs.new_norm_result(DEV)
        zs.zero_grad_sqnorm_finalize(ws2, n, 0.0, 1.0, out_n)
        torch.cuda.synchronize()
        assert bits_equal_f32(raw(dst), ref), (s, e)
        assert bytes(out_f.cpu().numpy()) == bytes(out_n.cpu().numpy())
        cr = oracle.clip(oracle.sqnorm(ref), 0.0, 1.0)
        r = zs.decode_norm_result(out_f)
        assert abs(r.norm - cr.norm) <= RTOL_NORM * cr.norm
        # AdamW reading the grads through the table over the same shard
        p0 = torch.linspace(-0.02, 0.02, n, device=DEV)
        m = torch.zeros(n, device=DEV)
        v = torch.zeros(n, device=DEV)
        lowp = torch.empty(n, dtype=torch.bfloat16, device=DEV)
        st = oracle.new_state(raw(p0))
        zs.zero_adamw_step_tensors(p0, m, v, d_table, 2, total, torch.bfloat16, s, 0.5, lowp, 3e-4, 0.9, 0.95,
                                   1e-8, 0.1, 1, out_f)
        sc = oracle.adamw_scalars(3e-4, 0.9, 0.95, 1e-8, 0.1, 1)
        oracle.adamw(st.p, st.m, st.v, ref, sc, r.clip_coef, st.lowp)
        torch.cuda.synchronize()
        for got, want in ((p0, st.p), (m, st.m), (v, st.v)):
            assert bits_equal_f32(raw(got), want), (s, e)
        assert np.array_equal(raw(lowp), st.lowp)


def test_reduce_chunks_past_2_31():
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    n = (1 << 31) + 3000
    stride = n + 5  # odd stride: the element path for every block but the first
    chunks = torch.empty(2, stride, dtype=torch.bfloat16, device=DEV)
    _fill_bf16(chunks.view(-1), 21)
    acc = torch.empty(n, device=DEV)
    zs.zero_reduce_chunks(acc, chunks, n, 0.5, False)
    torch.cuda.synchronize()
    for a, b in ((0, 40000), ((1 << 31) - 20000, (1 << 31) + 2000), (n - 33000, n)):
        blocks = np.ascontiguousarray(raw(chunks[:, a:b]))
        ref = np.empty(b - a, np.float32)
        oracle.reduce_chunks(ref, blocks, "bf16", b - a, 0.5, False)
        assert bits_equal_f32(raw(acc[a:b]), ref), (a, b)
    del chunks
    # vector path: 32-byte aligned accumulator, 16-byte aligned blocks of n + 8 elements
    n2 = (1 << 31) + 4096
    chunks2 = torch.empty(2, n2 + 8, dtype=torch.bfloat16, device=DEV)
    _fill_bf16(chunks2.view(-1), 31)
    acc2 = torch.empty(n2, device=DEV)
    zs.zero_reduce_chunks(acc2, chunks2, n2, 0.5, False)
    torch.cuda.synchronize()
    for a, b in (((1 << 31) - 32768, n2), (0, 40000)):
        blocks = np.ascontiguousarray(raw(chunks2[:, a:b]))
        ref = np.empty(b - a, np.float32)
        oracle.reduce_chunks(ref, blocks, "bf16", b - a, 0.5, False)
        assert bits_equal_f32(raw(acc2[a:b]), ref), (a, b)
