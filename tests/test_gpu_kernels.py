"""GPU parity of each kernel against the CPU oracle, through the C ABI.

Adversarial cases: empty, 1, 7, 8, 9 elements, sizes spanning several tiles
with a ragged tail, every start alignment within a 32-byte line, source and
destination misaligned relative to each other, tensors without grad,
zero-size tensors, shard cuts inside tensors, non-finite values.  Every
buffer sits inside a larger allocation whose guard bands are checked after
the call.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from _helpers import (RTOL_NORM, assert_close_f32, assert_lowp_ulp, assert_lowp_ulp_f16, bits_equal_f32,
                      norm_result_tensor, raw)

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
GUARD = 40


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from fsdp_sharded_mixed_flatparameter_gb300 import build, zero_shard
    build.build()
    zero_shard.lib()
    torch.cuda.init()


class Guarded:
    """A device buffer at a chosen element offset inside a NaN-filled allocation."""

    def __init__(self, n, dtype, offset, fill: torch.Tensor = None):
        self.base = torch.empty(n + offset + GUARD, dtype=dtype, device=DEV)
        self.base.view(torch.uint8).fill_(0xFF)  # NaN pattern for float types
        self.offset, self.n = offset, n
        self.t = self.base[offset:offset + n]
        if fill is not None:
            self.t.copy_(fill.to(DEV))
        self.snap = self.base.clone()

    def check_guards(self):
        b, s = self.base.view(torch.uint8), self.snap.view(torch.uint8)
        es = self.base.element_size()
        lo, hi = self.offset * es, (self.offset + self.n) * es
        assert torch.equal(b[:lo], s[:lo]) and torch.equal(b[hi:], s[hi:]), "write outside the buffer"


def _rand(n, seed, std=1.0, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(n, generator=g) * std).to(dtype)


# ----------------------------------------------------------------- K4 AdamW
SIZES = [0, 1, 7, 8, 9, 31, 257, 4096 + 13, 100003]


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("lowp", [torch.bfloat16, torch.float16, None])
def test_adamw_matches_oracle_bit_exact(n, lowp):
    """Fused AdamW vs the oracle for 3 steps, each buffer at its own alignment.
    The kernel follows the oracle's rounding sequence, so the fp32 state is
    expected bit for bit; the bar (1e-6 relative, 1 ulp) is checked as well."""
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    rng = np.random.default_rng(n + 7)
    for trial, (po, mo, vo, go, lo) in enumerate([(0, 0, 0, 0, 0), (3, 3, 3, 3, 5), (5, 5, 5, 5, 2),
                                                    (1, 2, 3, 4, 1), (7, 7, 7, 7, 7)]):
        p0 = _rand(n, 10 + trial, 0.02)
        P = Guarded(n, torch.float32, po, p0)
        M = Guarded(n, torch.float32, mo, torch.zeros(n))
        V = Guarded(n, torch.float32, vo, torch.zeros(n))
        L = Guarded(n, lowp, lo) if lowp is not None else None
        st = oracle.new_state(p0.numpy())
        lr, b1, b2, eps, wd = 3e-4, 0.9, 0.95, 1e-8, 0.1
        for t in range(1, 4):
            g = _rand(n, 100 * t + trial, 10.0 ** rng.uniform(-6, -1))
            if n > 3:
                g[1] = 0.0
            G = Guarded(n, torch.float32, go, g)
            coef = float(np.float32(rng.uniform(0.2, 1.0)))
            clip = norm_result_tensor(DEV, norm=1.0 / coef, coef=coef)
            zs.zero_adamw_step(P.t, M.t, V.t, G.t, None if L is None else L.t, lr, b1, b2, eps, wd, t, clip)
            sc = oracle.adamw_scalars(lr, b1, b2, eps, wd, t)
            oracle.adamw(st.p, st.m, st.v, g.numpy(), sc, np.float32(coef), st.lowp,
                         "f16" if lowp == torch.float16 else "bf16")
        torch.cuda.synchronize()
        for B in (P, M, V) + ((L,) if L is not None else ()):
            B.check_guards()
        for name, B, ref in (("p", P, st.p), ("m", M, st.m), ("v", V, st.v)):
            got = raw(B.t)
            assert_close_f32(got, ref, name=f"{name} trial {trial}")
            assert bits_equal_f32(got, ref), f"{name} not bit-exact, trial {trial}"
        if L is not None:
            (assert_lowp_ulp_f16 if lowp == torch.float16 else assert_lowp_ulp)(raw(L.t), st.lowp, name="lowp")
            assert np.array_equal(raw(L.t), st.lowp), "low-precision copy not bit-exact"


def test_adamw_skips_on_nonfinite_norm():
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    n = 5000
    P = Guarded(n, torch.float32, 0, _rand(n, 1, 0.02))
    M = Guarded(n, torch.float32, 0, _rand(n, 2, 1e-3))
    V = Guarded(n, torch.float32, 0, _rand(n, 3, 1e-3) ** 2)
    L = Guarded(n, torch.bfloat16, 0)
    G = Guarded(n, torch.float32, 0, _rand(n, 4, 1e-3))
    before = [B.base.clone() for B in (P, M, V, L)]
    clip = norm_result_tensor(DEV, norm=math.inf, coef=0.0, finite=False)
    zs.zero_adamw_step(P.t, M.t, V.t, G.t, L.t, 1e-3, 0.9, 0.999, 1e-8, 0.01, 5, clip)
    torch.cuda.synchronize()
    for b, B in zip(before, (P, M, V, L)):
        assert torch.equal(b.view(torch.uint8), B.base.view(torch.uint8))


def test_adamw_without_clip_and_special_values():
    """No clip result (coefficient 1); inf/NaN/huge grads propagate as in the oracle."""
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    n = 1000
    g = _rand(n, 9, 1e-2)
    g[10], g[11], g[12], g[13] = math.inf, -math.inf, math.nan, 3e38
    p0 = _rand(n, 8, 0.02)
    p0[20] = 70000.0  # overflows f16 on the write-back
    P, M, V = (Guarded(n, torch.float32, 0, x) for x in (p0, torch.zeros(n), torch.zeros(n)))
    G = Guarded(n, torch.float32, 0, g)
    L = Guarded(n, torch.float16, 0)
    zs.zero_adamw_step(P.t, M.t, V.t, G.t, L.t, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1, None)
    st = oracle.new_state(p0.numpy())
    oracle.adamw(st.p, st.m, st.v, g.numpy(), oracle.adamw_scalars(1e-3, 0.9, 0.999, 1e-8, 0.0, 1), 1.0, st.lowp,
                 "f16")
    torch.cuda.synchronize()
    for B, ref in ((P, st.p), (M, st.m), (V, st.v)):
        assert bits_equal_f32(raw(B.t), ref)
    assert_lowp_ulp_f16(raw(L.t), st.lowp)


# --------------------------------------------------------------- K3 sqnorm
NORM_SIZES = [0, 1, 5, 32767, 32768, 32769, 3 * 32768 + 5, 1_000_003, 12_582_917]


@pytest.mark.parametrize("n", NORM_SIZES)
@pytest.mark.parametrize("offset", [0, 1])
def test_grad_sqnorm_matches_oracle(n, offset):
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    g = _rand(n, n % 1000 + offset, 1e-3) * torch.exp(torch.linspace(-8, 8, n)) if n else torch.zeros(0)
    G = Guarded(n, torch.float32, offset, g)
    ws = torch.empty(max(zs.zero_grad_sqnorm_workspace_bytes(n), 8), dtype=torch.uint8, device=DEV)
    out = zs.new_norm_result(DEV)
    for max_norm, extra in ((1.0, 0.0), (0.5, 2.5), (math.inf, 0.0)):
        zs.zero_grad_sqnorm(G.t, extra, max_norm, ws, out)
        r1 = zs.decode_norm_result(out)
        zs.zero_grad_sqnorm(G.t, extra, max_norm, ws, out)
        r2 = zs.decode_norm_result(out)
        assert r1 == r2, "not deterministic"
        cr = oracle.clip(oracle.sqnorm(g.numpy()), extra, max_norm)
        assert r1.finite and cr.finite
        if cr.norm == 0.0:
            assert r1.norm == 0.0
        else:
            assert abs(r1.norm - cr.norm) <= RTOL_NORM * cr.norm, (r1.norm, cr.norm)
            assert abs(r1.norm - cr.norm) <= 1e-12 * cr.norm  # the kernel's own error budget (double-float)
        assert abs(r1.clip_coef - cr.coef) <= RTOL_NORM * cr.coef
    G.check_guards()


def test_grad_sqnorm_closed_form_and_launch_independence():
    """All-equal c: sum of squares c^2 n exactly (c with few mantissa bits)."""
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    for n, c in ((32768 * 7 + 3, 0.75), (4_000_000, 3.0517578125e-05), (1, -1.5)):
        G = Guarded(n, torch.float32, 0, torch.full((n,), c))
        ws = torch.empty(zs.zero_grad_sqnorm_workspace_bytes(n), dtype=torch.uint8, device=DEV)
        out = zs.new_norm_result(DEV)
        zs.zero_grad_sqnorm(G.t, 0.0, math.inf, ws, out)
        r = zs.decode_norm_result(out)
        assert r.sqnorm == n * c * c and r.clip_coef == 1.0


def test_grad_sqnorm_nonfinite_and_empty():
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    n = 100000
    for bad in (math.inf, -math.inf, math.nan):
        g = _rand(n, 3, 1e-3)
        g[77777] = bad
        G = Guarded(n, torch.float32, 0, g)
        ws = torch.empty(zs.zero_grad_sqnorm_workspace_bytes(n), dtype=torch.uint8, device=DEV)
        out = zs.new_norm_result(DEV)
        zs.zero_grad_sqnorm(G.t, 0.0, 1.0, ws, out)
        assert not zs.decode_norm_result(out).finite
    out = zs.new_norm_result(DEV)
    zs.zero_grad_sqnorm(torch.zeros(0, device=DEV), 4.0, 1.0, None, out)
    r = zs.decode_norm_result(out)
    assert r.finite and r.norm == 2.0 and r.clip_coef == np.float32(1.0 / (2.0 + 1e-6))


# ---------------------------------------------------------------- K2 accum
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("n", [0, 1, 9, 1000, 262147])
def test_accum_matches_oracle_bit_exact(dtype, n):
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    tdt = W.torch_dtype(dtype)
    for ao, so in ((0, 0), (3, 3), (1, 6), (0, 5), (7, 0)):
        A = Guarded(n, torch.float32, ao)
        ref = np.zeros(n, np.float32)
        flag = torch.zeros(1, dtype=torch.int32, device=DEV)
        for j, scale in enumerate((0.125, 0.125, 1.0 / 3.0)):
            x = _rand(n, 50 * j + ao + so, 1e-3, tdt)
            S = Guarded(n, tdt, so, x)
            zs.zero_accum(A.t, S.t, scale, accumulate=j > 0, found_nonfinite=flag)
            oracle.accum(ref, raw(x), dtype, scale, accumulate=j > 0)
            S.check_guards()
        torch.cuda.synchronize()
        A.check_guards()
        assert bits_equal_f32(raw(A.t), ref), (ao, so)
        assert flag.item() == 0


def test_accum_flags_nonfinite():
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    n = 10007
    for where in (0, 5, 5000, n - 1):
        x = _rand(n, 1, 1e-3, torch.float16)
        x[where] = math.inf
        acc = torch.zeros(n, device=DEV)
        flag = torch.zeros(1, dtype=torch.int32, device=DEV)
        zs.zero_accum(acc, x.to(DEV), 0.125, False, flag)
        assert flag.item() == 1
    # a finite value that overflows once scaled is flagged too
    x = torch.full((100,), 3e38)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    zs.zero_accum(torch.zeros(100, device=DEV), x.to(DEV), 4.0, False, flag)
    assert flag.item() == 1


# -------------------------------------------------------------- K1 flatten
def _table_case(numels, dtype, null=(), seed=0, elem_offsets=None):
    """Per-tensor device grads: each tensor at its own element offset in its own allocation."""
    tdt = W.torch_dtype(dtype)
    host, dev = [], []
    g = torch.Generator().manual_seed(seed)
    for i, n in enumerate(numels):
        if i in null:
            host.append(None)
            dev.append(None)
            continue
        x = (torch.randn(n, generator=g) * 1e-2).to(tdt)
        off = 0 if elem_offsets is None else elem_offsets[i % len(elem_offsets)]
        base = torch.empty(n + off + 8, dtype=tdt, device=DEV)
        v = base[off:off + n]
        v.copy_(x.to(DEV))
        host.append(x)
        dev.append(v)
    return host, dev


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_flatten_ragged_matches_oracle_bit_exact(dtype):
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    numels = list(W.ragged_numels(300, seed=5, max_log2=14))
    numels[4] = 0
    numels[17] = 0
    numels[40] = 20000  # spans several 8192-element tiles
    host, dev = _table_case(numels, dtype, null=(2, 9, 40), seed=3, elem_offsets=[0, 1, 3, 8, 5])
    table, total = zs.zero_tensor_table(dev, numels)
    d_table = zs.device_table(table, len(numels), DEV)
    rawh = [raw(h) for h in host]
    for world, rank in ((1, 0), (4, 2), (7, 6), (3, 1), (16, 15)):
        s, e = oracle.shard_range(total, world, rank)
        for dst_off in (0, 1, 4):
            D = Guarded(e - s, torch.float32, dst_off)
            ref = np.zeros(e - s, np.float32)
            flag = torch.zeros(1, dtype=torch.int32, device=DEV)
            for j, scale in enumerate((0.125, 0.125, 1.0)):
                zs.zero_flatten_cast(d_table, len(numels), total, W.torch_dtype(dtype), s, e, scale, j > 0, D.t,
                                     flag)
                oracle.flatten(rawh, numels, dtype, s, e, scale, ref, accumulate=j > 0)
            torch.cuda.synchronize()
            D.check_guards()
            assert bits_equal_f32(raw(D.t), ref), (world, rank, dst_off)
            assert flag.item() == 0


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_flatten_big_misaligned_tensors(dtype):
    """Tensors spanning many 8192-element tiles whose sources are not co-aligned with the
    destination (every element offset 0..7): the 16-bit tiles inside a tensor are realigned
    in registers, the rest staged; bit for bit against the oracle, and the fused norm's
    partials equal to the separate norm kernel's over the written values."""
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    numels = [5, 40000, 3, 70001, 17, 30000, 9000, 1, 25000, 8208, 8217]
    host, dev = _table_case(numels, dtype, seed=9, elem_offsets=[0, 1, 2, 3, 5, 7, 6, 4])
    table, total = zs.zero_tensor_table(dev, numels)
    d_table = zs.device_table(table, len(numels), DEV)
    rawh = [raw(h) for h in host]
    for world, rank in ((1, 0), (3, 1), (5, 4)):
        s, e = oracle.shard_range(total, world, rank)
        D = Guarded(e - s, torch.float32, 0)
        ref = np.zeros(e - s, np.float32)
        flag = torch.zeros(1, dtype=torch.int32, device=DEV)
        ws = torch.empty(zs.zero_grad_sqnorm_workspace_bytes(e - s), dtype=torch.uint8, device=DEV)
        for j, scale in enumerate((0.25, 0.25, 0.5)):
            last = j == 2
            zs.zero_flatten_cast(d_table, len(numels), total, W.torch_dtype(dtype), s, e, scale, j > 0, D.t, flag,
                                 ws if last else None)
            oracle.flatten(rawh, numels, dtype, s, e, scale, ref, accumulate=j > 0)
        torch.cuda.synchronize()
        D.check_guards()
        assert bits_equal_f32(raw(D.t), ref), (world, rank)
        assert flag.item() == 0
        out_f, out_s = zs.new_norm_result(DEV), zs.new_norm_result(DEV)
        zs.zero_grad_sqnorm_finalize(ws, e - s, 0.0, 1.0, out_f)
        zs.zero_grad_sqnorm(D.t.clone(), 0.0, 1.0, torch.empty_like(ws), out_s)
        torch.cuda.synchronize()
        assert bytes(out_f.cpu().numpy()) == bytes(out_s.cpu().numpy()), (world, rank)


def test_flatten_big_aligned_tensors_fast_path():
    """Llama-shaped list (tensors aligned, tiles inside one tensor) vs torch.cat and the oracle."""
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    wl = W.small_llama(layers=2, hidden=256, mlp=688, vocab=1000)
    tg = W.tensor_grads(wl, 1, 0, device=DEV)
    table, total = zs.zero_tensor_table(tg.tensors, wl.numels)
    d_table = zs.device_table(table, wl.n_tensors, DEV)
    full = torch.cat([t.float() for t in tg.tensors])
    for world, rank in ((1, 0), (8, 3), (5, 4)):
        s, e = oracle.shard_range(total, world, rank)
        dst = torch.empty(e - s, device=DEV)
        zs.zero_flatten_cast(d_table, wl.n_tensors, total, torch.bfloat16, s, e, 1.0, False, dst)
        assert torch.equal(dst.view(torch.int32), full[s:e].view(torch.int32))


def test_flatten_flags_nonfinite():
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    numels = [100, 50000, 7]
    host, dev = _table_case(numels, "bf16", seed=1)
    dev[1][33333] = math.nan
    table, total = zs.zero_tensor_table(dev, numels)
    d_table = zs.device_table(table, 3, DEV)
    dst = torch.empty(total, device=DEV)
    flag = torch.zeros(1, dtype=torch.int32, device=DEV)
    zs.zero_flatten_cast(d_table, 3, total, torch.bfloat16, 0, 100 + 33333, 1.0, False, dst, flag)
    assert flag.item() == 0  # the NaN lies outside the range
    zs.zero_flatten_cast(d_table, 3, total, torch.bfloat16, 0, total, 1.0, False, dst, flag)
    assert flag.item() == 1


# ------------------------------------------------- fused norm (K1/K2 + finalize)
def _norm_pair(zs, buf, n, extra=0.0, max_norm=1.0, fused_ws=None):
    """Separate norm over `buf` and the finalize of `fused_ws`: (workspace, result) of each."""
    ws_s = torch.zeros(max(zs.zero_grad_sqnorm_workspace_bytes(n), 8), dtype=torch.uint8, device=DEV)
    out_s, out_f = zs.new_norm_result(DEV), zs.new_norm_result(DEV)
    zs.zero_grad_sqnorm(buf, extra, max_norm, ws_s, out_s)
    zs.zero_grad_sqnorm_finalize(fused_ws, n, extra, max_norm, out_f)
    return ws_s, zs.decode_norm_result(out_s), zs.decode_norm_result(out_f)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_flatten_fused_norm_equals_separate_norm(dtype):
    """The last micro-batch's flatten writes the same values and, bit for bit, the same
    norm partials as a separate norm pass over what it wrote."""
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    for numels, offs in ((list(W.ragged_numels(300, seed=7, max_log2=14)), [0, 1, 3, 8, 5]),
                         (list(W.llama_numels(2, 256, 688, 1000)), [0])):
        host, dev = _table_case(numels, dtype, null=(2,), seed=11, elem_offsets=offs)
        table, total = zs.zero_tensor_table(dev, numels)
        d_table = zs.device_table(table, len(numels), DEV)
        rawh = [raw(h) for h in host]
        for world, rank in ((1, 0), (3, 1), (8, 7)):
            s, e = oracle.shard_range(total, world, rank)
            n = e - s
            for dst_off in (0, 1):
                D = Guarded(n, torch.float32, dst_off)
                ws_f = torch.full((max(zs.zero_grad_sqnorm_workspace_bytes(n), 8),), 0xAB, dtype=torch.uint8,
                                  device=DEV)
                ref = np.zeros(n, np.float32)
                zs.zero_flatten_cast(d_table, len(numels), total, W.torch_dtype(dtype), s, e, 0.5, False, D.t)
                oracle.flatten(rawh, numels, dtype, s, e, 0.5, ref, accumulate=False)
                zs.zero_flatten_cast(d_table, len(numels), total, W.torch_dtype(dtype), s, e, 0.5, True, D.t,
                                     norm_ws=ws_f)
                oracle.flatten(rawh, numels, dtype, s, e, 0.5, ref, accumulate=True)
                torch.cuda.synchronize()
                D.check_guards()
                assert bits_equal_f32(raw(D.t), ref), (world, rank, dst_off)
                nb = zs.zero_grad_sqnorm_workspace_bytes(n)
                ws_s, r_s, r_f = _norm_pair(zs, D.t, n, fused_ws=ws_f)
                assert torch.equal(ws_f[:nb], ws_s[:nb]), "fused partials differ from the separate norm"
                assert r_f == r_s
                cr = oracle.clip(oracle.sqnorm(ref), 0.0, 1.0)
                assert abs(r_f.norm - cr.norm) <= 1e-12 * cr.norm


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("n", [1, 9, 32768, 32769, 262147, 1_000_003])
def test_accum_fused_norm_equals_separate_norm(dtype, n):
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    tdt = W.torch_dtype(dtype)
    for ao, so in ((0, 0), (3, 3), (0, 5)):
        A = Guarded(n, torch.float32, ao)
        ref = np.zeros(n, np.float32)
        ws_f = torch.full((zs.zero_grad_sqnorm_workspace_bytes(n),), 0xCD, dtype=torch.uint8, device=DEV)
        for j in range(3):
            x = _rand(n, 70 * j + ao + so, 1e-2, tdt)
            S = Guarded(n, tdt, so, x)
            last = j == 2
            zs.zero_accum(A.t, S.t, 0.125, accumulate=j > 0, norm_ws=ws_f if last else None)
            oracle.accum(ref, raw(x), dtype, 0.125, accumulate=j > 0)
        torch.cuda.synchronize()
        A.check_guards()
        assert bits_equal_f32(raw(A.t), ref), (ao, so)
        ws_s, r_s, r_f = _norm_pair(zs, A.t, n, extra=0.5, max_norm=0.25, fused_ws=ws_f)
        nb = zs.zero_grad_sqnorm_workspace_bytes(n)
        assert torch.equal(ws_f[:nb], ws_s[:nb]), (ao, so)
        assert r_f == r_s


def _spread_bits(n, dtype, rng):
    """16-bit patterns over most of the format's range: random sign, exponent and
    significand, subnormals and zeros included (squares from underflow to ~2^80)."""
    sign = rng.integers(0, 2, n).astype(np.uint16) << 15
    if dtype == "bf16":
        ex = rng.integers(0, 168, n).astype(np.uint16) << 7
        man = rng.integers(0, 128, n).astype(np.uint16)
    else:
        ex = rng.integers(0, 31, n).astype(np.uint16) << 10
        man = rng.integers(0, 1024, n).astype(np.uint16)
    return sign | ex | man


def _bits_tensors(numels, dtype, seed, elem_offsets=(0,)):
    rng = np.random.default_rng(seed)
    tdt = W.torch_dtype(dtype)
    host, dev = [], []
    for i, n in enumerate(numels):
        bits = _spread_bits(n, dtype, rng)
        x = torch.from_numpy(bits.view(np.int16).copy()).view(tdt)
        off = elem_offsets[i % len(elem_offsets)]
        base = torch.zeros(n + off + 8, dtype=tdt, device=DEV)
        base[off:off + n].copy_(x.to(DEV))
        host.append(x)
        dev.append(base[off:off + n])
    return host, dev


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_exact_square_norm_equals_separate_norm(dtype):
    """The norm-only pass over 16-bit grads with a power-of-two scale takes the
    exact-square path (no residual term, non-finite flag from the sum).  Its partials equal
    bit for bit those of the writing pass with the fused norm and of the separate norm
    over the written buffer, over values from underflowing squares to ~2^80; a
    non-power-of-two scale takes the general path and agrees the same way."""
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    tdt = W.torch_dtype(dtype)
    cases = ((list(W.llama_numels(2, 256, 688, 1000)), (0,)),                     # in-tensor tiles
             (list(W.ragged_numels(200, seed=9, max_log2=15)), (0, 1, 3, 8, 5)))  # staged tiles
    for numels, offs in cases:
        host, dev = _bits_tensors(numels, dtype, seed=len(numels), elem_offsets=offs)
        table, total = zs.zero_tensor_table(dev, numels)
        d_table = zs.device_table(table, len(numels), DEV)
        rawh = [raw(h) for h in host]
        for world, rank in ((1, 0), (3, 1)):
            s, e = oracle.shard_range(total, world, rank)
            n = e - s
            nb = zs.zero_grad_sqnorm_workspace_bytes(n)
            for scale in (1.0, 0.125, 2.0 ** -20, 4.0, 0.3):
                ref = np.zeros(n, np.float32)
                bad_ref = oracle.flatten(rawh, numels, dtype, s, e, scale, ref, accumulate=False)
                plain = torch.empty(n, device=DEV)
                fused = torch.empty(n, device=DEV)
                ws_a = torch.full((nb,), 0x5A, dtype=torch.uint8, device=DEV)
                ws_b = torch.full((nb,), 0xA5, dtype=torch.uint8, device=DEV)
                flags = torch.zeros(3, dtype=torch.int32, device=DEV)
                zs.zero_flatten_cast(d_table, len(numels), total, tdt, s, e, scale, False, plain, flags[0:1])
                zs.zero_flatten_cast(d_table, len(numels), total, tdt, s, e, scale, False, None, flags[1:2],
                                     norm_ws=ws_a)
                zs.zero_flatten_cast(d_table, len(numels), total, tdt, s, e, scale, False, fused, flags[2:3],
                                     norm_ws=ws_b)
                torch.cuda.synchronize()
                assert bits_equal_f32(raw(plain), ref) and torch.equal(plain.view(torch.int32),
                                                                       fused.view(torch.int32)), scale
                assert flags.tolist() == [int(bad_ref)] * 3, (scale, flags.tolist())
                ws_s, r_s, r_a = _norm_pair(zs, plain, n, fused_ws=ws_a)
                assert torch.equal(ws_a, ws_s[:nb]), (numels[:2], world, rank, scale)
                assert torch.equal(ws_b, ws_s[:nb]), (numels[:2], world, rank, scale)
                assert r_a == r_s
                if math.isfinite(r_s.norm):
                    cr = oracle.clip(oracle.sqnorm(ref), 0.0, 1.0)
                    assert abs(r_s.norm - cr.norm) <= 1e-12 * cr.norm


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_exact_square_norm_flags_nonfinite(dtype):
    """The exact-square path (flag decided from the sum, values re-read) raises the flag for inf and NaN grads,
    in in-tensor and boundary tiles alike, and only for them: a finite bf16 grad whose
    square overflows binary32 makes the norm non-finite without raising the flag."""
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    tdt = W.torch_dtype(dtype)
    numels = list(W.llama_numels(1, 1024, 2752, 2000))  # tensors large enough for K1n's exact-square path
    assert sum(numels) // len(numels) > 16 * 32768
    specials = [math.inf, -math.inf, math.nan] + ([2.0 ** 70] if dtype == "bf16" else [])
    for value in specials:
        # inside a tensor (vector tiles), in a norm tensor between two large ones and at the very
        # end (tiles with tensor boundaries: element by element)
        for where in ((0, 5000), (4, 40000), (1, 5000), (8, 100), (len(numels) - 1, numels[-1] - 1)):
            g = torch.Generator().manual_seed(3)
            host = [(torch.randn(n, generator=g) * 1e-2).to(tdt) for n in numels]
            host[where[0]][where[1]] = value
            dev = [h.to(DEV) for h in host]
            table, total = zs.zero_tensor_table(dev, numels)
            d_table = zs.device_table(table, len(numels), DEV)
            nb = zs.zero_grad_sqnorm_workspace_bytes(total)
            ws = torch.zeros(nb, dtype=torch.uint8, device=DEV)
            flag = torch.zeros(1, dtype=torch.int32, device=DEV)
            zs.zero_flatten_cast(d_table, len(numels), total, tdt, 0, total, 1.0, False, None, flag, norm_ws=ws)
            out = zs.new_norm_result(DEV)
            zs.zero_grad_sqnorm_finalize(ws, total, 0.0, 1.0, out)
            r = zs.decode_norm_result(out)
            ref = np.zeros(total, np.float32)
            bad_ref = oracle.flatten([raw(h) for h in host], numels, dtype, 0, total, 1.0, ref, accumulate=False)
            assert flag.item() == int(bad_ref) == int(not math.isfinite(value)), (value, where)
            assert not math.isfinite(r.norm) and not r.finite, (value, where)


def test_flatten_reads_pinned_host_grads():
    """Grads in pinned host memory: the flatten kernel reads them over the host link
    (transfer and flatten in one pass), bit for bit as from device memory."""
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    numels = list(W.ragged_numels(120, seed=9, max_log2=15))
    host, _ = _table_case(numels, "bf16", null=(4,), seed=2)
    pinned = [None if h is None else h.pin_memory() for h in host]
    table, total = zs.zero_tensor_table(pinned, numels)
    d_table = zs.device_table(table, len(numels), DEV)
    s, e = oracle.shard_range(total, 3, 1)
    dst = torch.empty(e - s, device=DEV)
    ws = torch.empty(zs.zero_grad_sqnorm_workspace_bytes(e - s), dtype=torch.uint8, device=DEV)
    zs.zero_flatten_cast(d_table, len(numels), total, torch.bfloat16, s, e, 1.0, False, dst, norm_ws=ws)
    ref = np.zeros(e - s, np.float32)
    oracle.flatten([raw(h) for h in host], numels, "bf16", s, e, 1.0, ref, accumulate=False)
    torch.cuda.synchronize()
    assert bits_equal_f32(raw(dst), ref)
    with pytest.raises(ValueError):
        zs.zero_tensor_table([torch.zeros(4, dtype=torch.bfloat16)], [4])  # pageable host memory is refused


@pytest.mark.parametrize("lowp", [torch.bfloat16, torch.float16])
def test_lowp_writeback_exhaustive_through_adamw(lowp):
    """The AdamW kernel's low-precision write-back over every one of the 2^32 binary32
    patterns: with lr = 0, weight decay 0 and zero grads the update leaves p as it is
    (p*1 - 0*0), so the kernel writes round-to-nearest-even(p) for any p; compared with
    the oracle's rounding (NaN in, NaN out)."""
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    chunk = 1 << 30
    zeros = torch.zeros(chunk, device=DEV)
    m, v, g = zeros.clone(), zeros.clone(), zeros
    out = torch.empty(chunk, dtype=lowp, device=DEV)
    base = np.arange(chunk, dtype=np.uint32)
    bits = np.empty(chunk, dtype=np.uint32)
    ref = np.empty(chunk, dtype=np.uint16)
    rne = oracle.bf16_rne if lowp == torch.bfloat16 else oracle.f16_rne
    expo = 0x7F80 if lowp == torch.bfloat16 else 0x7C00
    for lo in range(0, 1 << 32, chunk):
        np.add(base, np.uint32(lo), out=bits)
        p = torch.from_numpy(bits.view(np.float32)).to(DEV)
        m.zero_()
        v.zero_()
        zs.zero_adamw_step(p, m, v, g, out, 0.0, 0.9, 0.999, 1e-8, 0.0, 1)
        got = out.view(torch.int16).cpu().numpy().view(np.uint16)
        rne(bits.view(np.float32), out=ref)
        nan = ((bits >> 23) & 0xFF) == 0xFF
        nan &= (bits & 0x7FFFFF) != 0
        assert np.array_equal(got[~nan], ref[~nan]), lo
        gn = got[nan]
        assert np.all((gn & expo) == expo) and np.all((gn & (0x7FFF ^ expo)) != 0), lo
        assert np.array_equal(p.view(torch.int32).cpu().numpy().view(np.uint32)[~nan], bits[~nan]), lo  # p kept


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_cast_and_exact_square_norm_exhaustive_over_16bit_patterns(dtype):
    """Every one of the 65,536 bf16 / f16 patterns through the flatten/cast (scales 1, 1/8, 4
    and 0.3, fresh and accumulating) and the flat accumulate, bit-exact against the oracle
    (NaN to NaN); and the exact-square norm path (norm-only, power-of-two scales) over every
    finite pattern below 2^40 gives the same partials as the general path's separate norm."""
    from fsdp_sharded_mixed_flatparameter_gb300 import zero_shard as zs
    tdt = W.torch_dtype(dtype)
    allbits = np.arange(1 << 16, dtype=np.uint16)
    x = torch.from_numpy(allbits.view(np.int16).copy()).view(tdt)
    xd = x.to(DEV)
    numels = [1 << 16]
    table, total = zs.zero_tensor_table([xd], numels)
    d_table = zs.device_table(table, 1, DEV)
    for scale in (1.0, 0.125, 4.0, 0.3):
        for acc_first in (False, True):
            ref = np.full(total, 0.5, np.float32)
            dst = torch.full((total,), 0.5, device=DEV)
            oracle.flatten([allbits], numels, dtype, 0, total, scale, ref, accumulate=acc_first)
            zs.zero_flatten_cast(d_table, 1, total, tdt, 0, total, scale, acc_first, dst)
            acc = torch.full((total,), 0.5, device=DEV)
            ref2 = np.full(total, 0.5, np.float32)
            oracle.accum(ref2, allbits, dtype, scale, accumulate=acc_first)
            zs.zero_accum(acc, xd, scale, acc_first)
            for got, want in ((raw(dst), ref), (raw(acc), ref2)):
                nan = np.isnan(want)
                assert np.array_equal(np.isnan(got), nan), (scale, acc_first)
                assert bits_equal_f32(got[~nan], want[~nan]), (scale, acc_first)
    # every finite pattern whose scaled square sums stay in binary32 range (|x| < 2^40:
    # all f16 values; bf16 below 2^40, the subnormals and both zeros included)
    expo = (allbits >> (7 if dtype == "bf16" else 10)) & (0xFF if dtype == "bf16" else 0x1F)
    finite = allbits[expo < (127 + 40 if dtype == "bf16" else 0x1F)]
    # several norm tiles, each element in different positions; one tensor of more than 16 norm
    # tiles, so that the norm-only pass takes K1n (whose exact-square path this checks)
    reps = np.tile(finite, -(-(17 * 32768) // finite.size))
    fd = torch.from_numpy(reps.view(np.int16).copy()).view(tdt).to(DEV)
    n = fd.numel()
    table, total = zs.zero_tensor_table([fd], [n])
    d_table = zs.device_table(table, 1, DEV)
    nb = zs.zero_grad_sqnorm_workspace_bytes(n)
    for scale in (1.0, 2.0 ** -12, 8.0):
        ws_exact = torch.full((nb,), 0x3C, dtype=torch.uint8, device=DEV)
        zs.zero_flatten_cast(d_table, 1, total, tdt, 0, total, scale, False, None, norm_ws=ws_exact)
        flat = torch.empty(n, device=DEV)
        zs.zero_flatten_cast(d_table, 1, total, tdt, 0, total, scale, False, flat)
        ws_s, r_s, r_e = _norm_pair(zs, flat, n, fused_ws=ws_exact)
        assert torch.equal(ws_exact, ws_s[:nb]), scale
        assert r_s == r_e
