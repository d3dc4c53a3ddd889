"""Pins of the CPU oracle against things other than itself (no GPU).

Each test ties one oracle function to a closed form, an invariant, a library
routine (torch / numpy) or a brute force in exact arithmetic, chosen so that a
plausible slip in the oracle (a dropped term, a wrong sign or index, a swapped
operand, a wrong rounding) fails at least one of them.
"""
import math
import os
import random
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def ulp32(x: float) -> float:
    x = abs(float(np.float32(x)))
    if x == 0.0:
        return float(np.finfo(np.float32).smallest_subnormal)
    return float(np.spacing(np.float32(x)))


# ------------------------------------------------------------------- A1 shard range
def test_shard_range_golden():
    """Hand-worked ranges (formula of ZeRO1Optimizer.__init__), incl. the empty-range reading."""
    with open(os.path.join(GOLDEN, "shard_ranges.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) >= 10
    for t, w, r, s, e in rows:
        assert oracle.shard_range(int(t), int(w), int(r)) == (int(s), int(e)), (t, w, r)


def test_shard_range_partition_bruteforce():
    """For every total <= 300 and world <= 17 the ranks' ranges are contiguous, in rank
    order, cover [0,total), never exceed ceil(total/world), and every rank before the
    tail holds exactly ceil(total/world) elements.  Those properties fix the partition."""
    for total in range(0, 301):
        for world in range(1, 18):
            chunk = -(-total // world)
            pos = 0
            seen_short = False
            for rank in range(world):
                s, e = oracle.shard_range(total, world, rank)
                assert s == pos and e >= s, (total, world, rank)
                assert e - s <= chunk
                if e - s < chunk:
                    seen_short = True
                else:
                    assert not seen_short, "a full shard after a short one"
                pos = e
            assert pos == total


def test_shard_range_invalid():
    for args in [(-1, 2, 0), (10, 0, 0), (10, 2, 2), (10, 2, -1)]:
        with pytest.raises(ValueError):
            oracle.shard_range(*args)


def test_shard_range_large_totals_no_overflow():
    # 13B-shaped total; rank * chunk needs 64-bit arithmetic
    t = W.llama13b_zero3().total
    assert t == 13015864320
    assert oracle.shard_range(t, 8, 7) == (11388881280, 13015864320)
    s, e = oracle.shard_range(2**62, 3, 2)
    assert e == 2**62 and s == 2 * (-(-(2**62) // 3))


# ------------------------------------------------------------------- A2 flat offsets
def test_flat_offsets_match_torch_cat():
    """Offsets are where each tensor lands in torch.cat of the flattened list."""
    rng = np.random.default_rng(1)
    numels = [int(x) for x in rng.integers(0, 50, size=40)]
    numels[3] = 0
    off = oracle.flat_offsets(numels)
    cat = torch.cat([torch.full((n,), i, dtype=torch.int64) for i, n in enumerate(numels)])
    assert off[-1] == cat.numel()
    for i, n in enumerate(numels):
        if n:
            idx = (cat == i).nonzero().flatten()
            assert idx[0].item() == off[i] and idx[-1].item() == off[i] + n - 1


def test_model_totals():
    assert W.gpt2_zero1().total == 124439808 and W.gpt2_zero1().n_tensors == 148
    assert W.llama7b().total == 6738415616 and W.llama7b().n_tensors == 291
    assert W.llama13b_zero3().total == 13015864320 and W.llama13b_zero3().n_tensors == 363
    assert W.tiny().total == 1261891 and W.tiny().total % 8 == 3
    assert int(oracle.flat_offsets(W.llama7b().numels)[-1]) == 6738415616


# ------------------------------------------------------------------ dtype decoding
def test_bf16_decode_exhaustive():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.to_f32(bits, "bf16")
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f16_decode_exhaustive():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.to_f32(bits, "f16")
    ref = bits.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _f32_patterns():
    hi = np.arange(65536, dtype=np.uint32) << 16
    lows = np.array([0x0000, 0x0001, 0x0FFF, 0x1000, 0x1001, 0x1FFF, 0x2000, 0x3000, 0x3001,
                     0x7FFF, 0x8000, 0x8001, 0xEFFF, 0xF000, 0xF001, 0xFFFF], dtype=np.uint32)
    pats = (hi[:, None] | lows[None, :]).ravel()
    rnd = np.random.default_rng(7).integers(0, 2**32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    return np.concatenate([pats, rnd]).view(np.float32)


def test_bf16_rne_vs_torch():
    """f32 -> bf16 round-to-nearest-even vs torch's .to(bfloat16), every high half x rounding cases."""
    x = _f32_patterns()
    ours = oracle.bf16_rne(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    # NaN stays NaN (quiet) and keeps its sign
    on = ours[nan]
    assert np.all((on & 0x7F80) == 0x7F80) and np.all((on & 0x007F) != 0)
    assert np.array_equal(on >> 15, (x[nan].view(np.uint32) >> 31).astype(np.uint16))


def test_f16_rne_vs_numpy():
    x = _f32_patterns()
    ours = oracle.f16_rne(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all((ours[nan] & 0x7C00) == 0x7C00) and np.all((ours[nan] & 0x03FF) != 0)


def test_rne_exhaustive_over_all_binary32_patterns():
    """Both roundings over every one of the 2^32 binary32 bit patterns, in chunks, against
    torch's conversions (.to(bfloat16), .to(float16): round to nearest even); NaN inputs
    give a NaN of the same sign."""
    chunk = 1 << 26
    base = np.arange(chunk, dtype=np.uint32)
    bits = np.empty(chunk, dtype=np.uint32)
    x = bits.view(np.float32)
    ours = np.empty(chunk, dtype=np.uint16)  # buffers reused across chunks
    neq = np.empty(chunk, dtype=bool)
    ref_t = {torch.bfloat16: torch.empty(chunk, dtype=torch.bfloat16), torch.float16: torch.empty(chunk, dtype=torch.float16)}
    for lo in range(0, 1 << 32, chunk):
        np.add(base, np.uint32(lo), out=bits)
        has_nan = (lo & 0x7FFFFFFF) + chunk > 0x7F800000  # the chunks that reach the NaN patterns
        for rne, tdt, expo, mant in ((oracle.bf16_rne, torch.bfloat16, 0x7F80, 0x007F),
                                     (oracle.f16_rne, torch.float16, 0x7C00, 0x03FF)):
            rne(x, out=ours)
            ref = ref_t[tdt].copy_(torch.from_numpy(x)).view(torch.int16).numpy().view(np.uint16)
            if not has_nan:
                assert not np.not_equal(ours, ref, out=neq).any(), (lo, tdt)
                continue
            nan = np.isnan(x)
            assert np.array_equal(ours[~nan], ref[~nan]), (lo, tdt)
            on = ours[nan]
            assert np.all((on & expo) == expo) and np.all((on & mant) != 0), (lo, tdt)
            assert np.array_equal(on >> 15, (bits[nan] >> 31).astype(np.uint16)), (lo, tdt)


# ---------------------------------------------------------- A3 flatten / cast
def _grads(numels, dtype, seed, null=()):
    g = torch.Generator().manual_seed(seed)
    dt = W.torch_dtype(dtype)
    out = []
    for i, n in enumerate(numels):
        out.append(None if i in null else (torch.randn(n, generator=g) * 1e-2).to(dt))
    return out


def _np_raw(t):
    if t is None:
        return None
    if t.dtype == torch.float32:
        return t.contiguous().numpy()
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_flatten_matches_torch_cat_slice(dtype):
    """dst = scale * cat([g.float().view(-1)])[s:e] with zeros for tensors without grad."""
    numels = [7, 1, 0, 33, 128, 5, 64, 3, 250, 9]
    grads = _grads(numels, dtype, seed=5, null=(5,))
    full = torch.cat([torch.zeros(n) if g is None else g.float().view(-1) for g, n in zip(grads, numels)])
    total = full.numel()
    raw = [_np_raw(g) for g in grads]
    for s, e in [(0, total), (3, 44), (40, 41), (41, 41), (100, 500), (0, 0), (total - 1, total)]:
        for scale in (1.0, 0.125, 3.0):
            dst = np.full(max(e - s, 1), np.nan, dtype=np.float32)
            oracle.flatten(raw, numels, dtype, s, e, scale, dst, accumulate=False)
            ref = (full[s:e] * scale).numpy()
            assert np.array_equal(dst[:e - s].view(np.uint32), ref.view(np.uint32)), (s, e, scale)
            # accumulate adds fl(scale*x) to what is there
            base = np.linspace(-1, 1, e - s, dtype=np.float32)
            dst2 = base.copy()
            oracle.flatten(raw, numels, dtype, s, e, scale, dst2, accumulate=True)
            ref2 = (torch.from_numpy(base) + full[s:e] * scale).numpy()
            assert np.array_equal(dst2.view(np.uint32), ref2.view(np.uint32))


def test_flatten_nonfinite_flag():
    numels = [4, 4]
    g = [np.zeros(4, np.float32), np.array([0, np.inf, 0, 0], np.float32)]
    dst = np.zeros(8, np.float32)
    assert oracle.flatten(g, numels, "f32", 0, 8, 1.0, dst, False)
    assert not oracle.flatten(g, numels, "f32", 0, 5, 1.0, dst, False)  # inf lies outside [0,5)
    # finite input that overflows once scaled is flagged too (GradScaler unscale semantics)
    g2 = [np.full(4, 3e38, np.float32), np.zeros(4, np.float32)]
    assert oracle.flatten(g2, numels, "f32", 0, 8, 4.0, dst, False)


# ----------------------------------------------------- A4 accumulate / average
def test_accumulation_equivalence_power_of_two_scale():
    """Sum over 8 micro-batches of fl(g_j / 8) equals fl(sum_j g_j) / 8 bit for bit
    (the gradient-accumulation page: grad(loss/8) summed 8 times is the mean grad)."""
    rng = np.random.default_rng(11)
    n, M = 5000, 8
    gs = [(rng.standard_normal(n) * 1e-3).astype(np.float32) for _ in range(M)]
    for dtype in ("f32", "bf16", "f16"):
        if dtype == "f32":
            raws = gs
        elif dtype == "bf16":
            raws = [oracle.bf16_rne(g) for g in gs]
        else:
            raws = [oracle.f16_rne(g) for g in gs]
        a = np.zeros(n, np.float32)
        b = np.zeros(n, np.float32)
        for j, r in enumerate(raws):
            oracle.accum(a, r, dtype, 1.0 / M, accumulate=j > 0)
            oracle.accum(b, r, dtype, 1.0, accumulate=j > 0)
        assert np.array_equal(a, b / np.float32(M)), dtype


def test_accum_vs_exact_fraction():
    """Each accumulated value is within M rounding errors of the exact rational sum."""
    rng = np.random.default_rng(12)
    n, M = 64, 6
    gs = [(rng.standard_normal(n) * 10 ** rng.uniform(-6, 2)).astype(np.float32) for _ in range(M)]
    scale = np.float32(1.0 / 3.0)  # not a power of two: products round
    acc = np.zeros(n, np.float32)
    for j, g in enumerate(gs):
        oracle.accum(acc, g, "f32", float(scale), accumulate=j > 0)
    for k in range(n):
        exact = sum(Fraction(float(scale)) * Fraction(float(g[k])) for g in gs)
        mag = sum(abs(Fraction(float(scale)) * Fraction(float(g[k]))) for g in gs)
        err = abs(Fraction(float(acc[k])) - exact)
        assert err <= mag * Fraction(2 * M, 2**24), k


def test_accum_first_overwrites():
    acc = np.full(10, 123.0, np.float32)
    src = np.arange(10, dtype=np.float32)
    oracle.accum(acc, src, "f32", 0.5, accumulate=False)
    assert np.array_equal(acc, src * np.float32(0.5))


# ------------------------------------------------ ZeRO-2/3 reduce-scatter (NEXT-2)
def _padded_rank_blocks(grads, world):
    """Rank q's received blocks: block r = rank r's flat grad over q's chunk (padded to world*chunk)."""
    total = grads[0].size
    chunk = -(-total // world)
    padded = [np.concatenate([g, np.zeros(world * chunk - total, g.dtype)]) for g in grads]
    return chunk, [np.ascontiguousarray(np.stack([p[q * chunk:(q + 1) * chunk] for p in padded])) for q in range(world)]


@pytest.mark.parametrize("world", [2, 4, 8])
@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_reduce_chunks_is_reduce_scatter_then_divide(world, dtype):
    """The ZeRO page's ZeRO-2 reduce_gradients: reduce_scatter_tensor(SUM) of the ranks'
    flat grads, then /= world_size.  Concatenating every rank's reduced chunk equals the
    ranks' grads summed in rank order by torch in float32, divided by world_size, bit for
    bit (scaling each term by the power of two 1/world first is exact)."""
    rng = np.random.default_rng(40 + world)
    total = 10_007  # not a multiple of any world size: a short last chunk
    g32 = [(rng.standard_normal(total) * 1e-3).astype(np.float32) for _ in range(world)]
    conv = {"f32": lambda x: x, "bf16": oracle.bf16_rne, "f16": oracle.f16_rne}[dtype]
    raws = [conv(g) for g in g32]
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[dtype]
    as_t = (lambda r: torch.from_numpy(r)) if dtype == "f32" else \
        (lambda r: torch.from_numpy(r.view(np.int16)).view(tdt))
    ref = as_t(raws[0]).float()
    for r in raws[1:]:
        ref = ref + as_t(r).float()  # one binary32 add per rank, rank order
    ref = (ref / world).numpy()
    chunk, blocks = _padded_rank_blocks(raws, world)
    got = []
    for q in range(world):
        s, e = oracle.shard_range(total, world, q)
        assert s == min(q * chunk, total)
        acc = np.full(max(e - s, 1), np.nan, np.float32)
        assert not oracle.reduce_chunks(acc, blocks[q], dtype, e - s, 1.0 / world, accumulate=False)
        got.append(acc[:e - s])
    assert np.array_equal(np.concatenate(got), ref)


def test_reduce_chunks_accumulate_and_rank_order():
    """accumulate adds every rank's scaled value to the existing accumulator in rank order
    (micro-batches reduced one after another); checked against torch float32 adds in that
    order, with values whose sums depend on the order."""
    rng = np.random.default_rng(5)
    n, world = 513, 3
    acc0 = (rng.standard_normal(n) * 1e3).astype(np.float32)
    blocks = np.ascontiguousarray(np.stack([(rng.standard_normal(n + 7) * 10.0 ** k).astype(np.float32)
                                            for k in (3, -4, 1)]))
    scale = 0.3  # not a power of two: every product rounds
    acc = acc0.copy()
    oracle.reduce_chunks(acc, blocks, "f32", n, scale, accumulate=True)
    ref = torch.from_numpy(acc0.copy())
    sc = torch.tensor(scale, dtype=torch.float32)
    for r in range(world):
        ref = ref + sc * torch.from_numpy(blocks[r, :n].copy())
    assert np.array_equal(acc, ref.numpy())
    rev = acc0.copy()
    oracle.reduce_chunks(rev, np.ascontiguousarray(blocks[::-1]), "f32", n, scale, accumulate=True)
    assert not np.array_equal(rev, acc), "a different rank order must give different bits here"


def test_reduce_chunks_vs_exact_fraction_and_padding():
    """Every value is within world rounding errors of the exact rational sum; the padding
    beyond n in every block (NaN here) is never read; an inf inside the range raises the flag."""
    rng = np.random.default_rng(6)
    n, world, stride = 48, 5, 53
    blocks = np.full((world, stride), np.nan, np.float32)
    blocks[:, :n] = (rng.standard_normal((world, n)) * 10.0 ** rng.uniform(-5, 2, (world, 1))).astype(np.float32)
    scale = np.float32(1.0 / 3.0)
    acc = np.zeros(n, np.float32)
    assert not oracle.reduce_chunks(acc, blocks, "f32", n, float(scale), accumulate=False)
    for k in range(n):
        terms = [Fraction(float(scale)) * Fraction(float(blocks[r, k])) for r in range(world)]
        err = abs(Fraction(float(acc[k])) - sum(terms))
        assert err <= sum(abs(t) for t in terms) * Fraction(2 * world, 2**24), k
    blocks[3, 7] = np.inf
    assert oracle.reduce_chunks(acc, blocks, "f32", n, float(scale), accumulate=False)


# ----------------------------------------------------------- A5 grad norm + clip
def test_sqnorm_closed_form_all_equal():
    """sum of n copies of c^2 is n*c^2 exactly when that is representable."""
    for c in (0.75, -1.5, 3.0517578125e-05, 1.0 + 2**-11):
        for n in (1, 7, 4096, 1 << 20):
            g = np.full(n, c, np.float32)
            assert oracle.sqnorm(g) == n * (c * c)


def test_sqnorm_vs_fraction_and_torch():
    rng = np.random.default_rng(3)
    for n in (1, 2, 17, 64):
        g = (rng.standard_normal(n) * 10 ** rng.uniform(-5, 3, size=n)).astype(np.float32)
        exact = sum(Fraction(float(x)) ** 2 for x in g)
        assert abs(Fraction(oracle.sqnorm(g)) - exact) <= exact * Fraction(1, 2**51)
    g = (rng.standard_normal(1 << 20) * 1e-3).astype(np.float32)
    ref = torch.linalg.vector_norm(torch.from_numpy(g).double()).item() ** 2
    assert abs(oracle.sqnorm(g) - ref) <= 1e-12 * ref


def test_sqnorm_nonfinite():
    g = np.ones(10, np.float32)
    g[3] = np.inf
    assert oracle.sqnorm(g) == math.inf
    g[5] = np.nan
    assert math.isnan(oracle.sqnorm(g))
    assert oracle.sqnorm(np.zeros(0, np.float32)) == 0.0


def test_clip_vs_torch_clip_grad_norm():
    """Norm and scaled grads match torch.nn.utils.clip_grad_norm_ (float64 params)."""
    rng = np.random.default_rng(4)
    for max_norm in (1.0, 0.5, 1e3, math.inf):
        shapes = [(17,), (5, 9), (300,)]
        gs = [(rng.standard_normal(s) * 0.2).astype(np.float32) for s in shapes]
        params = [torch.nn.Parameter(torch.zeros(s, dtype=torch.float64)) for s in shapes]
        for p, g in zip(params, gs):
            p.grad = torch.from_numpy(g.astype(np.float64))
        tn = torch.nn.utils.clip_grad_norm_(params, max_norm).item()
        flat = np.concatenate([g.ravel() for g in gs])
        cr = oracle.clip(oracle.sqnorm(flat), 0.0, max_norm)
        assert cr.finite and abs(cr.norm - tn) <= 1e-13 * tn
        ours = flat.astype(np.float64) * cr.coef
        theirs = torch.cat([p.grad.view(-1) for p in params]).numpy()
        assert np.allclose(ours, theirs, rtol=1e-7, atol=0), max_norm


def test_clip_edge_cases():
    # zero grads: no clipping
    assert oracle.clip(0.0, 0.0, 1.0).coef == 1.0
    # exactly at max_norm the +1e-6 guard still scales below one (as clip_grad_norm_ does)
    cr = oracle.clip(1.0, 0.0, 1.0)
    assert cr.coef == np.float32(1.0 / (1.0 + 1e-6)) and cr.coef < 1.0
    # below the threshold: coefficient exactly one
    assert oracle.clip(0.25, 0.0, 1.0).coef == 1.0
    # extra_sqnorm (other ranks' share) adds before the square root
    cr = oracle.clip(9.0, 16.0, 1.0)
    assert cr.norm == 5.0 and cr.coef == np.float32(1.0 / (5.0 + 1e-6))
    # non-finite norms are flagged (the step is skipped)
    assert not oracle.clip(math.inf, 0.0, 1.0).finite
    assert not oracle.clip(math.nan, 0.0, 1.0).finite
    # no clipping with max_norm = inf
    assert oracle.clip(1e30, 0.0, math.inf).coef == 1.0


# --------------------------------------------------------------- A6 AdamW
def test_adamw_step1_closed_form():
    """At t=1 bias correction gives m_hat = g, v_hat = g^2, so
    p1 = p0 (1 - lr wd) - lr g / (|g| + eps)  (to a few binary32 roundings)."""
    rng = np.random.default_rng(21)
    n = 4096
    lr, b1, b2, eps, wd = 3e-4, 0.9, 0.95, 1e-8, 0.1
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g = (rng.standard_normal(n) * 10 ** rng.uniform(-9, 0, size=n)).astype(np.float32)
    g[:16] = 0.0
    st = oracle.new_state(p0)
    sc = oracle.adamw_scalars(lr, b1, b2, eps, wd, 1)
    oracle.adamw(st.p, st.m, st.v, g, sc, 1.0, st.lowp)
    p0d, gd = p0.astype(np.float64), g.astype(np.float64)
    upd = -lr * gd / (np.abs(gd) + eps)
    closed = p0d * (1 - lr * wd) + upd
    for k in range(n):
        tol = 3 * ulp32(closed[k]) + 1e-6 * abs(upd[k])
        assert abs(st.p[k] - closed[k]) <= tol, (k, st.p[k], closed[k])
    # zero grad: the update is exactly zero, only the decay acts
    assert np.array_equal(st.p[:16], (p0[:16] * np.float32(1 - lr * wd)))
    # state after one step: m = (1-b1) g, v = (1-b2) g^2
    assert np.allclose(st.m, (1 - b1) * gd, rtol=2.5e-7, atol=0)
    assert np.allclose(st.v, (1 - b2) * gd * gd, rtol=4e-7, atol=1e-45)
    # the low-precision copy is the RNE of the new master
    assert np.array_equal(st.lowp, oracle.bf16_rne(st.p))


def _torch_reference(p0, grads, lr, betas, eps, wd, max_norm, adam_cls):
    p = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    opt = adam_cls([p], lr=lr, betas=betas, eps=eps, weight_decay=wd, foreach=False, fused=False)
    for g in grads:
        p.grad = torch.from_numpy(g.copy())
        if max_norm is not None:
            torch.nn.utils.clip_grad_norm_([p], max_norm)
        opt.step()
    st = opt.state[p]
    return p.detach().numpy(), st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()


@pytest.mark.parametrize("wd,max_norm", [(0.0, None), (0.1, None), (0.05, 0.5), (0.0, 1.0)])
def test_adamw_trajectory_vs_torch_optim(wd, max_norm):
    """10 steps of clip_grad_norm_ + AdamW (Adam when wd == 0) vs torch.optim, non-foreach, CPU."""
    rng = np.random.default_rng(31)
    n, T = 3000, 10
    lr, betas, eps = 1e-3, (0.9, 0.999), 1e-8
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    grads = [(rng.standard_normal(n) * 0.05).astype(np.float32) for _ in range(T)]
    cls = torch.optim.AdamW if wd > 0 else torch.optim.Adam
    tp, tm, tv = _torch_reference(p0, grads, lr, betas, eps, wd, max_norm, cls)
    st = oracle.new_state(p0)
    for g in grads:
        cr = oracle.step_reference(st, g, lr=lr, betas=betas, eps=eps, wd=wd,
                                   max_norm=math.inf if max_norm is None else max_norm)
        assert cr.finite
        if max_norm is not None:
            assert cr.coef < 1.0  # clipping active in these cases
    assert st.t == T
    # the two sides round differently (torch uses lerp_ for m, scalar step_size in
    # binary64), so the bound is a few binary32 roundings at the arrays' own scale
    for ours, ref in ((st.p, tp), (st.m, tm), (st.v, tv)):
        scale = float(np.abs(ref).max())
        assert np.all(np.abs(ours - ref) <= 1e-6 * np.abs(ref) + 1e-6 * scale)
        assert float(np.median(np.abs(ours - ref) / np.maximum(np.abs(ref), 1e-30))) < 2e-7


def test_adamw_vs_exact_arithmetic_small():
    """5 steps at n=48 against the same recurrence in exact rational arithmetic
    (sqrt taken in binary64), within a binary32 error budget."""
    rng = np.random.default_rng(41)
    n, T = 48, 5
    lr, b1, b2, eps, wd = 1e-2, 0.9, 0.99, 1e-6, 0.01
    p0 = (rng.standard_normal(n) * 0.5).astype(np.float32)
    grads = [(rng.standard_normal(n) * 0.1).astype(np.float32) for _ in range(T)]
    st = oracle.new_state(p0)
    P = [Fraction(float(x)) for x in p0]
    Mm = [Fraction(0)] * n
    V = [Fraction(0)] * n
    for t, g in enumerate(grads, start=1):
        sc = oracle.adamw_scalars(lr, b1, b2, eps, wd, t)
        oracle.adamw(st.p, st.m, st.v, g, sc, 1.0, st.lowp)
        bc1 = 1 - Fraction(b1) ** t
        bc2 = 1 - Fraction(b2) ** t
        for k in range(n):
            gk = Fraction(float(g[k]))
            P[k] = P[k] * (1 - Fraction(lr) * Fraction(wd))
            Mm[k] = Fraction(b1) * Mm[k] + (1 - Fraction(b1)) * gk
            V[k] = Fraction(b2) * V[k] + (1 - Fraction(b2)) * gk * gk
            d = Fraction(math.sqrt(float(V[k]))) / Fraction(math.sqrt(float(bc2))) + Fraction(eps)
            P[k] = P[k] - Fraction(lr) / bc1 * Mm[k] / d
    for k in range(n):
        assert abs(float(st.m[k]) - float(Mm[k])) <= 1e-6 * abs(float(Mm[k])) + 1e-30
        assert abs(float(st.v[k]) - float(V[k])) <= 2e-6 * abs(float(V[k])) + 1e-30
        assert abs(float(st.p[k]) - float(P[k])) <= 1e-6 * abs(float(P[k])) + 1e-9


def test_shard_slice_equivalence():
    """Concatenating every rank's update of its own range gives the N=1 update, bit for bit
    (the update is element-wise and independent, as the memory-ledger page notes)."""
    rng = np.random.default_rng(51)
    total = 1000003
    p0 = (rng.standard_normal(total) * 0.02).astype(np.float32)
    g = (rng.standard_normal(total) * 1e-3).astype(np.float32)
    sc = oracle.adamw_scalars(1e-4, 0.9, 0.999, 1e-8, 0.01, 3)
    full = oracle.new_state(p0)
    full.m[:] = (rng.standard_normal(total) * 1e-4).astype(np.float32)
    full.v[:] = (rng.standard_normal(total) * 1e-4).astype(np.float32) ** 2
    m0, v0 = full.m.copy(), full.v.copy()
    oracle.adamw(full.p, full.m, full.v, g, sc, np.float32(0.7), full.lowp)
    for world in (3, 8):
        parts = []
        for r in range(world):
            s, e = oracle.shard_range(total, world, r)
            st = oracle.StepState(p=p0[s:e].copy(), m=m0[s:e].copy(), v=v0[s:e].copy(),
                                  lowp=np.zeros(e - s, np.uint16))
            oracle.adamw(st.p, st.m, st.v, np.ascontiguousarray(g[s:e]), sc, np.float32(0.7), st.lowp)
            parts.append(st)
        for name in ("p", "m", "v", "lowp"):
            cat = np.concatenate([getattr(x, name) for x in parts])
            assert np.array_equal(cat, getattr(full, name)), (world, name)


def test_adamw_scalars_bias_correction():
    sc = oracle.adamw_scalars(3e-4, 0.9, 0.95, 1e-8, 0.1, 1)
    assert sc[0] == np.float32(3e-4 / 0.1) or abs(sc[0] - 3e-3) <= ulp32(3e-3)
    assert abs(sc[1] - math.sqrt(0.05)) <= ulp32(math.sqrt(0.05))
    assert sc[2] == np.float32(1 - 3e-5)
    sc = oracle.adamw_scalars(3e-4, 0.9, 0.95, 1e-8, 0.1, 100000)
    assert sc[0] == np.float32(3e-4) and sc[1] == np.float32(1.0)


def test_skip_on_nonfinite_norm_leaves_state():
    """A non-finite grad norm skips the step: state and step counter stay as they were."""
    p0 = np.linspace(-1, 1, 100, dtype=np.float32)
    st = oracle.new_state(p0)
    g = np.full(100, 1e-3, np.float32)
    oracle.step_reference(st, g, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, wd=0.0, max_norm=1.0)
    snap = (st.p.copy(), st.m.copy(), st.v.copy(), st.lowp.copy(), st.t)
    g2 = g.copy()
    g2[7] = np.nan
    cr = oracle.step_reference(st, g2, lr=1e-3, betas=(0.9, 0.999), eps=1e-8, wd=0.0, max_norm=1.0)
    assert not cr.finite
    for a, b in zip(snap[:4], (st.p, st.m, st.v, st.lowp)):
        assert np.array_equal(a, b)
    assert st.t == snap[4] == 1


def test_fp16_lowp_writeback():
    p0 = np.array([1.0, 65504.0, 70000.0, 1e-8, -3.0e-5], np.float32)
    st = oracle.new_state(p0)
    g = np.zeros_like(p0)
    sc = oracle.adamw_scalars(1e-3, 0.9, 0.999, 1e-8, 0.0, 1)
    oracle.adamw(st.p, st.m, st.v, g, sc, 1.0, st.lowp, lowp_dtype="f16")
    with np.errstate(over="ignore"):
        assert np.array_equal(st.lowp, st.p.astype(np.float16).view(np.uint16))


# ------------------------------------------------------- dynamic loss scale
@pytest.mark.parametrize("interval", [1, 3, 50])
def test_loss_scale_policy_vs_torch_gradscaler(interval):
    """The oracle's scale trajectory equals torch.amp.GradScaler's for random overflow patterns."""
    rng = np.random.default_rng(interval)
    found = [bool(x) for x in rng.random(300) < 0.15]
    gs = torch.amp.GradScaler("cpu", init_scale=2.0 ** 16, growth_factor=2.0, backoff_factor=0.5,
                              growth_interval=interval)
    p = torch.nn.Parameter(torch.zeros(2))
    opt = torch.optim.SGD([p], lr=0.0)
    ref = []
    for f in found:
        gs.scale(torch.tensor(1.0))
        p.grad = torch.full((2,), float("inf") if f else 1.0)
        gs.unscale_(opt)
        gs.step(opt)
        gs.update()
        ref.append(gs.get_scale())
    assert oracle.loss_scale_trajectory(found, 2.0 ** 16, 2.0, 0.5, interval) == ref


def test_unscale_folded_into_accumulation_is_exact():
    """Scaling each micro-batch by 1/(S*M) equals accumulating with 1/M and unscaling by 1/S afterwards
    (GradScaler.unscale_ after accumulation), bit for bit, for power-of-two S and M."""
    rng = np.random.default_rng(5)
    S, M, n = 2.0 ** 16, 8, 4000
    xs = [oracle.f16_rne((rng.standard_normal(n) * 1e-5 * S).astype(np.float32)) for _ in range(M)]
    a = np.zeros(n, np.float32)
    b = np.zeros(n, np.float32)
    for j, x in enumerate(xs):
        oracle.accum(a, x, "f16", 1.0 / (S * M), accumulate=j > 0)
        oracle.accum(b, x, "f16", 1.0 / M, accumulate=j > 0)
    assert np.array_equal(a, b * np.float32(1.0 / S))


# ------------------------------------------- configuration-scale cross-checks
def _close_at_scale(ours, ref):
    scale = float(np.abs(ref).max())
    assert np.all(np.abs(ours - ref) <= 1e-6 * np.abs(ref) + 1e-6 * scale)
    assert float(np.median(np.abs(ours - ref) / np.maximum(np.abs(ref), 1e-30))) < 2e-7


def test_tiny_config_vs_torch_adamw():
    """The tiny configuration at full size (4 fp32 tensors, 1,261,891 params, its
    hyper-parameters, 3 steps, its seeded inputs): the oracle's flatten + AdamW against
    torch.optim.AdamW (non-foreach) on the four tensors."""
    wl = W.tiny()
    s, e = oracle.shard_range(wl.total, 1, 0)
    p0 = W.master_init(wl, s, e).numpy()
    offs = oracle.flat_offsets(wl.numels)
    params = [torch.nn.Parameter(torch.from_numpy(p0[offs[i]:offs[i + 1]].copy())) for i in range(len(wl.numels))]
    opt = torch.optim.AdamW(params, lr=wl.lr, betas=wl.betas, eps=wl.eps, weight_decay=wl.weight_decay,
                            foreach=False, fused=False)
    st = oracle.new_state(p0)
    for t in range(1, wl.steps + 1):
        tg = W.tensor_grads(wl, t, 0, device="cpu")
        g = np.zeros(e - s, np.float32)
        oracle.flatten([x.numpy() for x in tg.tensors], wl.numels, "f32", s, e, 1.0, g, accumulate=False)
        assert np.array_equal(g, torch.cat(tg.tensors).numpy())
        cr = oracle.step_reference(st, g, lr=wl.lr, betas=wl.betas, eps=wl.eps, wd=wl.weight_decay,
                                   max_norm=wl.max_norm)
        assert cr.finite and cr.coef == 1.0
        for prm, x in zip(params, tg.tensors):
            prm.grad = x.clone()
        opt.step()
    for name, ours in (("p", st.p), ("m", st.m), ("v", st.v)):
        if name == "p":
            ref = torch.cat([x.detach() for x in params]).numpy()
        else:
            ref = torch.cat([opt.state[x]["exp_avg" if name == "m" else "exp_avg_sq"] for x in params]).numpy()
        _close_at_scale(ours, ref)


def test_gpt2_zero1_config_vs_torch_adamw_and_clip():
    """The GPT-2 ZeRO-1 configuration at full size (148 tensors, 124,439,808 params, rank 3
    of 8, bf16 grads averaged over 8 micro-batches, clip 1.0 on the whole buffer's norm),
    2 steps: the oracle's flatten/accumulate, global norm and shard update against torch --
    the flat averaged grad summed with torch ops, clip_grad_norm_ over the whole buffer,
    torch.optim.Adam (non-foreach) over it -- compared on rank 3's slice.

    clip_grad_norm_ runs on a float64 copy of the grad: torch's float32 CPU norm of these
    1.2e8 values is 1.3 % off (3.8929 against 3.9440), so its float32 result is no
    reference; the float64 one agrees with the oracle to ~1e-11."""
    wl = W.gpt2_zero1()
    s, e = oracle.shard_range(wl.total, wl.world_size, wl.rank)
    offs = oracle.flat_offsets(wl.numels)
    M = wl.micro_batches
    p_full = W.master_init(wl, 0, wl.total)
    prm = torch.nn.Parameter(p_full.clone())
    opt = torch.optim.Adam([prm], lr=wl.lr, betas=wl.betas, eps=wl.eps, weight_decay=0.0, foreach=False, fused=False)
    st = oracle.new_state(p_full[s:e].numpy())
    for t in range(1, 3):
        acc = np.zeros(wl.total, np.float32)
        ref = torch.zeros(wl.total)
        for j in range(M):
            tg = W.tensor_grads(wl, t, j, device="cpu")
            raw16 = [x.view(torch.int16).numpy().view(np.uint16) for x in tg.tensors]
            oracle.flatten(raw16, wl.numels, "bf16", 0, wl.total, 1.0 / M, acc, accumulate=j > 0)
            for i, x in enumerate(tg.tensors):
                ref[offs[i]:offs[i + 1]].add_(x.float().mul_(1.0 / M))
            del tg, raw16
        assert np.array_equal(acc, ref.numpy())  # power-of-two scale: the same sums bit for bit
        cr = oracle.step_reference(st, np.ascontiguousarray(acc[s:e]), lr=wl.lr, betas=wl.betas, eps=wl.eps,
                                   wd=wl.weight_decay, max_norm=wl.max_norm, norm_grad=acc)
        assert cr.finite and cr.coef < 1.0  # clipping is active in this configuration
        p64 = torch.nn.Parameter(torch.zeros(wl.total, dtype=torch.float64))
        p64.grad = ref.double()
        tn = torch.nn.utils.clip_grad_norm_([p64], wl.max_norm).item()
        del p64
        assert abs(tn - cr.norm) <= 1e-10 * cr.norm
        assert cr.coef == np.float32(wl.max_norm / (tn + 1e-6))
        prm.grad = ref.mul_(cr.coef)  # the clipped grad in float32, as the update applies it
        opt.step()
    _close_at_scale(st.p, prm.detach()[s:e].numpy())
    _close_at_scale(st.m, opt.state[prm]["exp_avg"][s:e].numpy())
    _close_at_scale(st.v, opt.state[prm]["exp_avg_sq"][s:e].numpy())
