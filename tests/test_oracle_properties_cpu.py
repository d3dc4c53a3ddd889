"""Randomised properties of the oracle (hypothesis), beside the fixed pins: random
tensor lists, shard cuts, dtypes, scales and hyper-parameters.  Skipped where
hypothesis is not installed."""
import math

import numpy as np
import pytest
import torch

import oracle

hyp = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

SETTINGS = settings(max_examples=60, deadline=None)


@SETTINGS
@given(total=st.integers(0, 10 ** 12), world=st.integers(1, 257))
def test_shard_ranges_partition_the_buffer(total, world):
    chunk = -(-total // world)
    prev_end = 0
    for rank in sorted({0, world - 1, world // 2, min(world - 1, 3)}):
        s, e = oracle.shard_range(total, world, rank)
        assert 0 <= s <= e <= total and e - s <= chunk
        assert s == min(rank * chunk, total)
    # adjacent ranks tile the buffer
    for rank in range(min(world, 40)):
        s, e = oracle.shard_range(total, world, rank)
        assert s == prev_end or s == total
        prev_end = e


@SETTINGS
@given(data=st.data(), dtype=st.sampled_from(["f32", "bf16", "f16"]),
       scale=st.sampled_from([1.0, 0.5, 0.125, 0.3, 4.0]))
def test_flatten_matches_torch_cat_slice(data, dtype, scale):
    numels = data.draw(st.lists(st.integers(0, 300), min_size=1, max_size=12))
    total = sum(numels)
    s = data.draw(st.integers(0, total))
    e = data.draw(st.integers(s, total))
    null = data.draw(st.sets(st.integers(0, len(numels) - 1), max_size=3))
    g = torch.Generator().manual_seed(data.draw(st.integers(0, 2 ** 31 - 1)))
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[dtype]
    ts = [None if i in null else (torch.randn(n, generator=g) * 3).to(tdt) for i, n in enumerate(numels)]
    raw = [None if t is None else (t.numpy() if dtype == "f32" else t.view(torch.int16).numpy().view(np.uint16))
           for t in ts]
    dst = np.zeros(max(e - s, 1), np.float32)[: e - s]
    oracle.flatten(raw, numels, dtype, s, e, scale, dst, accumulate=False)
    full = torch.cat([torch.zeros(n) if t is None else t.float() for t, n in zip(ts, numels)]) if numels else torch.zeros(0)
    ref = (full[s:e] * torch.tensor(scale, dtype=torch.float32)).numpy()
    assert np.array_equal(dst.view(np.uint32), ref.view(np.uint32))


@SETTINGS
@given(seed=st.integers(0, 2 ** 31 - 1), n=st.integers(1, 2000), m=st.sampled_from([2, 4, 8]))
def test_accumulation_equivalence(seed, n, m):
    """sum_j fl(g_j / m) == fl(sum_j g_j) / m for power-of-two m (normal-range values)."""
    rng = np.random.default_rng(seed)
    gs = [(rng.standard_normal(n) * 1e-2).astype(np.float32) for _ in range(m)]
    acc = np.zeros(n, np.float32)
    for j, g in enumerate(gs):
        oracle.accum(acc, g, "f32", 1.0 / m, accumulate=j > 0)
    direct = np.zeros(n, np.float32)
    for j, g in enumerate(gs):
        oracle.accum(direct, g, "f32", 1.0, accumulate=j > 0)
    assert np.array_equal(acc, (direct * np.float32(1.0 / m)).astype(np.float32))


@SETTINGS
@given(seed=st.integers(0, 2 ** 31 - 1), lr=st.floats(1e-6, 1e-2), b1=st.floats(0.0, 0.99),
       b2=st.floats(0.5, 0.9999), wd=st.floats(0.0, 0.3))
def test_adamw_step1_closed_form(seed, lr, b1, b2, wd):
    """Step 1 from m = v = 0: p1 = p0 (1 - lr wd) - lr g / (|g| + eps), to a few binary32 roundings."""
    rng = np.random.default_rng(seed)
    n, eps = 257, 1e-8
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    st_ = oracle.new_state(p0)
    sc = oracle.adamw_scalars(lr, b1, b2, eps, wd, 1)
    oracle.adamw(st_.p, st_.m, st_.v, g, sc, 1.0, st_.lowp)
    ref = p0.astype(np.float64) * (1 - lr * wd) - lr * g / (np.abs(g.astype(np.float64)) + eps)
    upd = lr * np.abs(g) / (np.abs(g) + eps)
    assert np.all(np.abs(st_.p - ref) <= 4e-7 * np.abs(ref) + 4e-6 * upd + 1e-12)
    assert np.allclose(st_.m, (1 - b1) * g.astype(np.float64), rtol=1e-6, atol=0)


@SETTINGS
@given(seed=st.integers(0, 2 ** 31 - 1), n=st.integers(1, 5000), max_norm=st.floats(1e-3, 10.0))
def test_sqnorm_and_clip_vs_float64(seed, n, max_norm):
    rng = np.random.default_rng(seed)
    g = (rng.standard_normal(n) * 10.0 ** rng.integers(-6, 3)).astype(np.float32)
    sq = oracle.sqnorm(g)
    ref = math.fsum(float(x) * float(x) for x in g)
    assert abs(sq - ref) <= 1e-15 * ref
    cr = oracle.clip(sq, 0.0, max_norm)
    q = max_norm / (math.sqrt(ref) + 1e-6)
    assert cr.coef == (np.float32(q) if q < 1.0 else np.float32(1.0))


@SETTINGS
@given(data=st.data(), dtype=st.sampled_from(["f32", "bf16", "f16"]), log_world=st.integers(0, 4),
       accumulate=st.booleans())
def test_reduce_chunks_is_the_rank_order_sum_divided(data, dtype, log_world, accumulate):
    """For a power-of-two world size, the rank-order sum of the scaled blocks equals torch's
    float32 rank-order sum divided by the world size, on any block length, padding and
    starting accumulator (values kept away from subnormals)."""
    world = 1 << log_world
    n = data.draw(st.integers(0, 200))
    pad = data.draw(st.integers(0, 9))
    seed = data.draw(st.integers(0, 2 ** 31))
    rng = np.random.default_rng(seed)
    vals = (rng.standard_normal((world, n + pad)) * 10.0 ** rng.uniform(-3, 3)).astype(np.float32)
    if dtype == "f32":
        blocks = vals
        as_f32 = vals
    else:
        conv = oracle.bf16_rne if dtype == "bf16" else oracle.f16_rne
        blocks = np.stack([conv(v) for v in vals]).reshape(world, n + pad)
        as_f32 = np.stack([oracle.to_f32(b, dtype) for b in blocks]).reshape(world, n + pad)
    acc0 = (rng.standard_normal(max(n, 1)) * 10.0).astype(np.float32)
    got = acc0.copy()
    oracle.reduce_chunks(got, np.ascontiguousarray(blocks), dtype, n, 1.0 / world, accumulate)
    ref = torch.from_numpy(as_f32[0, :n].copy())
    for r in range(1, world):
        ref = ref + torch.from_numpy(as_f32[r, :n].copy())
    ref = ref / world
    if accumulate:  # the accumulator is added first, then each scaled block: compare that order directly
        ref = torch.from_numpy(acc0[:n].copy())
        for r in range(world):
            ref = ref + torch.from_numpy(as_f32[r, :n].copy()) * torch.tensor(1.0 / world, dtype=torch.float32)
    assert np.array_equal(got[:n], ref.numpy())
