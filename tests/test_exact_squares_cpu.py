"""The grad norm's exact-square shortcut, checked exhaustively on the CPU.

For 16-bit grads scaled by a power of two the norm-only pass skips the
rounding residual e = fma(y, y, -fl(y*y)) of each square and tests for
non-finite grads only where a thread's sum went non-finite.  Both rest on
IEEE-754 binary32 facts checked here:

* the residual rounds to a zero for y = fl(s * w), s a power of two
  (the square of a significand of at most 11 bits fits in 24 bits; where the
  square underflows the residual is at most half of the smallest subnormal);
* the same is false in general (a non-power-of-two scale), so the check can fail;
* an inf or NaN value leaves the double-float sum of squares non-finite.

The binary32 results are emulated in binary64, where the square of a binary32
value is exact and the binary64 -> binary32 cast rounds once to nearest even.
"""
import numpy as np
import pytest


def _all_bf16():
    return (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)


def _all_f16():
    return np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float32)


def _residual(y):
    """fl32(y*y - fl32(y*y)) for finite y whose square does not overflow: what the fma returns."""
    y64 = y.astype(np.float64)
    sq = y64 * y64                               # exact: at most 48 significant bits, in range
    with np.errstate(over="ignore"):
        p = sq.astype(np.float32)                # the binary32 product
    keep = np.isfinite(p)
    diff = sq[keep] - p[keep].astype(np.float64)  # exact (representable)
    return diff.astype(np.float32), keep


def _scaled(w, s):
    with np.errstate(over="ignore"):
        return (w * np.float32(s)).astype(np.float32)


@pytest.mark.parametrize("fmt", ["bf16", "f16"])
def test_square_residual_is_zero_for_power_of_two_scales(fmt):
    w = _all_bf16() if fmt == "bf16" else _all_f16()
    w = w[np.isfinite(w)]
    n_underflow = 0
    for k in range(-150, 128, 1):
        s = np.ldexp(np.float32(1.0), k)
        if not np.isfinite(s) or s == 0 or s < np.finfo(np.float32).tiny:
            continue  # normal powers of two only, as the launcher requires
        for sign in (1.0, -1.0):
            y = _scaled(w, sign * s)
            y = y[np.isfinite(y)]
            e, keep = _residual(y)
            assert not np.any(e != 0), (fmt, k, y[keep][e != 0][:4])
            yk = y[keep].astype(np.float64)
            n_underflow += int(np.count_nonzero((yk * yk < 2.0 ** -126) & (yk != 0)))
    assert n_underflow > 1000  # the underflow range was really exercised


def test_square_residual_is_not_zero_in_general():
    w = _all_bf16()
    w = w[np.isfinite(w) & (np.abs(w) > 1e-10) & (np.abs(w) < 1e10)]
    e, _ = _residual(_scaled(w, 1.0 / 3.0))
    assert np.count_nonzero(e) > 1000
    rng = np.random.default_rng(0)
    e, _ = _residual(rng.standard_normal(10000).astype(np.float32))
    assert np.count_nonzero(e) > 9000


def _df_sum_of_squares(x):
    """The exact-square accumulation of one lane, emulated in binary32: p = x*x,
    s = h + p with TwoSum's error into l (numpy float32 ops round like the kernel's)."""
    f = np.float32
    h, l = f(0), f(0)
    with np.errstate(over="ignore", invalid="ignore"):
        for v in x.astype(np.float32):
            p = f(v * v)
            s = f(h + p)
            bp = f(s - h)
            t = f(f(h - f(s - bp)) + f(p - bp))
            h, l = s, f(l + t)
    return h, l


def test_nonfinite_value_makes_the_sum_nonfinite():
    """The norm-only pass decides the non-finite flag only where a thread's sum went
    non-finite: an inf or NaN anywhere in the lane leaves h non-finite, however many
    finite values follow; a finite value whose square overflows does the same (so the
    flag itself comes from re-reading the values, not from the sum)."""
    rng = np.random.default_rng(3)
    bad_values = [np.inf, -np.inf, np.nan]
    for trial in range(300):
        x = (rng.standard_normal(64) * 10.0 ** rng.integers(-20, 10)).astype(np.float32)
        i = int(rng.integers(0, 64))
        x[i] = bad_values[trial % 3]
        h, _ = _df_sum_of_squares(x)
        assert not np.isfinite(h), (trial, i)
        x[i] = np.float32(1.0)
        h, _ = _df_sum_of_squares(x)
        assert np.isfinite(h), trial
    x = np.full(8, 1e-3, np.float32)
    x[3] = np.float32(2.0 ** 70)  # finite, square beyond binary32
    h, _ = _df_sum_of_squares(x)
    assert not np.isfinite(h)
