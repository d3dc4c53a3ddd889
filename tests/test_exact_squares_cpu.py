"""The grad norm's exact-square shortcut, checked exhaustively on the CPU.

For 16-bit grads scaled by a power of two the norm kernels skip the
rounding residual e = fma(y, y, -fl(y*y)) of each square and use a packed
fma y*0 + z as the non-finite probe.  Both rest on IEEE-754 binary32 facts
checked here over every bf16 and f16 value:

* the residual rounds to a zero for y = fl(s * w), s a power of two
  (the square of a significand of at most 11 bits fits in 24 bits; where the
  square underflows the residual is at most half of the smallest subnormal);
* the same is false in general (a non-power-of-two scale), so the check can fail;
* y*0 + (+0) is a zero for finite y and NaN for inf/NaN.

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


def test_zero_probe_flags_exactly_the_nonfinite_values():
    y = _all_bf16()
    with np.errstate(invalid="ignore"):
        z = y * np.float32(0.0) + np.float32(0.0)
    assert np.array_equal(np.isnan(z), ~np.isfinite(y))
    assert np.all(z[np.isfinite(y)] == 0)
