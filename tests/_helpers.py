"""Shared helpers of the GPU parity tests: tensor <-> numpy views, the
comparison bars, and host-built inputs for the C ABI."""
from __future__ import annotations

import ctypes
import math
from typing import Optional

import numpy as np
import torch

# Acceptance bars of the step (also what bench/smoke use).
RTOL_STATE = 1e-6     # fp32 master / exp_avg / exp_avg_sq, relative
ZERO_ATOL = 1e-36     # where the oracle's value is |x| < 1e-30
RTOL_NORM = 1e-5      # grad norm, relative
MAX_LOWP_ULP = 1      # bf16 / f16 parameter copy


def raw(t: Optional[torch.Tensor]) -> Optional[np.ndarray]:
    """Host numpy view of a tensor as the oracle takes it: f32 as float32,
    16-bit floats as their uint16 bit patterns."""
    if t is None:
        return None
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.float32:
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def rel_err(gpu: np.ndarray, ref: np.ndarray) -> float:
    gpu = np.asarray(gpu, np.float32)
    ref = np.asarray(ref, np.float32)
    ok = ~np.isnan(ref)
    big = ok & (np.abs(ref) >= 1e-30)
    e = np.abs(gpu[big].astype(np.float64) - ref[big]) / np.abs(ref[big].astype(np.float64))
    return float(e.max()) if e.size else 0.0


def assert_close_f32(gpu, ref, rtol: float = RTOL_STATE, name: str = "") -> None:
    gpu = np.asarray(gpu, np.float32)
    ref = np.asarray(ref, np.float32)
    assert gpu.shape == ref.shape, name
    nan_r = np.isnan(ref)
    assert np.array_equal(np.isnan(gpu), nan_r), f"{name}: NaN positions differ"
    ok = ~nan_r
    big = ok & (np.abs(ref) >= 1e-30)
    small = ok & ~big
    err = np.abs(gpu.astype(np.float64) - ref.astype(np.float64))
    if big.any():
        worst = float((err[big] / np.abs(ref[big].astype(np.float64))).max())
        assert worst <= rtol, f"{name}: max relative error {worst:.3g} > {rtol}"
    if small.any():
        assert float(err[small].max()) <= ZERO_ATOL, f"{name}: near-zero values differ"


def _ordered(bits: np.ndarray) -> np.ndarray:
    """Sign-magnitude 16-bit float patterns -> integers in value order."""
    b = bits.astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def assert_lowp_ulp(gpu_bits: np.ndarray, ref_bits: np.ndarray, max_ulp: int = MAX_LOWP_ULP, name: str = "") -> None:
    g = np.asarray(gpu_bits, np.uint16)
    r = np.asarray(ref_bits, np.uint16)
    nan_g = (g & 0x7FFF) > 0x7F80
    nan_r = (r & 0x7FFF) > 0x7F80
    assert np.array_equal(nan_g, nan_r), f"{name}: NaN positions differ"
    d = np.abs(_ordered(g[~nan_r]) - _ordered(r[~nan_r]))
    if d.size:
        assert int(d.max()) <= max_ulp, f"{name}: {int(d.max())} ulp apart"


def assert_lowp_ulp_f16(gpu_bits, ref_bits, max_ulp: int = MAX_LOWP_ULP, name: str = "") -> None:
    g = np.asarray(gpu_bits, np.uint16)
    r = np.asarray(ref_bits, np.uint16)
    nan_g = (g & 0x7FFF) > 0x7C00
    nan_r = (r & 0x7FFF) > 0x7C00
    assert np.array_equal(nan_g, nan_r), f"{name}: NaN positions differ"
    d = np.abs(_ordered(g[~nan_r]) - _ordered(r[~nan_r]))
    if d.size:
        assert int(d.max()) <= max_ulp, f"{name}: {int(d.max())} ulp apart"


def bits_equal_f32(a: np.ndarray, b: np.ndarray) -> bool:
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    na, nb = np.isnan(a), np.isnan(b)
    return bool(np.array_equal(na, nb) and np.array_equal(a[~na].view(np.uint32), b[~nb].view(np.uint32)))


def norm_result_tensor(device, norm: float = 1.0, coef: float = 1.0, finite: bool = True) -> torch.Tensor:
    """A zero_norm_result built on the host (an input chosen by the test)."""
    from fsdp_sharded_mixed_flatparameter_gb300.zero_shard import zero_norm_result
    r = zero_norm_result(norm * norm, norm, coef, 1 if finite else 0)
    return torch.frombuffer(bytearray(bytes(r)), dtype=torch.uint8).to(device)


def offset_view(n: int, dtype: torch.dtype, offset: int, device, fill: Optional[torch.Tensor] = None) -> torch.Tensor:
    """A length-n view that starts `offset` elements into a fresh allocation."""
    base = torch.empty(n + offset + 16, dtype=dtype, device=device)
    v = base[offset:offset + n]
    if fill is not None:
        v.copy_(fill)
    return v
