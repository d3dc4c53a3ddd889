"""CPU oracle of the flat-shard optimizer step -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never uses it, and it
uses nothing of the CUDA library.

``oracle.c`` holds the arithmetic (single-threaded, binary32 op by op in the
pages' order, binary64 compensated sum for the grad norm); this module only
builds it with gcc and marshals numpy arrays into it.  ``step_reference``
composes the functions into one optimizer step the way the pages' training
loops do: flatten/accumulate -> clip_grad_norm_ -> AdamW step.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

F32, BF16, F16 = 0, 1, 2
DTYPE_CODE = {"f32": F32, "bf16": BF16, "f16": F16}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc, -O2, no fp contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-fPIC", "-shared",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            i64, i32, f32, f64, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_double, ctypes.c_void_p
            L.orc_shard_range.argtypes = [i64, i32, i32, ctypes.POINTER(i64), ctypes.POINTER(i64)]
            L.orc_shard_range.restype = ctypes.c_int
            L.orc_flat_offsets.argtypes = [vp, i32, vp]
            L.orc_flatten.argtypes = [vp, vp, i32, ctypes.c_int, i64, i64, f32, ctypes.c_int, vp, vp]
            L.orc_accum.argtypes = [vp, vp, ctypes.c_int, i64, f32, ctypes.c_int, vp]
            L.orc_reduce_chunks.argtypes = [vp, vp, ctypes.c_int, i32, i64, i64, f32, ctypes.c_int, vp]
            L.orc_sqnorm.argtypes = [vp, i64]
            L.orc_sqnorm.restype = f64
            L.orc_clip.argtypes = [f64, f64, f64, ctypes.POINTER(f64), ctypes.POINTER(f64),
                                   ctypes.POINTER(f32), ctypes.POINTER(i32)]
            L.orc_adamw_scalars.argtypes = [f64, f64, f64, f64, f64, i64, vp]
            L.orc_adamw.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, i64, vp, f32]
            L.orc_bf16_rne.argtypes = [f32]
            L.orc_bf16_rne.restype = ctypes.c_uint16
            L.orc_f16_rne.argtypes = [f32]
            L.orc_f16_rne.restype = ctypes.c_uint16
            L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
            L.orc_bf16_to_f32.restype = f32
            L.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
            L.orc_f16_to_f32.restype = f32
            for nm in ("orc_bf16_rne_array", "orc_f16_rne_array"):
                getattr(L, nm).argtypes = [vp, vp, i64]
            L.orc_to_f32_array.argtypes = [vp, ctypes.c_int, vp, i64]
            L.orc_loss_scale_update.argtypes = [ctypes.POINTER(f32), ctypes.POINTER(i32), i32, f64, f64, i32]
            _lib = L
    return _lib


def _p(a: Optional[np.ndarray]):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a: np.ndarray, dtype) -> np.ndarray:
    assert a.dtype == dtype and a.flags.c_contiguous, (a.dtype, dtype)
    return a


# ---------------------------------------------------------------- elementary
def shard_range(total: int, world: int, rank: int):
    s, e = ctypes.c_int64(), ctypes.c_int64()
    if lib().orc_shard_range(total, world, rank, ctypes.byref(s), ctypes.byref(e)) != 0:
        raise ValueError("invalid shard arguments")
    return s.value, e.value


def flat_offsets(numels: Sequence[int]) -> np.ndarray:
    nm = np.ascontiguousarray(np.asarray(numels, dtype=np.int64))
    out = np.zeros(len(nm) + 1, dtype=np.int64)
    lib().orc_flat_offsets(_p(nm), len(nm), _p(out))
    return out


def _raw(a: np.ndarray) -> np.ndarray:
    """bf16/f16 grads travel as uint16 bit patterns, f32 as float32."""
    assert a.dtype in (np.float32, np.uint16) and a.flags.c_contiguous
    return a


def flatten(srcs: Sequence[Optional[np.ndarray]], numels: Sequence[int], dtype: str, s: int, e: int,
            scale: float, dst: np.ndarray, accumulate: bool) -> bool:
    """dst[0:e-s] (+)= scale * flat(srcs)[s:e]; returns True if a non-finite value was met."""
    _c(dst, np.float32)
    assert dst.size >= e - s
    n = len(numels)
    ptrs = (ctypes.c_void_p * n)(*[None if x is None else _raw(x).ctypes.data for x in srcs])
    nm = np.ascontiguousarray(np.asarray(numels, dtype=np.int64))
    flag = np.zeros(1, dtype=np.int32)
    lib().orc_flatten(ptrs, _p(nm), n, DTYPE_CODE[dtype], s, e, scale, int(bool(accumulate)), _p(dst), _p(flag))
    return bool(flag[0])


def accum(acc: np.ndarray, src: np.ndarray, dtype: str, scale: float, accumulate: bool) -> bool:
    _c(acc, np.float32)
    _raw(src)
    assert src.size == acc.size
    flag = np.zeros(1, dtype=np.int32)
    lib().orc_accum(_p(acc), _p(src), DTYPE_CODE[dtype], acc.size, scale, int(bool(accumulate)), _p(flag))
    return bool(flag[0])


def reduce_chunks(acc: np.ndarray, chunks: np.ndarray, dtype: str, n: int, scale: float, accumulate: bool) -> bool:
    """acc[0:n] (+)= sum over r in rank order of scale * chunks[r, 0:n] (a 2-D array of
    n_chunks blocks); returns True if a non-finite scaled value was met."""
    _c(acc, np.float32)
    assert chunks.ndim == 2 and chunks.flags.c_contiguous and chunks.dtype in (np.float32, np.uint16)
    assert acc.size >= n and chunks.shape[1] >= n
    flag = np.zeros(1, dtype=np.int32)
    lib().orc_reduce_chunks(_p(acc), _p(chunks), DTYPE_CODE[dtype], chunks.shape[0], chunks.shape[1], n, scale,
                            int(bool(accumulate)), _p(flag))
    return bool(flag[0])


def sqnorm(g: np.ndarray) -> float:
    _c(g, np.float32)
    return lib().orc_sqnorm(_p(g), g.size)


@dataclass
class ClipResult:
    sqnorm: float
    norm: float
    coef: float     # binary32 value, as a Python float
    finite: bool


def clip(sq_local: float, extra_sqnorm: float, max_norm: float) -> ClipResult:
    sq, nv, cf, fin = ctypes.c_double(), ctypes.c_double(), ctypes.c_float(), ctypes.c_int32()
    lib().orc_clip(sq_local, extra_sqnorm, max_norm, ctypes.byref(sq), ctypes.byref(nv),
                   ctypes.byref(cf), ctypes.byref(fin))
    return ClipResult(sq.value, nv.value, cf.value, bool(fin.value))


def adamw_scalars(lr: float, beta1: float, beta2: float, eps: float, wd: float, t: int) -> np.ndarray:
    out = np.zeros(8, dtype=np.float32)
    lib().orc_adamw_scalars(lr, beta1, beta2, eps, wd, t, _p(out))
    return out


def adamw(p: np.ndarray, m: np.ndarray, v: np.ndarray, g: np.ndarray, scalars: np.ndarray, coef: float,
          lowp: Optional[np.ndarray] = None, lowp_dtype: str = "bf16") -> None:
    for a in (p, m, v, g):
        _c(a, np.float32)
    assert p.size == m.size == v.size == g.size
    if lowp is not None:
        _c(lowp, np.uint16)
        assert lowp.size == p.size
    _c(scalars, np.float32)
    lib().orc_adamw(_p(p), _p(m), _p(v), _p(g), _p(lowp), DTYPE_CODE[lowp_dtype], p.size, _p(scalars), coef)


def bf16_rne(x: np.ndarray, out: Optional[np.ndarray] = None) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint16) if out is None else _c(out, np.uint16)
    assert y.size == x.size
    lib().orc_bf16_rne_array(_p(x), _p(y), x.size)
    return y


def f16_rne(x: np.ndarray, out: Optional[np.ndarray] = None) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty(x.shape, dtype=np.uint16) if out is None else _c(out, np.uint16)
    assert y.size == x.size
    lib().orc_f16_rne_array(_p(x), _p(y), x.size)
    return y


def to_f32(x: np.ndarray, dtype: str) -> np.ndarray:
    x = np.ascontiguousarray(x)
    y = np.empty(x.shape, dtype=np.float32)
    lib().orc_to_f32_array(_p(x), DTYPE_CODE[dtype], _p(y), x.size)
    return y


def loss_scale_trajectory(found_infs, init_scale=2.0 ** 16, growth=2.0, backoff=0.5, interval=2000):
    """Scale after each step of a GradScaler-style dynamic loss scale."""
    sc, good = ctypes.c_float(init_scale), ctypes.c_int32(0)
    out = []
    for f in found_infs:
        lib().orc_loss_scale_update(ctypes.byref(sc), ctypes.byref(good), int(bool(f)), growth, backoff, interval)
        out.append(sc.value)
    return out


# ---------------------------------------------------------------- one step
@dataclass
class StepState:
    """The rank's optimizer state: fp32 master, exp_avg, exp_avg_sq, the low-precision copy, step t."""
    p: np.ndarray
    m: np.ndarray
    v: np.ndarray
    lowp: np.ndarray
    t: int = 0


def new_state(master: np.ndarray) -> StepState:
    master = np.ascontiguousarray(master, dtype=np.float32).copy()
    return StepState(p=master, m=np.zeros_like(master), v=np.zeros_like(master),
                     lowp=np.zeros(master.shape, dtype=np.uint16), t=0)


def step_reference(state: StepState, grad: np.ndarray, *, lr: float, betas, eps: float, wd: float,
                   max_norm: float, extra_sqnorm: float = 0.0, norm_grad: Optional[np.ndarray] = None,
                   lowp_dtype: str = "bf16") -> ClipResult:
    """clip_grad_norm_ then AdamW over the shard, as the pages' loops order them.

    ``grad`` is the rank's flat fp32 grad shard (already flattened/accumulated).
    ``norm_grad`` is the buffer the norm is taken over (default: ``grad``;
    ZeRO-1 takes it over the whole averaged flat grad).  A non-finite norm
    skips the step and leaves the state and the step counter untouched.
    """
    sq = sqnorm(norm_grad if norm_grad is not None else grad)
    cr = clip(sq, extra_sqnorm, max_norm)
    if not cr.finite:
        return cr
    state.t += 1
    sc = adamw_scalars(lr, betas[0], betas[1], eps, wd, state.t)
    adamw(state.p, state.m, state.v, grad, sc, cr.coef, state.lowp, lowp_dtype)
    return cr
