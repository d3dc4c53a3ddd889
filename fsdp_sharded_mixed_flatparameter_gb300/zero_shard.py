"""ctypes binding of libzeroshard with the C ABI's names.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  Tensors are PyTorch tensors (device memory and streams come from
PyTorch); they are checked to be contiguous CUDA tensors of the right dtype
before their addresses are handed to the library, so that a host pointer can
never reach a kernel.  There is no CPU fallback: without the built library
every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import List, NamedTuple, Optional, Sequence, Tuple

import numpy as np
import torch

from . import build as _build

ZERO_OK, ZERO_EINVAL, ZERO_ECUDA = 0, 1, 2
ZERO_F32, ZERO_BF16, ZERO_F16 = 0, 1, 2

_DT = {torch.float32: ZERO_F32, torch.bfloat16: ZERO_BF16, torch.float16: ZERO_F16}


class ZeroError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{msg} (status {status})")
        self.status = status


class zero_tensor(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("numel", ctypes.c_int64), ("flat_offset", ctypes.c_int64)]


class zero_norm_result(ctypes.Structure):
    _fields_ = [("sqnorm", ctypes.c_double), ("norm", ctypes.c_double), ("clip_coef", ctypes.c_float),
                ("finite", ctypes.c_int32)]


class zero_adamw_hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double)]


class zero_loss_scale_state(ctypes.Structure):
    _fields_ = [("scale", ctypes.c_float), ("growth_tracker", ctypes.c_int32), ("unscale", ctypes.c_float),
                ("found_inf", ctypes.c_int32)]


class zero_adamw_device_state(ctypes.Structure):
    _fields_ = [("step", ctypes.c_int64), ("apply", ctypes.c_int32), ("status", ctypes.c_int32),
                ("scalars", ctypes.c_float * 8)]


NORM_RESULT_BYTES = ctypes.sizeof(zero_norm_result)
HPARAMS_BYTES = ctypes.sizeof(zero_adamw_hparams)
DEVICE_STATE_BYTES = ctypes.sizeof(zero_adamw_device_state)
TENSOR_ENTRY_BYTES = ctypes.sizeof(zero_tensor)
LOSS_SCALE_STATE_BYTES = ctypes.sizeof(zero_loss_scale_state)

_lib = None


def debug_build_selected() -> bool:
    """ZERO_SHARD_DEBUG=1 selects the self-checking debug library (built with -DZERO_DEBUG)."""
    return os.environ.get("ZERO_SHARD_DEBUG", "") == "1"


def library_path() -> str:
    return _build.DEBUG_LIB if debug_build_selected() else _build.LIB


def lib() -> ctypes.CDLL:
    """Load the in-tree libzeroshard.so (built by __graft_entry__.build())."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libzeroshard is not built ({path} missing): run __graft_entry__.build()")
    L = ctypes.CDLL(path)
    i32, i64, f32, f64, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_double, ctypes.c_void_p
    L.zero_shard_range.argtypes = [i64, i32, i32, ctypes.POINTER(i64), ctypes.POINTER(i64)]
    L.zero_tensor_table.argtypes = [vp, vp, i32, vp, ctypes.POINTER(i64)]
    sz = ctypes.c_size_t
    L.zero_flatten_cast.argtypes = [vp, i32, i64, ctypes.c_int, i64, i64, f32, vp, i32, vp, vp, vp, sz, vp]
    L.zero_accum.argtypes = [vp, vp, ctypes.c_int, i64, f32, vp, i32, vp, vp, sz, vp]
    L.zero_reduce_chunks.argtypes = [vp, vp, ctypes.c_int, i32, i64, i64, f32, vp, i32, vp, vp, sz, vp]
    L.zero_grad_sqnorm_finalize.argtypes = [vp, i64, f64, f64, vp, vp]
    L.zero_grad_sqnorm_combine.argtypes = [vp, i32, f64, vp, vp]
    L.zero_grad_sqnorm_workspace_bytes.argtypes = [i64]
    L.zero_grad_sqnorm_workspace_bytes.restype = ctypes.c_size_t
    L.zero_grad_sqnorm.argtypes = [vp, i64, f64, f64, vp, ctypes.c_size_t, vp, vp]
    L.zero_grad_sqnorm_noalloc.argtypes = [vp, i64, f64, f64, vp, vp]
    L.zero_adamw_step.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, i64, ctypes.POINTER(zero_adamw_hparams), i64,
                                  vp, vp]
    L.zero_adamw_step_tensors.argtypes = [vp, vp, vp, vp, i32, i64, ctypes.c_int, i64, f32, vp, vp, vp,
                                          ctypes.c_int, i64, ctypes.POINTER(zero_adamw_hparams), i64, vp, vp]
    L.zero_loss_scale_update.argtypes = [ctypes.POINTER(f32), ctypes.POINTER(i32), i32, f64, f64, i32]
    L.zero_loss_scale_update_device.argtypes = [vp, i32, f64, f64, i32, vp, vp]
    L.zero_adamw_scalars.argtypes = [ctypes.POINTER(zero_adamw_hparams), i64, vp]
    L.zero_debug_errors.argtypes = [vp, i32]
    L.zero_debug_selftest.argtypes = [i64, vp]
    L.zero_adamw_prepare_device.argtypes = [vp, vp, vp, vp]
    L.zero_adamw_step_device.argtypes = [vp, vp, vp, vp, vp, ctypes.c_int, i64, vp, vp, vp]
    L.zero_adamw_step_tensors_device.argtypes = [vp, vp, vp, vp, i32, i64, ctypes.c_int, i64, f32, vp, vp, vp,
                                                 ctypes.c_int, i64, vp, vp, vp]
    L.zero_status_string.argtypes = [ctypes.c_int]
    L.zero_status_string.restype = ctypes.c_char_p
    L.zero_last_error.argtypes = []
    L.zero_last_error.restype = ctypes.c_char_p
    for nm in ("zero_shard_range", "zero_tensor_table", "zero_flatten_cast", "zero_accum", "zero_reduce_chunks",
               "zero_grad_sqnorm",
               "zero_grad_sqnorm_finalize", "zero_grad_sqnorm_combine", "zero_grad_sqnorm_noalloc",
               "zero_adamw_step", "zero_adamw_step_tensors", "zero_loss_scale_update", "zero_loss_scale_update_device",
               "zero_adamw_scalars",
               "zero_adamw_prepare_device", "zero_adamw_step_device", "zero_adamw_step_tensors_device",
               "zero_debug_errors", "zero_debug_selftest"):
        getattr(L, nm).restype = ctypes.c_int
    _lib = L
    return L


def _check(st: int) -> None:
    if st != ZERO_OK:
        L = lib()
        raise ZeroError(st, f"{L.zero_status_string(st).decode()}: {L.zero_last_error().decode()}")


def _dev(t: Optional[torch.Tensor], name: str, dtype=None, allow_none: bool = False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _grad_ptr(t: torch.Tensor, name: str) -> int:
    """Address of a grad for the tensor table: a contiguous CUDA tensor, or a
    contiguous PINNED host tensor.  Pinned host memory is mapped into the
    device's unified address space at the same address, so the flatten
    kernel reads it directly over the host link (the host-to-device transfer
    and the flatten/cast become one pass).  Pageable host memory is refused."""
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.is_cuda:
        return t.data_ptr()
    if t.device.type == "cpu" and t.is_pinned():
        return t.data_ptr()
    raise ValueError(f"{name} must be a CUDA tensor or a pinned host tensor")


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


# ------------------------------------------------------------------ host only
def zero_shard_range(total: int, world_size: int, rank: int) -> Tuple[int, int]:
    s, e = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().zero_shard_range(total, world_size, rank, ctypes.byref(s), ctypes.byref(e)))
    return s.value, e.value


def zero_tensor_table(grads: Sequence[Optional[torch.Tensor]] = None, numels: Sequence[int] = None):
    """Host FlatParameter table for `grads` (None = no grad) or bare `numels`.

    Grads are CUDA tensors or pinned host tensors (read over the host link).
    Returns (table, total) where table is a ctypes array of zero_tensor.
    """
    if numels is None:
        numels = [0 if g is None else g.numel() for g in grads]
    n = len(numels)
    nm = np.ascontiguousarray(np.asarray(numels, dtype=np.int64))
    ptrs = None
    if grads is not None:
        ptrs = (ctypes.c_void_p * n)(*[None if g is None else _grad_ptr(g, f"grads[{i}]") for i, g in enumerate(grads)])
    table = (zero_tensor * max(n, 1))()
    total = ctypes.c_int64()
    _check(lib().zero_tensor_table(ptrs, ctypes.c_void_p(nm.ctypes.data), n, table, ctypes.byref(total)))
    return table, total.value


def device_table(table, n_tensors: int, device) -> torch.Tensor:
    """Copy a host table (from zero_tensor_table) into device memory (uint8 bytes)."""
    raw = bytes(memoryview(table))[: n_tensors * TENSOR_ENTRY_BYTES]
    host = torch.frombuffer(bytearray(raw), dtype=torch.uint8) if raw else torch.empty(0, dtype=torch.uint8)
    return host.to(device)


def zero_grad_sqnorm_workspace_bytes(n: int) -> int:
    return int(lib().zero_grad_sqnorm_workspace_bytes(n))


# --------------------------------------------------------------------- device
def _ws_bytes(ws: Optional[torch.Tensor]) -> int:
    return 0 if ws is None else ws.numel() * ws.element_size()


def _dscale(d_scale: Optional[torch.Tensor]):
    """A device float the kernels read their scale from (e.g. DeviceLossScale.unscale), or None."""
    if d_scale is None:
        return None
    if d_scale.dtype != torch.float32 or d_scale.numel() < 1:
        raise ValueError("d_scale must be a float32 device tensor")
    return _dev(d_scale, "d_scale")


# zero_flatten_cast's accumulate == 2: the norm of the accumulated sum only (nothing stored)
NORM_OF_SUM = 2


def _accum_mode(accumulate) -> int:
    if isinstance(accumulate, bool) or accumulate in (0, 1):
        return int(bool(accumulate))
    if accumulate == NORM_OF_SUM:
        return NORM_OF_SUM
    raise ValueError("accumulate must be False, True or NORM_OF_SUM")


def _check_acc(acc: Optional[torch.Tensor], n: int) -> None:
    if acc is not None and (acc.numel() != n or acc.dtype != torch.float32):
        raise ValueError("acc must be fp32 with master's size")


def zero_flatten_cast(d_table: torch.Tensor, n_tensors: int, total: int, src_dtype: torch.dtype, shard_start: int,
                      shard_end: int, scale: float, accumulate, dst: torch.Tensor,
                      found_nonfinite: Optional[torch.Tensor] = None, norm_ws: Optional[torch.Tensor] = None,
                      stream=None, d_scale: Optional[torch.Tensor] = None) -> None:
    """accumulate: False / True, or NORM_OF_SUM (2): the norm partials of dst + scale * x
    into norm_ws, dst only read."""
    if dst is not None and shard_end > shard_start and dst.numel() < shard_end - shard_start:
        raise ValueError("dst is smaller than the shard")
    tab = _dev(d_table, "d_table", torch.uint8, allow_none=n_tensors == 0)
    if n_tensors > 0 and d_table.numel() < n_tensors * TENSOR_ENTRY_BYTES:
        raise ValueError("d_table holds fewer entries than n_tensors")
    _check(lib().zero_flatten_cast(tab, n_tensors, total, _DT[src_dtype], shard_start, shard_end, scale,
                                   _dscale(d_scale), _accum_mode(accumulate),
                                   _dev(dst, "dst", torch.float32, allow_none=norm_ws is not None),
                                   _dev(found_nonfinite, "found_nonfinite", torch.int32, allow_none=True),
                                   _dev(norm_ws, "norm_ws", allow_none=True), _ws_bytes(norm_ws), _stream(stream)))


def zero_accum(acc: torch.Tensor, src: torch.Tensor, scale: float, accumulate: bool,
               found_nonfinite: Optional[torch.Tensor] = None, norm_ws: Optional[torch.Tensor] = None,
               stream=None, d_scale: Optional[torch.Tensor] = None) -> None:
    if src.numel() != acc.numel():
        raise ValueError("acc and src differ in size")
    _check(lib().zero_accum(_dev(acc, "acc", torch.float32), _dev(src, "src"), _DT[src.dtype], acc.numel(), scale,
                            _dscale(d_scale), int(bool(accumulate)),
                            _dev(found_nonfinite, "found_nonfinite", torch.int32, allow_none=True),
                            _dev(norm_ws, "norm_ws", allow_none=True), _ws_bytes(norm_ws), _stream(stream)))


def zero_reduce_chunks(acc: torch.Tensor, chunks: torch.Tensor, n: int, scale: float, accumulate: bool,
                       found_nonfinite: Optional[torch.Tensor] = None, norm_ws: Optional[torch.Tensor] = None,
                       stream=None, d_scale: Optional[torch.Tensor] = None) -> None:
    """acc[0:n] (+)= the rank-order sum of scale * chunks[r, 0:n] (chunks: a 2-D
    [n_chunks, chunk_stride] CUDA tensor of the received blocks, rank r's in row r)."""
    if chunks.dim() != 2:
        raise ValueError("chunks must be 2-D: [n_chunks, chunk_stride]")
    if chunks.dtype not in _DT:
        raise ValueError(f"chunks dtype {chunks.dtype} is not f32/bf16/f16")
    if acc.numel() < n or chunks.shape[1] < n:
        raise ValueError("acc or a chunk is shorter than n")
    _check(lib().zero_reduce_chunks(_dev(acc, "acc", torch.float32), _dev(chunks, "chunks"), _DT[chunks.dtype],
                                    chunks.shape[0], chunks.shape[1], n, scale, _dscale(d_scale),
                                    int(bool(accumulate)),
                                    _dev(found_nonfinite, "found_nonfinite", torch.int32, allow_none=True),
                                    _dev(norm_ws, "norm_ws", allow_none=True), _ws_bytes(norm_ws), _stream(stream)))


def zero_grad_sqnorm_finalize(ws: Optional[torch.Tensor], n: int, extra_sqnorm: float, max_norm: float,
                              out: torch.Tensor, stream=None) -> None:
    """Norm result from the partials a fused flatten/accumulate pass wrote for an n-element grad."""
    if out.numel() * out.element_size() < NORM_RESULT_BYTES:
        raise ValueError("out is smaller than zero_norm_result")
    if n > 0 and _ws_bytes(ws) < zero_grad_sqnorm_workspace_bytes(n):
        raise ValueError("ws is smaller than the partials of n elements")
    _check(lib().zero_grad_sqnorm_finalize(_dev(ws, "ws", allow_none=True), n, extra_sqnorm, max_norm,
                                           _dev(out, "out"), _stream(stream)))


def zero_grad_sqnorm(grad: torch.Tensor, extra_sqnorm: float, max_norm: float, ws: torch.Tensor,
                     out: torch.Tensor, stream=None) -> None:
    if out.numel() * out.element_size() < NORM_RESULT_BYTES:
        raise ValueError("out is smaller than zero_norm_result")
    _check(lib().zero_grad_sqnorm(_dev(grad, "grad", torch.float32), grad.numel(), extra_sqnorm, max_norm,
                                  _dev(ws, "ws", allow_none=True), 0 if ws is None else ws.numel() * ws.element_size(),
                                  _dev(out, "out"), _stream(stream)))


def zero_grad_sqnorm_noalloc(grad: torch.Tensor, extra_sqnorm: float, max_norm: float, out: torch.Tensor,
                             stream=None) -> None:
    """zero_grad_sqnorm for callers that cannot allocate a workspace (library-owned scratch)."""
    if out.numel() * out.element_size() < NORM_RESULT_BYTES:
        raise ValueError("out is smaller than zero_norm_result")
    _check(lib().zero_grad_sqnorm_noalloc(_dev(grad, "grad", torch.float32), grad.numel(), extra_sqnorm, max_norm,
                                          _dev(out, "out"), _stream(stream)))


def zero_grad_sqnorm_combine(sqnorms: torch.Tensor, max_norm: float, out: torch.Tensor, stream=None) -> None:
    """Global norm result from the ranks' local sums of squares (float64 CUDA vector, rank order)."""
    if out.numel() * out.element_size() < NORM_RESULT_BYTES:
        raise ValueError("out is smaller than zero_norm_result")
    _check(lib().zero_grad_sqnorm_combine(_dev(sqnorms, "sqnorms", torch.float64), sqnorms.numel(), max_norm,
                                          _dev(out, "out"), _stream(stream)))


def sqnorm_view(result: torch.Tensor) -> torch.Tensor:
    """The `sqnorm` field of a device zero_norm_result buffer as a 1-element float64 tensor view."""
    return result[:8].view(torch.float64)


def zero_adamw_step(master: torch.Tensor, exp_avg: torch.Tensor, exp_avg_sq: torch.Tensor, grad: torch.Tensor,
                    param_lowp: Optional[torch.Tensor], lr: float, beta1: float, beta2: float, eps: float,
                    weight_decay: float, step: int, clip: Optional[torch.Tensor] = None, stream=None) -> None:
    n = master.numel()
    for t, nm in ((exp_avg, "exp_avg"), (exp_avg_sq, "exp_avg_sq"), (grad, "grad")):
        if t.numel() != n:
            raise ValueError(f"{nm} differs in size from master")
    lowp_dt = ZERO_BF16
    if param_lowp is not None:
        if param_lowp.numel() != n:
            raise ValueError("param_lowp differs in size from master")
        if param_lowp.dtype not in (torch.bfloat16, torch.float16):
            raise ValueError("param_lowp must be bf16 or f16")
        lowp_dt = _DT[param_lowp.dtype]
    if clip is not None and clip.numel() * clip.element_size() < NORM_RESULT_BYTES:
        raise ValueError("clip is smaller than zero_norm_result")
    hp = zero_adamw_hparams(lr, beta1, beta2, eps, weight_decay)
    _check(lib().zero_adamw_step(_dev(master, "master", torch.float32), _dev(exp_avg, "exp_avg", torch.float32),
                                 _dev(exp_avg_sq, "exp_avg_sq", torch.float32), _dev(grad, "grad", torch.float32),
                                 _dev(param_lowp, "param_lowp", allow_none=True), lowp_dt, n, ctypes.byref(hp), step,
                                 _dev(clip, "clip", allow_none=True), _stream(stream)))


def zero_adamw_step_tensors(master: torch.Tensor, exp_avg: torch.Tensor, exp_avg_sq: torch.Tensor,
                            d_table: torch.Tensor, n_tensors: int, total: int, grad_dtype: torch.dtype,
                            shard_start: int, grad_scale: float, param_lowp: Optional[torch.Tensor], lr: float,
                            beta1: float, beta2: float, eps: float, weight_decay: float, step: int,
                            clip: Optional[torch.Tensor] = None, stream=None, acc: Optional[torch.Tensor] = None,
                            d_scale: Optional[torch.Tensor] = None) -> None:
    """AdamW over [shard_start, shard_start + n) with the grads read through the tensor table;
    acc: the earlier micro-batches' fp32 sum over the same n elements, added first (or None);
    d_scale: a device float used in place of grad_scale (or None)."""
    n = master.numel()
    for t, nm in ((exp_avg, "exp_avg"), (exp_avg_sq, "exp_avg_sq")):
        if t.numel() != n:
            raise ValueError(f"{nm} differs in size from master")
    _check_acc(acc, n)
    if n_tensors > 0 and d_table.numel() < n_tensors * TENSOR_ENTRY_BYTES:
        raise ValueError("d_table holds fewer entries than n_tensors")
    lowp_dt = ZERO_BF16
    if param_lowp is not None:
        if param_lowp.numel() != n or param_lowp.dtype not in (torch.bfloat16, torch.float16):
            raise ValueError("param_lowp must be bf16/f16 with master's size")
        lowp_dt = _DT[param_lowp.dtype]
    if clip is not None and clip.numel() * clip.element_size() < NORM_RESULT_BYTES:
        raise ValueError("clip is smaller than zero_norm_result")
    hp = zero_adamw_hparams(lr, beta1, beta2, eps, weight_decay)
    _check(lib().zero_adamw_step_tensors(_dev(master, "master", torch.float32), _dev(exp_avg, "exp_avg", torch.float32),
                                         _dev(exp_avg_sq, "exp_avg_sq", torch.float32),
                                         _dev(d_table, "d_table", torch.uint8, allow_none=n_tensors == 0), n_tensors,
                                         total, _DT[grad_dtype], shard_start, grad_scale, _dscale(d_scale),
                                         _dev(acc, "acc", torch.float32, allow_none=True),
                                         _dev(param_lowp, "param_lowp", allow_none=True), lowp_dt, n, ctypes.byref(hp),
                                         step, _dev(clip, "clip", allow_none=True), _stream(stream)))


# ------------------------------------------------- graph-capturable steps
def zero_adamw_scalars(lr: float, beta1: float, beta2: float, eps: float, weight_decay: float, step: int) -> np.ndarray:
    """The 8 binary32 scalars of step `step` (host): step_size, sqrt(1-beta2^t), 1-lr*wd,
    beta1, 1-beta1, beta2, 1-beta2, eps."""
    out = np.zeros(8, dtype=np.float32)
    hp = zero_adamw_hparams(lr, beta1, beta2, eps, weight_decay)
    _check(lib().zero_adamw_scalars(ctypes.byref(hp), step, ctypes.c_void_p(out.ctypes.data)))
    return out


def device_hparams(lr: float, beta1: float, beta2: float, eps: float, weight_decay: float, device,
                   out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """A zero_adamw_hparams in device memory (uint8 bytes); rewrites `out` in place when given."""
    hp = zero_adamw_hparams(lr, beta1, beta2, eps, weight_decay)
    host = torch.frombuffer(bytearray(bytes(memoryview(hp))), dtype=torch.uint8)
    if out is None:
        return host.to(device)
    out.copy_(host)
    return out


def new_adamw_device_state(device, step: int = 0) -> torch.Tensor:
    """Device buffer for one zero_adamw_device_state with the step count set (0: fresh)."""
    st = zero_adamw_device_state(step, 0, 0)
    return torch.frombuffer(bytearray(bytes(memoryview(st))), dtype=torch.uint8).to(device)


class AdamwDeviceState(NamedTuple):
    step: int
    apply: bool
    status: int
    scalars: np.ndarray


def decode_adamw_device_state(buf: torch.Tensor) -> AdamwDeviceState:
    raw = bytes(buf.detach().cpu().numpy().tobytes()[:DEVICE_STATE_BYTES])
    r = zero_adamw_device_state.from_buffer_copy(raw)
    return AdamwDeviceState(r.step, bool(r.apply), r.status, np.array(list(r.scalars), dtype=np.float32))


def _state_arg(state: torch.Tensor):
    if state.numel() * state.element_size() < DEVICE_STATE_BYTES:
        raise ValueError("state is smaller than zero_adamw_device_state")
    return _dev(state, "state")


def zero_adamw_prepare_device(d_hp: torch.Tensor, clip: Optional[torch.Tensor], state: torch.Tensor,
                              stream=None) -> None:
    """Advance the device step state for the next step (skipped on a non-finite norm)."""
    if d_hp.numel() * d_hp.element_size() < HPARAMS_BYTES:
        raise ValueError("d_hp is smaller than zero_adamw_hparams")
    if clip is not None and clip.numel() * clip.element_size() < NORM_RESULT_BYTES:
        raise ValueError("clip is smaller than zero_norm_result")
    _check(lib().zero_adamw_prepare_device(_dev(d_hp, "d_hp"), _dev(clip, "clip", allow_none=True),
                                           _state_arg(state), _stream(stream)))


def _lowp_arg(param_lowp: Optional[torch.Tensor], n: int):
    if param_lowp is None:
        return None, ZERO_BF16
    if param_lowp.numel() != n or param_lowp.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("param_lowp must be bf16/f16 with master's size")
    return _dev(param_lowp, "param_lowp"), _DT[param_lowp.dtype]


def zero_adamw_step_device(master: torch.Tensor, exp_avg: torch.Tensor, exp_avg_sq: torch.Tensor,
                           grad: torch.Tensor, param_lowp: Optional[torch.Tensor], state: torch.Tensor,
                           clip: Optional[torch.Tensor] = None, stream=None) -> None:
    """zero_adamw_step with the scalars and skip decision of the device step state."""
    n = master.numel()
    for t, nm in ((exp_avg, "exp_avg"), (exp_avg_sq, "exp_avg_sq"), (grad, "grad")):
        if t.numel() != n:
            raise ValueError(f"{nm} differs in size from master")
    if clip is not None and clip.numel() * clip.element_size() < NORM_RESULT_BYTES:
        raise ValueError("clip is smaller than zero_norm_result")
    lp, lowp_dt = _lowp_arg(param_lowp, n)
    _check(lib().zero_adamw_step_device(_dev(master, "master", torch.float32), _dev(exp_avg, "exp_avg", torch.float32),
                                        _dev(exp_avg_sq, "exp_avg_sq", torch.float32),
                                        _dev(grad, "grad", torch.float32), lp, lowp_dt, n, _state_arg(state),
                                        _dev(clip, "clip", allow_none=True), _stream(stream)))


def zero_adamw_step_tensors_device(master: torch.Tensor, exp_avg: torch.Tensor, exp_avg_sq: torch.Tensor,
                                   d_table: torch.Tensor, n_tensors: int, total: int, grad_dtype: torch.dtype,
                                   shard_start: int, grad_scale: float, param_lowp: Optional[torch.Tensor],
                                   state: torch.Tensor, clip: Optional[torch.Tensor] = None, stream=None,
                                   acc: Optional[torch.Tensor] = None, d_scale: Optional[torch.Tensor] = None) -> None:
    """zero_adamw_step_tensors with the scalars and skip decision of the device step state."""
    n = master.numel()
    for t, nm in ((exp_avg, "exp_avg"), (exp_avg_sq, "exp_avg_sq")):
        if t.numel() != n:
            raise ValueError(f"{nm} differs in size from master")
    _check_acc(acc, n)
    if n_tensors > 0 and d_table.numel() < n_tensors * TENSOR_ENTRY_BYTES:
        raise ValueError("d_table holds fewer entries than n_tensors")
    if clip is not None and clip.numel() * clip.element_size() < NORM_RESULT_BYTES:
        raise ValueError("clip is smaller than zero_norm_result")
    lp, lowp_dt = _lowp_arg(param_lowp, n)
    _check(lib().zero_adamw_step_tensors_device(
        _dev(master, "master", torch.float32), _dev(exp_avg, "exp_avg", torch.float32),
        _dev(exp_avg_sq, "exp_avg_sq", torch.float32), _dev(d_table, "d_table", torch.uint8, allow_none=n_tensors == 0),
        n_tensors, total, _DT[grad_dtype], shard_start, grad_scale, _dscale(d_scale),
        _dev(acc, "acc", torch.float32, allow_none=True), lp, lowp_dt, n, _state_arg(state),
        _dev(clip, "clip", allow_none=True), _stream(stream)))


# ------------------------------------------------------------ debug builds
class DebugRecord(NamedTuple):
    count: int
    site: int
    index: int
    block: int


def zero_debug_errors(reset: bool = False) -> DebugRecord:
    """Access-check violations the debug library recorded (ZeroError on a release library)."""
    out = np.zeros(4, dtype=np.uint64)
    _check(lib().zero_debug_errors(ctypes.c_void_p(out.ctypes.data), int(bool(reset))))
    return DebugRecord(*(int(x) for x in out))


def zero_debug_selftest(index: int, stream=None) -> None:
    _check(lib().zero_debug_selftest(index, _stream(stream)))


# ------------------------------------------------------------ norm result I/O
class NormResult(NamedTuple):
    sqnorm: float
    norm: float
    clip_coef: float
    finite: bool


def new_norm_result(device) -> torch.Tensor:
    """Device buffer for one zero_norm_result (8-byte aligned by the allocator)."""
    return torch.zeros(NORM_RESULT_BYTES, dtype=torch.uint8, device=device)


def decode_norm_result(buf: torch.Tensor) -> NormResult:
    """Read a zero_norm_result (device or host bytes) into Python values."""
    raw = bytes(buf.detach().cpu().numpy().tobytes()[:NORM_RESULT_BYTES])
    r = zero_norm_result.from_buffer_copy(raw)
    return NormResult(r.sqnorm, r.norm, r.clip_coef, bool(r.finite))


# ------------------------------------------------------------ loss scaling
class DynamicLossScale:
    """GradScaler-style dynamic loss scale (host policy: zero_loss_scale_update).

    Multiply the loss by ``scale`` before backward; pass ``unscale_factor(accum_steps)``
    as the flatten / accumulate ``scale`` (the unscale and the 1/accum_steps
    averaging in one exact multiply for power-of-two values); after the step call
    ``update(found_inf)`` with the kernels' non-finite flag.
    """

    def __init__(self, init_scale: float = 2.0 ** 16, growth_factor: float = 2.0, backoff_factor: float = 0.5,
                 growth_interval: int = 2000):
        self._scale = ctypes.c_float(init_scale)
        self._good = ctypes.c_int32(0)
        self.growth_factor, self.backoff_factor, self.growth_interval = growth_factor, backoff_factor, growth_interval

    @property
    def scale(self) -> float:
        return self._scale.value

    @property
    def growth_tracker(self) -> int:
        return self._good.value

    def unscale_factor(self, accum_steps: int = 1) -> float:
        return 1.0 / (float(self._scale.value) * accum_steps)

    def update(self, found_inf: bool) -> None:
        _check(lib().zero_loss_scale_update(ctypes.byref(self._scale), ctypes.byref(self._good), int(bool(found_inf)),
                                            self.growth_factor, self.backoff_factor, self.growth_interval))


def zero_loss_scale_update_device(state: torch.Tensor, accum_steps: int, growth_factor: float,
                                  backoff_factor: float, growth_interval: int,
                                  norm_result: Optional[torch.Tensor] = None, stream=None) -> None:
    """The loss-scale update on a zero_loss_scale_state in device memory (one thread)."""
    if state.numel() * state.element_size() < LOSS_SCALE_STATE_BYTES:
        raise ValueError("state is smaller than zero_loss_scale_state")
    if norm_result is not None and norm_result.numel() * norm_result.element_size() < NORM_RESULT_BYTES:
        raise ValueError("norm_result is smaller than zero_norm_result")
    _check(lib().zero_loss_scale_update_device(_dev(state, "state"), accum_steps, growth_factor, backoff_factor,
                                               growth_interval, _dev(norm_result, "norm_result", allow_none=True),
                                               _stream(stream)))


class DeviceLossScale:
    """The GradScaler-style dynamic loss scale kept in device memory (a
    zero_loss_scale_state), for mixed-precision steps captured in a CUDA graph.

    The grad passes read ``unscale`` (= 1/(scale * accum_steps)) from device
    memory when they run (``d_scale``) and raise ``found_inf``
    (``found_nonfinite``); ``launch_update()`` (one thread, capturable) backs
    the scale off or grows it on the device, recomputes ``unscale`` and clears
    the flag.  The same rule and roundings as DynamicLossScale.update, so both
    follow the same scale bit for bit.  ``scale``, ``growth_tracker`` and
    ``read()`` copy the state to the host (a synchronisation)."""

    def __init__(self, device, init_scale: float = 2.0 ** 16, growth_factor: float = 2.0,
                 backoff_factor: float = 0.5, growth_interval: int = 2000, accum_steps: int = 1):
        if accum_steps < 1:
            raise ValueError("accum_steps must be >= 1")
        self.growth_factor, self.backoff_factor, self.growth_interval = growth_factor, backoff_factor, growth_interval
        self.accum_steps = int(accum_steps)
        sc = ctypes.c_float(init_scale).value
        st = zero_loss_scale_state(sc, 0, ctypes.c_float(1.0 / (float(sc) * self.accum_steps)).value, 0)
        self.state = torch.frombuffer(bytearray(bytes(memoryview(st))), dtype=torch.uint8).to(device)
        self.unscale = self.state[8:12].view(torch.float32)     # the grad passes' d_scale
        self.found_inf = self.state[12:16].view(torch.int32)    # the grad passes' found_nonfinite

    def launch_update(self, norm_result: Optional[torch.Tensor] = None, stream=None) -> None:
        """Enqueue the update after a step (norm_result: the step's zero_norm_result, whose
        non-finite norm also counts as an overflow)."""
        zero_loss_scale_update_device(self.state, self.accum_steps, self.growth_factor, self.backoff_factor,
                                      self.growth_interval, norm_result, stream)

    def read(self) -> zero_loss_scale_state:
        raw = bytes(self.state.detach().cpu().numpy().tobytes()[:LOSS_SCALE_STATE_BYTES])
        return zero_loss_scale_state.from_buffer_copy(raw)

    @property
    def scale(self) -> float:
        return self.read().scale

    @property
    def growth_tracker(self) -> int:
        return self.read().growth_tracker
