"""FlatShardAdamW: one data-parallel rank's optimizer step over its flat shard.

Holds the rank's buffers (fp32 flat grad, fp32 master / exp_avg /
exp_avg_sq, the low-precision parameter copy, the grad-norm workspace and
result) and sequences the library calls of one training step the way the
pages' loops do: per micro-batch flatten/accumulate (loss / accum_steps),
then clip_grad_norm_, then the AdamW step with the step counter t
incremented before use, skipping the step when the grad norm is not finite
(the ZeRO page, section "组合策略": "if not isfinite(grad_norm): skip").

All arithmetic runs in libzeroshard's kernels; this class only allocates
buffers with PyTorch and keeps the host-side step counter.

Graph capture (``capturable=True``): the step counter and the skip decision
live on the device (zero_adamw_prepare_device), so flatten/accumulate plus
``launch_step()`` (or ``launch_step_tensors()``) make no host synchronisation
and can be captured once in a ``torch.cuda.CUDAGraph`` and replayed as whole
steps; the results are bit-identical to the host-counter steps.

Grad range: for ZeRO-2/3 and FSDP the rank holds grads of its own shard
only (``grad_range="shard"``, norm over the shard plus ``extra_sqnorm`` from
the other ranks).  For ZeRO-1 every rank holds the whole averaged flat grad
(the ZeRO page's ZeRO1Optimizer.step all-reduces it), so the grad buffer
covers the whole flat parameter (``grad_range="full"``), the norm is global,
and the update uses the rank's slice.
"""
from __future__ import annotations

import math
from typing import Dict, Optional, Sequence, Tuple

import torch

from . import zero_shard as zs


class FlatShardAdamW:
    def __init__(self, numels: Sequence[int], *, world_size: int = 1, rank: int = 0, lr: float = 1e-4,
                 betas: Tuple[float, float] = (0.9, 0.999), eps: float = 1e-8, weight_decay: float = 0.0,
                 max_norm: float = math.inf, lowp_dtype: Optional[torch.dtype] = torch.bfloat16,
                 grad_range: str = "shard", device="cuda", master: Optional[torch.Tensor] = None,
                 lowp_out: Optional[torch.Tensor] = None, grad_buffer: bool = True, capturable: bool = False,
                 workspace: Optional[torch.Tensor] = None):
        if grad_range not in ("shard", "full"):
            raise ValueError("grad_range must be 'shard' or 'full'")
        self.device = torch.device(device)
        self.numels = [int(n) for n in numels]
        self.total = int(sum(self.numels))
        self.world_size, self.rank = world_size, rank
        self.start, self.end = zs.zero_shard_range(self.total, world_size, rank)
        self.n = self.end - self.start
        self.glo, self.ghi = (0, self.total) if grad_range == "full" else (self.start, self.end)
        self.capturable = capturable
        self._hp = [float(lr), float(betas[0]), float(betas[1]), float(eps), float(weight_decay)]
        self.max_norm = max_norm
        dev = self.device
        # the fp32 flat grad; not needed when every step goes through step_tensors()
        self.grad = torch.empty(self.ghi - self.glo if grad_buffer else 0, dtype=torch.float32, device=dev)
        if master is None:
            master = torch.zeros(self.n, dtype=torch.float32, device=dev)
        if master.numel() != self.n or master.dtype != torch.float32:
            raise ValueError("master must be fp32 with the shard's size")
        self.master = master.to(dev).contiguous()
        self.exp_avg = torch.zeros(self.n, dtype=torch.float32, device=dev)
        self.exp_avg_sq = torch.zeros(self.n, dtype=torch.float32, device=dev)
        if lowp_out is not None:
            self.lowp = lowp_out  # e.g. the rank's slice of the full low-precision FlatParameter
        elif lowp_dtype is not None:
            self.lowp = torch.empty(self.n, dtype=lowp_dtype, device=dev)
        else:
            self.lowp = None
        need = zs.zero_grad_sqnorm_workspace_bytes(self.ghi - self.glo)
        if workspace is not None:  # e.g. this optimizer's slice of a workspace shared by several FSDP units
            if workspace.dtype != torch.uint8 or workspace.numel() < need or workspace.device != dev:
                raise ValueError(f"workspace must be >= {need} uint8 bytes on {dev}")
            self.ws = workspace
        else:
            self.ws = torch.empty(max(need, 8), dtype=torch.uint8, device=dev)
        self.norm_buf = zs.new_norm_result(dev)
        self.found_nonfinite = torch.zeros(1, dtype=torch.int32, device=dev)
        self._t = 0
        if capturable:
            self._dev_hp = zs.device_hparams(*self._hp, dev)
            self._dev_state = zs.new_adamw_device_state(dev)
        self._norm_ready = False  # the grad norm's tile partials are up to date in self.ws
        self._local_buf: Optional[torch.Tensor] = None
        self._registered = None
        self._tables: Dict[tuple, Tuple[torch.Tensor, int]] = {}
        self._flat_tables: Dict[tuple, torch.Tensor] = {}

    # ------------------------------------------------------- step counter
    @property
    def t(self) -> int:
        """Steps applied so far (with capturable=True read from the device: a sync)."""
        if self.capturable:
            return zs.decode_adamw_device_state(self._dev_state).step
        return self._t

    @t.setter
    def t(self, value: int) -> None:
        if self.capturable:
            self._dev_state.copy_(zs.new_adamw_device_state(self.device, int(value)))
        else:
            self._t = int(value)

    # -------------------------------------------------- hyper-parameters
    # Assigning lr / betas / eps / weight_decay (e.g. from a schedule) also rewrites the
    # device copy in place when capturable=True, so a captured graph reads the new values
    # at its next replay.
    def _set_hp(self, i: int, value: float) -> None:
        self._hp[i] = float(value)
        if self.capturable:
            zs.device_hparams(*self._hp, self.device, out=self._dev_hp)

    @property
    def lr(self) -> float:
        return self._hp[0]

    @lr.setter
    def lr(self, value: float) -> None:
        self._set_hp(0, value)

    @property
    def betas(self) -> Tuple[float, float]:
        return (self._hp[1], self._hp[2])

    @betas.setter
    def betas(self, value: Tuple[float, float]) -> None:
        self._hp[1] = float(value[0])
        self._set_hp(2, value[1])

    @property
    def eps(self) -> float:
        return self._hp[3]

    @eps.setter
    def eps(self, value: float) -> None:
        self._set_hp(3, value)

    @property
    def weight_decay(self) -> float:
        return self._hp[4]

    @weight_decay.setter
    def weight_decay(self, value: float) -> None:
        self._set_hp(4, value)

    def set_hparams(self, lr: Optional[float] = None, weight_decay: Optional[float] = None) -> None:
        """Change lr and/or weight decay (same as assigning the attributes)."""
        if lr is not None:
            self.lr = lr
        if weight_decay is not None:
            self.weight_decay = weight_decay

    # ---------------------------------------------------------------- grads
    def _table(self, grads: Sequence[Optional[torch.Tensor]]) -> torch.Tensor:
        # keyed by address, size and contiguity, so a cached table is only reused for
        # grads that passed the checks below when it was built
        key = tuple(None if g is None else (g.data_ptr(), g.numel(), g.is_contiguous()) for g in grads)
        hit = self._tables.get(key)
        if hit is None:
            if len(grads) != len(self.numels):
                raise ValueError("one grad (or None) per parameter tensor is required")
            for i, (g, n) in enumerate(zip(grads, self.numels)):
                if g is not None and g.numel() != n:
                    raise ValueError(f"grad {i} has {g.numel()} elements, expected {n}")
            table, total = zs.zero_tensor_table(grads, self.numels)
            assert total == self.total
            hit = (zs.device_table(table, len(grads), self.device), total)
            if len(self._tables) > 64:
                self._tables.clear()
            self._tables[key] = hit
        return hit[0]

    def device_table(self, grads: Sequence[Optional[torch.Tensor]]) -> Tuple[torch.Tensor, int, torch.dtype]:
        """The FlatParameter table of a grads list in device memory (built once per list of
        grad addresses and cached), with its tensor count and grad dtype.  Calling it before
        a CUDA graph capture keeps the table's host-to-device copy out of the graph."""
        return self._resolve(grads)

    def register_grads(self, grads: Sequence[Optional[torch.Tensor]]) -> None:
        """Fix the per-tensor grads once (e.g. views into one flat grad storage, as
        FSDP's FlatParameter keeps them).  flatten() / step_tensors() called without
        grads then reuse the device table and do no per-tensor host work, which
        matters for lists of thousands of tensors."""
        self._registered = (self._table(grads), len(grads), self._grad_dtype(grads))

    @staticmethod
    def _grad_dtype(grads) -> torch.dtype:
        dts = {g.dtype for g in grads if g is not None}
        if len(dts) > 1:
            raise ValueError("all grads must share one dtype")
        return dts.pop() if dts else torch.float32

    def _resolve(self, grads):
        if grads is None:
            if self._registered is None:
                raise ValueError("no grads given and none registered")
            return self._registered
        return self._table(grads), len(grads), self._grad_dtype(grads)

    def _scale_args(self, scale, loss_scale):
        """(host scale, device scale or None, non-finite flag) of a grad pass: with a
        DeviceLossScale the kernels read its unscale factor and raise its flag."""
        if loss_scale is None:
            return float(scale), None, self.found_nonfinite
        return 1.0, loss_scale.unscale, loss_scale.found_inf

    def flatten(self, grads: Optional[Sequence[Optional[torch.Tensor]]] = None, *, accumulate: bool,
                scale: float = 1.0, fuse_norm: bool = False, stream=None, loss_scale=None) -> None:
        """Flatten/cast per-tensor grads (or the registered ones) into the rank's flat
        fp32 grad (K1).

        fuse_norm: this is the last micro-batch; the same pass also computes the
        grad norm's tile partials, so step() only has to finalize them.
        loss_scale: a DeviceLossScale; the pass then multiplies by its unscale
        factor, read on the device when the kernel runs (so a captured graph
        follows the scale), and raises its overflow flag; `scale` is ignored.
        """
        table, count, dt = self._resolve(grads)
        sc, dsc, flag = self._scale_args(scale, loss_scale)
        zs.zero_flatten_cast(table, count, self.total, dt, self.glo, self.ghi, sc, accumulate,
                             self.grad, flag, self.ws if fuse_norm else None, stream, d_scale=dsc)
        self._norm_ready = fuse_norm

    def accum(self, flat_src: torch.Tensor, *, accumulate: bool, scale: float = 1.0, fuse_norm: bool = False,
              stream=None, loss_scale=None) -> None:
        """Accumulate a flat low-precision grad covering the grad range (K2); fuse_norm and
        loss_scale as for flatten()."""
        sc, dsc, flag = self._scale_args(scale, loss_scale)
        zs.zero_accum(self.grad, flat_src, sc, accumulate, flag, self.ws if fuse_norm else None, stream, d_scale=dsc)
        self._norm_ready = fuse_norm

    def reduce(self, chunks: torch.Tensor, *, accumulate: bool, scale: float, fuse_norm: bool = False,
               stream=None, loss_scale=None) -> None:
        """Reduce the ranks' received chunks of this shard into the fp32 shard grad (ZeRO-2/3,
        zero_reduce_chunks): chunks is [world_size, chunk] in rank order, the first n of each
        row are this shard's values; fuse_norm and loss_scale as for flatten()."""
        if self.glo != self.start:
            raise ValueError("reduce() needs a shard-only grad buffer (grad_range='shard')")
        sc, dsc, flag = self._scale_args(scale, loss_scale)
        zs.zero_reduce_chunks(self.grad, chunks, self.n, sc, accumulate, flag, self.ws if fuse_norm else None, stream,
                              d_scale=dsc)
        self._norm_ready = fuse_norm

    # ----------------------------------------------------------------- step
    def shard_grad(self) -> torch.Tensor:
        return self.grad[self.start - self.glo:self.end - self.glo]

    def _norm_into(self, out: torch.Tensor, extra_sqnorm: float, max_norm: float, stream) -> None:
        if self._norm_ready:
            zs.zero_grad_sqnorm_finalize(self.ws, self.grad.numel(), extra_sqnorm, max_norm, out, stream)
        else:
            zs.zero_grad_sqnorm(self.grad, extra_sqnorm, max_norm, self.ws, out, stream)
        self._norm_ready = False

    def local_sqnorm(self, stream=None) -> torch.Tensor:
        """Enqueue this rank's sum of squares over its grad buffer; returns it as a
        1-element float64 device tensor (the value the ranks exchange)."""
        if self._local_buf is None:
            self._local_buf = zs.new_norm_result(self.device)
        self._norm_into(self._local_buf, 0.0, math.inf, stream)
        return zs.sqnorm_view(self._local_buf)

    def launch_step(self, extra_sqnorm: float = 0.0, stream=None,
                    gathered_sqnorms: Optional[torch.Tensor] = None,
                    norm_result: Optional[torch.Tensor] = None) -> None:
        """Enqueue the grad norm and the AdamW step (K4) for t+1 without waiting.

        gathered_sqnorms: the ranks' local sums of squares in rank order (float64,
        on this device) for a global norm across ranks; otherwise the norm covers
        this rank's grad buffer plus `extra_sqnorm`.  norm_result: a zero_norm_result
        another optimizer already computed for this step (several FSDP units share
        one clip): used as is, nothing is computed.  When the norm turns out
        non-finite, K4 changes nothing on the device; finish_step() then leaves t
        unchanged.
        """
        clip = self.norm_buf if norm_result is None else norm_result
        if norm_result is not None:
            pass
        elif gathered_sqnorms is not None:
            zs.zero_grad_sqnorm_combine(gathered_sqnorms, self.max_norm, self.norm_buf, stream)
        else:
            self._norm_into(self.norm_buf, extra_sqnorm, self.max_norm, stream)
        if self.capturable:
            zs.zero_adamw_prepare_device(self._dev_hp, clip, self._dev_state, stream)
            zs.zero_adamw_step_device(self.master, self.exp_avg, self.exp_avg_sq, self.shard_grad(), self.lowp,
                                      self._dev_state, clip, stream)
        else:
            zs.zero_adamw_step(self.master, self.exp_avg, self.exp_avg_sq, self.shard_grad(), self.lowp, self.lr,
                               self.betas[0], self.betas[1], self.eps, self.weight_decay, self._t + 1,
                               clip, stream)

    def finish_step(self, stream=None, result: Optional[zs.NormResult] = None) -> zs.NormResult:
        """Read the step's grad norm (a device->host copy that waits for the step's
        work on `stream`, the stream the step was enqueued on; default: the current
        stream).  With capturable=True the device already advanced (or kept) the
        step count.  `result`: the same step's result already read from another
        optimizer that combined the same norm (several FSDP units): no second read."""
        if result is not None:
            r = result
        else:
            with torch.cuda.stream(torch_stream(stream, self.device)):
                r = zs.decode_norm_result(self.norm_buf)
        if r.finite and not self.capturable:
            self._t += 1
        return r

    def _global_norm(self, local: torch.Tensor, process_group, stream: torch.cuda.Stream) -> torch.Tensor:
        """The ranks' local sums of squares in rank order, on this device, ordered
        after `local` was written on `stream` and before later work on `stream`."""
        with torch.cuda.stream(stream):
            return gather_sqnorms(local, process_group)

    def step(self, extra_sqnorm: float = 0.0, stream=None, process_group=None) -> zs.NormResult:
        """One optimizer step.  With a torch.distributed process group of more than
        one rank and a shard-only grad buffer (ZeRO-2/3), the clip norm is global:
        the ranks exchange their 8-byte local sums of squares (all-gather, rank
        order) and every rank combines the same vector, so all ranks use the same
        coefficient and agree on skipping a non-finite step.  The exchange is
        ordered on `stream` like the kernels, whichever stream that is."""
        if process_group is not None and self.glo == self.start and _world(process_group) > 1:
            st = torch_stream(stream, self.device)
            local = self.local_sqnorm(st)
            self.launch_step(stream=st, gathered_sqnorms=self._global_norm(local, process_group, st))
        else:
            self.launch_step(extra_sqnorm, stream)
        return self.finish_step(stream)

    def step_tensors(self, grads: Optional[Sequence[Optional[torch.Tensor]]] = None, *, scale: float = 1.0,
                     stream=None, process_group=None, accumulated: bool = False,
                     loss_scale=None) -> zs.NormResult:
        """One step straight from per-tensor grads: a norm pass reads the grads through
        the FlatParameter table without writing them, then AdamW reads them again
        through the table.  No fp32 flat grad is written (30 instead of 36 bytes per
        parameter); the result is bit-identical to flatten(scale) + step().

        accumulated: these grads are the step's LAST micro-batch, and the grad buffer
        already holds the earlier ones (flatten()/accum() with accumulate=True after
        the first, without fuse_norm).  The norm pass and AdamW then add them to the
        buffer on the fly and the last micro-batch is never written (6 + 32 instead
        of 10 + 30 bytes per parameter); bit-identical to flatten(accumulate=True,
        scale) + step().

        loss_scale: a DeviceLossScale, as for flatten(): both passes read its unscale
        factor on the device and the norm pass raises its overflow flag; `scale` is
        ignored."""
        self.launch_step_tensors(grads, scale=scale, stream=stream, process_group=process_group,
                                 accumulated=accumulated, loss_scale=loss_scale)
        return self.finish_step(stream)

    def launch_step_tensors(self, grads: Optional[Sequence[Optional[torch.Tensor]]] = None, *, scale: float = 1.0,
                            stream=None, process_group=None, accumulated: bool = False, loss_scale=None) -> None:
        """Enqueue step_tensors() without waiting (capturable with registered grads)."""
        table, count, dt = self._resolve(grads)
        self._launch_direct(table, count, self.total, dt, self.glo, self.ghi, self.start, scale, accumulated, stream,
                            process_group, loss_scale)

    def step_flat(self, flat_src: torch.Tensor, *, scale: float = 1.0, stream=None, process_group=None,
                  accumulated: bool = False, loss_scale=None) -> zs.NormResult:
        """step_tensors() for a flat low-precision grad covering the grad range (what
        accum() takes: ZeRO-2/3 and FSDP, where the rank receives its shard's grads
        already flat): the last micro-batch is read by the norm pass and by AdamW and
        never written.  Bit-identical to accum(flat_src, accumulate=accumulated,
        scale) + step()."""
        self.launch_step_flat(flat_src, scale=scale, stream=stream, process_group=process_group,
                              accumulated=accumulated, loss_scale=loss_scale)
        return self.finish_step(stream)

    def launch_step_flat(self, flat_src: torch.Tensor, *, scale: float = 1.0, stream=None, process_group=None,
                         accumulated: bool = False, loss_scale=None) -> None:
        """Enqueue step_flat() without waiting (capturable once device_flat_table(flat_src)
        has been called outside the capture)."""
        table = self.device_flat_table(flat_src)
        span = self.ghi - self.glo
        self._launch_direct(table, 1, span, flat_src.dtype, 0, span, self.start - self.glo, scale, accumulated, stream,
                            process_group, loss_scale)

    def device_flat_table(self, flat_src: torch.Tensor) -> torch.Tensor:
        """The one-entry tensor table of a flat grad over the grad range, in device memory
        (built once per address and cached; call it before a CUDA graph capture)."""
        span = self.ghi - self.glo
        if flat_src.numel() != span or flat_src.dim() != 1:
            raise ValueError(f"flat_src must be 1-D with the grad range's {span} elements")
        key = (flat_src.data_ptr(), flat_src.numel(), flat_src.is_contiguous())
        hit = self._flat_tables.get(key)
        if hit is None:
            table, total = zs.zero_tensor_table([flat_src], [span])
            assert total == span
            hit = zs.device_table(table, 1, self.device)
            if len(self._flat_tables) > 64:
                self._flat_tables.clear()
            self._flat_tables[key] = hit
        return hit

    def _launch_direct(self, table, count: int, total: int, dt, lo: int, hi: int, shard_start: int, scale: float,
                       accumulated: bool, stream, process_group, loss_scale=None) -> None:
        """The direct path over a tensor table: flat indices [lo, hi) are the grad range,
        [shard_start, shard_start + n) the shard."""
        if accumulated and self.grad.numel() != self.ghi - self.glo:
            raise ValueError("accumulated=True needs the grad buffer (grad_buffer=True)")
        sc, dsc, flag = self._scale_args(scale, loss_scale)
        if accumulated:
            zs.zero_flatten_cast(table, count, total, dt, lo, hi, sc, zs.NORM_OF_SUM, self.grad, flag, self.ws, stream,
                                 d_scale=dsc)
        else:
            zs.zero_flatten_cast(table, count, total, dt, lo, hi, sc, False, None, flag, self.ws, stream, d_scale=dsc)
        if process_group is not None and self.glo == self.start and _world(process_group) > 1:
            if self._local_buf is None:
                self._local_buf = zs.new_norm_result(self.device)
            st = torch_stream(stream, self.device)
            zs.zero_grad_sqnorm_finalize(self.ws, self.ghi - self.glo, 0.0, math.inf, self._local_buf, st)
            gathered = self._global_norm(zs.sqnorm_view(self._local_buf), process_group, st)
            zs.zero_grad_sqnorm_combine(gathered, self.max_norm, self.norm_buf, st)
        else:
            zs.zero_grad_sqnorm_finalize(self.ws, self.ghi - self.glo, 0.0, self.max_norm, self.norm_buf, stream)
        self._norm_ready = False
        acc = self.shard_grad() if accumulated else None
        if self.capturable:
            zs.zero_adamw_prepare_device(self._dev_hp, self.norm_buf, self._dev_state, stream)
            zs.zero_adamw_step_tensors_device(self.master, self.exp_avg, self.exp_avg_sq, table, count, total,
                                              dt, shard_start, sc, self.lowp, self._dev_state, self.norm_buf,
                                              stream, acc=acc, d_scale=dsc)
        else:
            zs.zero_adamw_step_tensors(self.master, self.exp_avg, self.exp_avg_sq, table, count, total, dt,
                                       shard_start, sc, self.lowp, self.lr, self.betas[0], self.betas[1],
                                       self.eps, self.weight_decay, self._t + 1, self.norm_buf, stream, acc=acc,
                                       d_scale=dsc)

    # -------------------------------------------------------- checkpoint
    def state_dict(self) -> dict:
        """The rank's optimizer state on the host: step counter, fp32 master /
        exp_avg / exp_avg_sq and the low-precision copy (a flat shard each)."""
        sd = {"t": self.t, "start": self.start, "end": self.end, "master": self.master.cpu(),
              "exp_avg": self.exp_avg.cpu(), "exp_avg_sq": self.exp_avg_sq.cpu()}
        if self.lowp is not None:
            sd["lowp"] = self.lowp.cpu()
        return sd

    def load_state_dict(self, sd: dict) -> None:
        if (sd["start"], sd["end"]) != (self.start, self.end):
            raise ValueError("state belongs to another shard")
        self.t = int(sd["t"])
        self.master.copy_(sd["master"])
        self.exp_avg.copy_(sd["exp_avg"])
        self.exp_avg_sq.copy_(sd["exp_avg_sq"])
        if self.lowp is not None and "lowp" in sd:
            self.lowp.copy_(sd["lowp"])

    def resident_bytes(self) -> int:
        """Device bytes this rank holds for the step (grad + state + low-precision copy)."""
        b = 4 * (self.grad.numel() + 3 * self.n)  # grad is empty without a grad buffer
        if self.lowp is not None:
            b += self.lowp.numel() * self.lowp.element_size()
        return b


def _world(group) -> int:
    import torch.distributed as dist
    return dist.get_world_size(group)


def torch_stream(stream, device) -> torch.cuda.Stream:
    """A torch stream object for a stream argument of this package: None (the
    current stream of `device`), a torch.cuda.Stream, or a raw cudaStream_t
    handle (wrapped, not owned)."""
    if stream is None:
        return torch.cuda.current_stream(device)
    if isinstance(stream, torch.cuda.Stream):
        return stream
    return torch.cuda.ExternalStream(int(stream), device=device)


def _backend(group) -> str:
    import torch.distributed as dist
    return str(dist.get_backend(group)).lower()


def gather_sqnorms(local: torch.Tensor, group) -> torch.Tensor:
    """All-gather every rank's 1-element float64 sum of squares, in rank order.

    The step's norm exchange (8 bytes per rank).  With NCCL the device tensor
    is gathered directly, ordered on torch's current stream.  With a backend
    that works on host memory (gloo) a device value is staged through the host:
    the copy out waits for the current stream, and the gathered vector is
    copied back to the device on it.  Run it under ``torch.cuda.stream(s)`` to
    order it on another stream s."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    staged = local.is_cuda and _backend(group) != "nccl"
    x = local.detach().to("cpu") if staged else local.contiguous()
    parts = [torch.empty_like(x) for _ in range(world)]
    dist.all_gather(parts, x, group=group)
    out = torch.cat(parts)
    return out.to(local.device) if staged else out
