"""ZeRO-2/3 data plane of one rank: the exchanges around the flat-shard step.

The ZeRO page's ZeRO-2 step (section "ZeRO-2: 附加切分梯度",
ZeRO2Optimizer: reduce_gradients, step, _allgather_params) and the
memory-ledger page's FlatParameter (section "FSDP 的关键抽象：FlatParameter":
one large reduce-scatter and one all-gather per FlatParameter; MixedPrecision:
reduce in fp32), laid out for one GPU per rank:

  1. backward leaves every rank's grads in its full flat low-precision grad
     ``flat_grad`` (the FlatParameter's grad, padded to world_size equal
     chunks; the padding stays zero);
  2. exchange: an all-to-all of that buffer, so that each rank receives every
     rank's chunk of its own shard -- the data movement of a reduce-scatter,
     in the grads' own 16-bit type;
  3. reduce: ``zero_reduce_chunks`` adds the received chunks in rank order
     in fp32, each scaled by 1/world_size (the page's SUM then
     /= world_size), into the rank's fp32 shard grad, with the grad norm's
     tile partials fused into the same pass on the last micro-batch;
  4. step: the global norm (8-byte all-gather of the ranks' local sums of
     squares, combined in rank order) and AdamW on the shard
     (``FlatShardAdamW``), whose low-precision write-back lands directly in
     this rank's slice of the full low-precision FlatParameter ``flat_param``;
  5. all-gather of the slices in place, so that every rank holds the whole
     updated low-precision FlatParameter for the next forward.

Summing in a kernel of this library instead of inside the collective keeps
the reduction in fp32 and in rank order -- deterministic, and the same bits
on every rank and every run -- while the wire carries 2 bytes per element.
The collectives are torch.distributed calls (NCCL on device buffers; with a
backend that works on host memory, such as gloo, device buffers are staged
through the host); every arithmetic step runs in libzeroshard's kernels.
"""
from __future__ import annotations

import contextlib
import math
from typing import List, Optional, Sequence, Tuple

import torch

from . import zero_shard as zs
from .optimizer import FlatShardAdamW, gather_sqnorms, torch_stream


def chunk_layout(total: int, world_size: int) -> Tuple[int, int]:
    """(chunk, padded): the ZeRO page's chunk = ceil(total / world_size) (the
    length of rank 0's shard) and the padded length world_size * chunk that an
    exchange of equal chunks needs."""
    s0, e0 = zs.zero_shard_range(total, world_size, 0)
    chunk = e0 - s0
    return chunk, chunk * world_size


def _staged(t: torch.Tensor, group) -> bool:
    import torch.distributed as dist
    return t.is_cuda and str(dist.get_backend(group)).lower() != "nccl"


def exchange_chunks(send: torch.Tensor, recv: torch.Tensor, group) -> None:
    """All-to-all of equal chunks: block j of `recv` receives block `rank` of
    rank j's `send` (both 1-D, world_size * chunk elements).  Ordered on torch's
    current stream."""
    import torch.distributed as dist
    if send.numel() != recv.numel() or send.dtype != recv.dtype:
        raise ValueError("send and recv must match in size and dtype")
    if _staged(send, group):
        host_recv = torch.empty(recv.shape, dtype=recv.dtype)
        dist.all_to_all_single(host_recv, send.to("cpu"), group=group)
        recv.copy_(host_recv)
    else:
        dist.all_to_all_single(recv, send, group=group)


def gather_shards(full: torch.Tensor, group) -> None:
    """In-place all-gather: block r of `full` (world_size equal blocks) is
    replaced by rank r's block.  Ordered on torch's current stream."""
    import torch.distributed as dist
    world, rank = dist.get_world_size(group), dist.get_rank(group)
    if full.numel() % world:
        raise ValueError("full is not world_size equal blocks")
    chunk = full.numel() // world
    mine = full[rank * chunk:(rank + 1) * chunk]
    if _staged(full, group):
        host = torch.empty(full.shape, dtype=full.dtype)
        dist.all_gather_into_tensor(host, mine.to("cpu"), group=group)
        full.copy_(host)
    else:
        dist.all_gather_into_tensor(full, mine, group=group)


class ZeroDataPlane:
    """One rank's ZeRO-2/3 step with its exchanges (see the module docstring).

    numels: the FlatParameter's tensor sizes in order.  group: a
    torch.distributed process group (world size and rank come from it); None
    means one rank.  ``flat_grad`` is where backward writes the grads
    (``grad_views()`` gives the per-tensor views); ``flat_param`` is the full
    low-precision FlatParameter (``param_views()``).  Other keyword arguments
    go to FlatShardAdamW (lr, betas, eps, weight_decay, max_norm, master,
    capturable)."""

    def __init__(self, numels: Sequence[int], *, group=None, grad_dtype: torch.dtype = torch.bfloat16,
                 lowp_dtype: torch.dtype = torch.bfloat16, device="cuda", **adam_kw):
        import torch.distributed as dist
        self.group = group
        if group is not None:
            self.world_size, self.rank = dist.get_world_size(group), dist.get_rank(group)
        else:
            self.world_size, self.rank = 1, 0
        self.device = torch.device(device)
        self.numels = [int(n) for n in numels]
        self.total = int(sum(self.numels))
        self.chunk, self.padded = chunk_layout(self.total, self.world_size)
        self.flat_param = torch.zeros(self.padded, dtype=lowp_dtype, device=self.device)
        self.flat_grad = torch.zeros(self.padded, dtype=grad_dtype, device=self.device)
        self.recv = torch.empty(self.padded if self.world_size > 1 else 0, dtype=grad_dtype, device=self.device)
        start, end = zs.zero_shard_range(self.total, self.world_size, self.rank)
        self.opt = FlatShardAdamW(self.numels, world_size=self.world_size, rank=self.rank, grad_range="shard",
                                  device=self.device, lowp_out=self.flat_param[start:end], **adam_kw)

    # ---------------------------------------------------------------- views
    def _views(self, flat: torch.Tensor) -> List[torch.Tensor]:
        out, pos = [], 0
        for n in self.numels:
            out.append(flat[pos:pos + n])
            pos += n
        return out

    def grad_views(self) -> List[torch.Tensor]:
        """Per-tensor views of flat_grad, in FlatParameter order (what backward fills)."""
        return self._views(self.flat_grad)

    def param_views(self) -> List[torch.Tensor]:
        """Per-tensor views of the full low-precision FlatParameter."""
        return self._views(self.flat_param)

    # ---------------------------------------------------------------- steps
    def reduce_scatter_grads(self, *, accumulate: bool = False, scale: Optional[float] = None,
                             fuse_norm: bool = True, stream=None) -> None:
        """Exchange flat_grad's chunks and reduce this rank's in fp32 into its shard grad.

        scale: defaults to 1/world_size (the page's average); with micro-batches
        reduced one at a time pass 1/(world_size * accum_steps), accumulate=True
        after the first, and fuse_norm only on the last."""
        opt = self.opt
        st = torch_stream(stream, self.device)
        sc = 1.0 / self.world_size if scale is None else float(scale)
        if self.world_size > 1:
            with torch.cuda.stream(st):
                exchange_chunks(self.flat_grad, self.recv, self.group)
            chunks = self.recv.view(self.world_size, self.chunk)
        else:
            chunks = self.flat_grad.view(1, self.padded)
        opt.reduce(chunks, accumulate=accumulate, scale=sc, fuse_norm=fuse_norm, stream=st)

    def _on(self, stream):
        """Order host-issued collectives on `stream` (device buffers); host buffers need nothing."""
        if self.device.type != "cuda":
            return contextlib.nullcontext()
        return torch.cuda.stream(torch_stream(stream, self.device))

    def all_gather_params(self, stream=None) -> None:
        """Every rank's updated low-precision slice into every rank's flat_param."""
        if self.world_size > 1:
            with self._on(stream):
                gather_shards(self.flat_param, self.group)

    def step(self, stream=None) -> zs.NormResult:
        """Clip with the global norm, AdamW on the shard, then all-gather the
        updated parameters (skipped with the step when the norm is not finite)."""
        r = self.opt.step(stream=stream, process_group=self.group)
        if r.finite:
            self.all_gather_params(stream)
        return r

    # ------------------------------------------------------------ checkpoint
    def state_dict(self) -> dict:
        """This rank's checkpoint: its optimizer shard (step count, fp32 master /
        exp_avg / exp_avg_sq, its low-precision slice) and the layout it belongs to."""
        sd = self.opt.state_dict()
        sd.update(world_size=self.world_size, rank=self.rank, total=self.total)
        return sd

    def load_state_dict(self, sd: dict, stream=None) -> None:
        """Restore this rank's shard, then all-gather the low-precision slices so that
        flat_param holds every rank's parameters again (every rank must call it)."""
        if (sd["world_size"], sd["rank"], sd["total"]) != (self.world_size, self.rank, self.total):
            raise ValueError("checkpoint of another layout (world size, rank or parameter count)")
        self.opt.load_state_dict(sd)
        self.all_gather_params(stream)

    def resident_bytes(self) -> int:
        """Device bytes of this rank: the shard's fp32 state and grad plus the full
        low-precision grad, receive buffer and parameters."""
        b = self.opt.resident_bytes() - (self.opt.lowp.numel() * self.opt.lowp.element_size())
        for t in (self.flat_param, self.flat_grad, self.recv):
            b += t.numel() * t.element_size()
        return b


class ZeroUnits:
    """A model wrapped as several FSDP units, one FlatParameter each, stepped together.

    The memory-ledger page (section "FSDP 的关键抽象：FlatParameter") wraps one unit per
    transformer block: each unit's parameters are flattened into their own FlatParameter,
    sharded and exchanged on their own (a ZeroDataPlane here), so that no all-gather ever
    has to hold the whole model.  clip_grad_norm_ still spans every parameter of the
    model.  The units' norm partials (fused into their reductions) go to consecutive
    slices of one shared workspace, so one finalize gives this rank's sum of squares over
    every unit; the ranks exchange those 8-byte values once; unit 0 combines them in rank
    order and every other unit's AdamW reads unit 0's result -- one norm, one
    coefficient and one skip decision for the whole model, in 2 launches plus one
    reduction and one AdamW per unit.

    units: the tensor sizes of each unit's FlatParameter; masters: each unit's fp32
    shard (optional); other keyword arguments go to every ZeroDataPlane."""

    def __init__(self, units: Sequence[Sequence[int]], *, group=None, masters: Optional[Sequence[torch.Tensor]] = None,
                 device="cuda", **kw):
        import torch.distributed as dist
        if masters is not None and len(masters) != len(units):
            raise ValueError("one master shard per unit")
        self.group = group
        world = dist.get_world_size(group) if group is not None else 1
        rank = dist.get_rank(group) if group is not None else 0
        dev = torch.device(device)
        # every unit's norm partials in consecutive slices of one workspace (8 bytes per tile)
        sizes = []
        for numels in units:
            s, e = zs.zero_shard_range(int(sum(numels)), world, rank)
            sizes.append(zs.zero_grad_sqnorm_workspace_bytes(e - s))
        self.ws = torch.empty(max(sum(sizes), 8), dtype=torch.uint8, device=dev)
        self.ws_tiles = sum(sizes) // 8
        offs = [0]
        for b in sizes:
            offs.append(offs[-1] + b)
        self.units = [ZeroDataPlane(numels, group=group, device=dev,
                                    master=None if masters is None else masters[i],
                                    workspace=self.ws[offs[i]:offs[i + 1]] if sizes[i] else None, **kw)
                      for i, numels in enumerate(units)]
        self._local = zs.new_norm_result(dev)

    def reduce_scatter_grads(self, **kw) -> None:
        """Every unit's exchange and reduction (ZeroDataPlane.reduce_scatter_grads); the
        norm partials are fused into the last micro-batch's reduction (fuse_norm)."""
        for u in self.units:
            u.reduce_scatter_grads(**kw)

    def launch_step(self, stream=None) -> None:
        """Enqueue the model's norm and every unit's AdamW without any host read (with
        capturable=True units the step count and skip decision stay on the device, so
        the reductions and this can be captured in one CUDA graph); read the result with
        finish_step()."""
        head = self.units[0]
        st = torch_stream(stream, head.device)
        self._launch(st)

    def finish_step(self, stream=None) -> zs.NormResult:
        """Read the step's result once for every unit (a device-to-host copy)."""
        head = self.units[0]
        st = torch_stream(stream, head.device)
        result = head.opt.finish_step(st)
        for u in self.units[1:]:
            u.opt.finish_step(st, result=result)
        return result

    def _launch(self, st) -> None:
        head = self.units[0]
        for u in self.units:  # a unit whose last reduction did not fuse the norm: its partials now
            if not u.opt._norm_ready and u.opt.n > 0:
                zs.zero_grad_sqnorm(u.opt.grad, 0.0, math.inf, u.opt.ws, self._local, st)
        # this rank's sum of squares over every unit's tiles (a tile count in elements)
        zs.zero_grad_sqnorm_finalize(self.ws, self.ws_tiles * 32768, 0.0, math.inf, self._local, st)
        local = zs.sqnorm_view(self._local)
        if head.world_size > 1:
            with torch.cuda.stream(st):
                gathered = gather_sqnorms(local, self.group)
        else:
            gathered = local
        head.opt.launch_step(stream=st, gathered_sqnorms=gathered)
        for u in self.units[1:]:
            u.opt.launch_step(stream=st, norm_result=head.opt.norm_buf)
        for u in self.units:
            u.opt._norm_ready = False

    def step(self, stream=None) -> zs.NormResult:
        """One step of every unit with the model's global norm; the units' parameters are
        all-gathered afterwards (nothing changes, and nothing is gathered, when the norm
        is not finite)."""
        head = self.units[0]
        st = torch_stream(stream, head.device)
        self._launch(st)
        result = self.finish_step(st)  # every unit used the same result: one device-to-host read
        if result.finite:
            for u in self.units:
                u.all_gather_params(st)
        return result
