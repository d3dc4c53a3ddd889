"""Synthetic workloads and seeded input generators for the flat-shard optimizer step.

This module only describes workloads (parameter-tensor shapes in FlatParameter
order, dtypes, hyper-parameters, step counts) and draws their random inputs.
It holds none of the method's arithmetic: no shard range, no flat offsets, no
casts, sums, norms or Adam update.  Both the CUDA path (tests, bench) and the
CPU oracle (tests) take their inputs from here, so that the two sides see the
same numbers while sharing no code.

Determinism: every random draw is keyed by (seed, stream, chunk index) and made
with a fresh ``torch.Generator`` per chunk of ``CHUNK`` elements, so a slice
[a, b) of a flat quantity is the same whether it is drawn alone or as part of
a larger range.  CPU and CUDA generators give different streams for the same
key; a test that compares the two sides draws once and copies.

Workload shapes follow the parameter lists of the models the pages train:
Llama-7B / Llama-13B (page "cann-recipes-train ZeRO", section on the Llama-7B
recipe; page on gradient accumulation for LLaMA-13B), GPT-2 small, and a
ragged multi-tensor stress list.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

CHUNK = 1 << 20  # elements per independently seeded draw

# stream identifiers for the key (seed, stream, chunk)
_STREAM_PARAM = 1
_STREAM_GRAD = 2


# --------------------------------------------------------------------------- shapes
def llama_numels(layers: int, hidden: int, mlp: int, vocab: int) -> List[int]:
    """Llama parameter sizes in HF module order (untied lm_head, RMSNorm weights).

    embed [V,h]; per layer q,k,v,o [h,h], gate [f,h], up [f,h], down [h,f],
    input norm [h], post-attention norm [h]; final norm [h]; lm_head [V,h].
    """
    out = [vocab * hidden]
    for _ in range(layers):
        out += [hidden * hidden] * 4
        out += [mlp * hidden] * 3
        out += [hidden, hidden]
    out += [hidden, vocab * hidden]
    return out


def gpt2_numels(layers: int = 12, hidden: int = 768, vocab: int = 50257, ctx: int = 1024) -> List[int]:
    """GPT-2 parameter sizes in HF order: wte, wpe, 12 x block, ln_f (w, b)."""
    h = hidden
    out = [vocab * h, ctx * h]
    for _ in range(layers):
        out += [h, h,                 # ln_1 weight, bias
                h * 3 * h, 3 * h,     # attn c_attn weight, bias
                h * h, h,             # attn c_proj weight, bias
                h, h,                 # ln_2 weight, bias
                h * 4 * h, 4 * h,     # mlp c_fc weight, bias
                4 * h * h, h]         # mlp c_proj weight, bias
    out += [h, h]
    return out


def ragged_numels(n_tensors: int = 20000, seed: int = 0, max_log2: int = 20) -> List[int]:
    """Log-uniform sizes floor(exp(U(0, max_log2 * ln 2))) in [1, 2^max_log2), numpy PCG64."""
    rng = np.random.Generator(np.random.PCG64(seed))
    u = rng.uniform(0.0, max_log2 * math.log(2.0), size=n_tensors)
    return [max(1, int(math.floor(math.exp(x)))) for x in u]


# ------------------------------------------------------------------------ workloads
@dataclass(frozen=True)
class Workload:
    """One synthetic configuration of the flat-shard AdamW step.

    mode:
      "flat"  - per-tensor grads flattened over this rank's shard; norm over the shard.
      "zero1" - per-tensor grads flattened over the whole buffer (every rank holds the
                full averaged grad), global norm over the whole buffer, update of the
                rank's shard only (page "cann-recipes-train ZeRO", ZeRO-1 step()).
      "zero3" - the rank receives flat grads of its own shard only (the output of a
                reduce-scatter), accumulated flat; norm over the shard.
    """
    name: str
    numels: Tuple[int, ...]
    grad_dtype: str                 # "f32" | "bf16" | "f16"
    world_size: int
    rank: int
    micro_batches: int
    mode: str
    lr: float
    betas: Tuple[float, float]
    eps: float
    weight_decay: float
    max_norm: float                 # math.inf: no clipping
    steps: int
    grad_std: float
    grad_dist: str = "normal"       # "normal" | "student_t3"
    zero_frac: float = 0.0          # fraction of grads set to exactly 0
    init_std: float = 0.02
    seed: int = 0
    lowp_dtype: str = "bf16"        # low-precision parameter copy written by the step
    null_grads: Tuple[int, ...] = ()  # tensor indices that carry no grad (read as zeros)

    @property
    def total(self) -> int:
        return int(sum(self.numels))

    @property
    def n_tensors(self) -> int:
        return len(self.numels)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


def tiny() -> Workload:
    """4 fp32 tensors, 1,261,891 params (not a multiple of 8); N=1; 3 steps; no clipping."""
    return Workload(name="tiny", numels=(262144, 262144, 262144, 475459), grad_dtype="f32",
                    world_size=1, rank=0, micro_batches=1, mode="flat",
                    lr=1e-4, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01,
                    max_norm=math.inf, steps=3, grad_std=0.02)


def gpt2_zero1() -> Workload:
    """GPT-2 small (148 tensors, 124,439,808 params), ZeRO-1 rank 3 of 8, bf16 grads x 8 micro-batches."""
    return Workload(name="gpt2_zero1_r3of8", numels=tuple(gpt2_numels()), grad_dtype="bf16",
                    world_size=8, rank=3, micro_batches=8, mode="zero1",
                    lr=1e-4, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.0,
                    max_norm=1.0, steps=10, grad_std=1e-3)


def llama7b() -> Workload:
    """Llama-7B-shaped flat buffer (291 tensors, 6,738,415,616 params), N=1, bf16 grads."""
    return Workload(name="llama7b_flat", numels=tuple(llama_numels(32, 4096, 11008, 32000)),
                    grad_dtype="bf16", world_size=1, rank=0, micro_batches=1, mode="flat",
                    lr=3e-4, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1,
                    max_norm=1.0, steps=5, grad_std=1e-4)


def llama13b_zero3() -> Workload:
    """Llama-13B-shaped (363 tensors), ZeRO-3 rank 7 of 8: fp16 flat shard grads x 8 micro-batches."""
    return Workload(name="llama13b_zero3_r7of8", numels=tuple(llama_numels(40, 5120, 13824, 32000)),
                    grad_dtype="f16", world_size=8, rank=7, micro_batches=8, mode="zero3",
                    lr=3e-4, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1,
                    max_norm=1.0, steps=20, grad_std=5e-4)


def ragged() -> Workload:
    """20,000 log-uniform tensors, rank 2 of 4, Student-t(3) bf16 grads with 1% exact zeros."""
    return Workload(name="ragged_r2of4", numels=tuple(ragged_numels()), grad_dtype="bf16",
                    world_size=4, rank=2, micro_batches=1, mode="flat",
                    lr=1e-4, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.05,
                    max_norm=0.5, steps=5, grad_std=1e-3, grad_dist="student_t3",
                    zero_frac=0.01)


ALL = {w().name: w for w in (tiny, gpt2_zero1, llama7b, llama13b_zero3, ragged)}


def llama13b_zero3_f16chunk() -> Workload:
    """The Llama-13B ZeRO-3 rank with the ZeRO page's ZeRO-3 update (section "ZeRO-3: 切分参数"):
    the rank's low-precision parameter chunk is fp16, and the page's Adam has no weight decay."""
    return llama13b_zero3().with_(name="llama13b_zero3_r7of8_f16chunk", lowp_dtype="f16", weight_decay=0.0)


# variants of the five configurations (bench lines and parity tests, not configurations of their own)
VARIANTS = {w().name: w for w in (llama13b_zero3_f16chunk,)}


def small_llama(layers: int = 2, hidden: int = 256, mlp: int = 688, vocab: int = 1000, **kw) -> Workload:
    """A Llama-shaped list small enough for the oracle to finish in seconds."""
    base = llama7b().with_(name=f"llama_l{layers}_h{hidden}",
                           numels=tuple(llama_numels(layers, hidden, mlp, vocab)))
    return base.with_(**kw) if kw else base


def small_ragged(n_tensors: int = 600, seed: int = 3, max_log2: int = 12, **kw) -> Workload:
    base = ragged().with_(name=f"ragged_{n_tensors}", numels=tuple(ragged_numels(n_tensors, seed, max_log2)))
    return base.with_(**kw) if kw else base


# ----------------------------------------------------------------------- generators
_TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def torch_dtype(name: str) -> torch.dtype:
    return _TORCH_DTYPE[name]


def _key(seed: int, stream: int, a: int, b: int, chunk: int) -> int:
    # a plain mixing of small integers into a 63-bit seed (splitmix64 finaliser)
    x = (seed * 0x9E3779B97F4A7C15 + stream * 0xBF58476D1CE4E5B9 + a * 0x94D049BB133111EB
         + b * 0x2545F4914F6CDD1D + chunk * 0xD6E8FEB86659FD93) & 0xFFFFFFFFFFFFFFFF
    x ^= x >> 30
    x = (x * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
    x ^= x >> 27
    x = (x * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
    x ^= x >> 31
    return x & 0x7FFFFFFFFFFFFFFF


def _fill(out: torch.Tensor, lo: int, hi: int, key_fn, draw) -> None:
    """Fill out[0:hi-lo] with draw(n, generator) for logical positions [lo, hi), chunk-keyed."""
    dev = out.device
    c0, c1 = lo // CHUNK, (hi - 1) // CHUNK if hi > lo else lo // CHUNK - 1
    for c in range(c0, c1 + 1):
        a, b = max(lo, c * CHUNK), min(hi, (c + 1) * CHUNK)
        g = torch.Generator(device=dev)
        g.manual_seed(key_fn(c))
        vals = draw(CHUNK, g)  # always draw the whole chunk: slices stay consistent
        out[a - lo:b - lo].copy_(vals[a - c * CHUNK:b - c * CHUNK])


def _draw_fn(dist: str, std: float, zero_frac: float, dev):
    def draw(n, g):
        if dist == "normal":
            x = torch.randn(n, generator=g, device=dev, dtype=torch.float32) * std
        elif dist == "student_t3":
            z = torch.randn(n, generator=g, device=dev, dtype=torch.float32)
            w = torch.randn(3, n, generator=g, device=dev, dtype=torch.float32)
            chi2 = (w * w).sum(0)
            x = z / torch.sqrt(chi2 / 3.0) * std
        else:
            raise ValueError(dist)
        if zero_frac > 0.0:
            u = torch.rand(n, generator=g, device=dev, dtype=torch.float32)
            x = torch.where(u < zero_frac, torch.zeros_like(x), x)
        return x
    return draw


def master_init(wl: Workload, start: int, end: int, device="cpu") -> torch.Tensor:
    """fp32 master weights for flat positions [start, end): i.i.d. N(0, init_std^2)."""
    out = torch.empty(end - start, dtype=torch.float32, device=device)
    if end > start:
        _fill(out, start, end, lambda c: _key(wl.seed, _STREAM_PARAM, 0, 0, c),
              _draw_fn("normal", wl.init_std, 0.0, out.device))
    return out


def flat_grads(wl: Workload, step: int, micro: int, start: int, end: int, device="cpu",
               out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Flat low-precision grads for flat positions [start, end) of (step, micro-batch)."""
    dt = torch_dtype(wl.grad_dtype)
    if out is None:
        out = torch.empty(end - start, dtype=dt, device=device)
    if end > start:
        _fill(out, start, end, lambda c: _key(wl.seed, _STREAM_GRAD, step, micro, c),
              lambda n, g: _draw_fn(wl.grad_dist, wl.grad_std, wl.zero_frac, out.device)(n, g).to(dt))
    return out


@dataclass
class TensorGrads:
    """Per-tensor grads of one micro-batch, as views into one padded storage buffer.

    Each tensor starts at a multiple of ``align`` elements inside ``storage`` (as
    separate allocations would), so tensor starts are aligned while flat offsets
    are not.  ``tensors[i] is None`` for tensors that carry no grad.
    """
    storage: torch.Tensor
    starts: List[int]
    tensors: List[Optional[torch.Tensor]] = field(default_factory=list)


def padded_layout(numels: Sequence[int], align: int = 128) -> Tuple[List[int], int]:
    """Storage start of each tensor when each is placed on an ``align``-element boundary."""
    starts, pos = [], 0
    for n in numels:
        starts.append(pos)
        pos += (int(n) + align - 1) // align * align
    return starts, pos


def tensor_grads(wl: Workload, step: int, micro: int, device="cpu", align: int = 128,
                 storage: Optional[torch.Tensor] = None) -> TensorGrads:
    """Per-tensor grads of (step, micro-batch) for every tensor of the workload."""
    starts, size = padded_layout(wl.numels, align)
    dt = torch_dtype(wl.grad_dtype)
    if storage is None:
        storage = torch.empty(size, dtype=dt, device=device)
    assert storage.numel() >= size and storage.dtype == dt
    if size:
        _fill(storage[:size], 0, size, lambda c: _key(wl.seed, _STREAM_GRAD, step, micro, c),
              lambda n, g: _draw_fn(wl.grad_dist, wl.grad_std, wl.zero_frac, storage.device)(n, g).to(dt))
    nulls = set(wl.null_grads)
    tensors = [None if i in nulls else storage[s:s + n] for i, (s, n) in enumerate(zip(starts, wl.numels))]
    return TensorGrads(storage=storage, starts=starts, tensors=tensors)
