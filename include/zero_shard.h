/*
 * zero_shard.h -- C ABI of libzeroshard: one data-parallel rank's optimizer
 * step over its flat 1-D shard (ZeRO-1/2/3, FSDP FlatParameter), on one GPU.
 *
 * The step has four parts, each one call below:
 *   zero_flatten_cast  per-tensor grads -> the rank's flat fp32 grad shard
 *                      (optionally accumulating micro-batches, scaled)
 *   zero_accum         flat low-precision grads -> flat fp32 accumulator
 *   zero_grad_sqnorm   global L2 grad norm and the clip coefficient
 *   zero_adamw_step    fused bias-corrected AdamW on fp32 master / exp_avg /
 *                      exp_avg_sq with a bf16 (or f16) parameter write-back
 * plus the host-only helpers zero_shard_range and zero_tensor_table.  Around
 * them: zero_reduce_chunks (the local reduction of a ZeRO-2/3 reduce-scatter),
 * zero_grad_sqnorm_finalize / _combine (the norm from fused partials and from
 * the ranks' sums), the loss-scale updates (host and device), the AdamW
 * variants that read the grads through the tensor table or take their
 * scalars from a device step state (graph-capturable steps), and
 * zero_grad_sqnorm_noalloc.
 *
 * Sources: the ZeRO page (ai6s.net, "cann-recipes-train" ZeRO-1/2/3 on
 * Ascend), the memory-ledger / FlatParameter page (ybb.press,
 * "大模型分布式训练并行与显存工程实战") and the LLaMA-13B gradient accumulation
 * page (ai6s.net).  Each entry point names the passage that defines it.
 *
 * Conventions for every call:
 *  - Memory.  The library allocates nothing (device or host) and keeps no
 *    state between calls (beyond the fixed scratch array of
 *    zero_grad_sqnorm_noalloc and the debug build's violation record).  The
 *    caller owns every buffer.  Pointers prefixed d_ are device addresses;
 *    everything else is host memory.
 *  - Streams.  `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *    default stream).  Device work is enqueued asynchronously on it; no call
 *    synchronises the host except where stated.
 *  - Errors.  Arguments are checked on the host before anything is launched;
 *    a bad argument returns ZERO_EINVAL and launches nothing.  A CUDA error
 *    reported by the launch returns ZERO_ECUDA.  zero_last_error() gives a
 *    readable message for the calling thread's last failure.
 *  - n == 0 (or an empty shard) is a valid no-op that returns ZERO_OK.
 *  - Alignment.  Any element-aligned address is accepted.  The fast paths
 *    need 32-byte aligned fp32 buffers; other alignments take slower but
 *    equally exact paths.
 *  - Aliasing.  Outputs must not overlap inputs, except where a buffer is
 *    updated in place by design (d_dst with accumulate, d_acc, the AdamW
 *    state).
 *  - Floating point.  Every result is reproducible bit for bit run to run;
 *    no call uses atomics on floating-point data.
 */
#ifndef ZERO_SHARD_H_
#define ZERO_SHARD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum zero_status {
  ZERO_OK = 0,
  ZERO_EINVAL = 1, /* invalid argument; nothing was launched */
  ZERO_ECUDA = 2   /* the CUDA runtime reported an error */
} zero_status;

typedef enum zero_dtype {
  ZERO_F32 = 0,
  ZERO_BF16 = 1,
  ZERO_F16 = 2
} zero_dtype;

/* One parameter's gradient in the FlatParameter layout.  ptr == NULL means
 * the parameter has no grad; it reads as zeros (the ZeRO page's
 * _flatten_gradients fills such a tensor with torch.zeros). */
typedef struct zero_tensor {
  const void* ptr;     /* address of element 0, contiguous: device memory, or pinned
                          host memory (mapped at the same address; the kernel then
                          reads it over the host link, fusing the transfer) */
  int64_t numel;       /* number of elements, >= 0 */
  int64_t flat_offset; /* start of this tensor in the flat buffer */
} zero_tensor;

/* Result of zero_grad_sqnorm, written to device memory. */
typedef struct zero_norm_result {
  double sqnorm;    /* local sum of squares + extra_sqnorm */
  double norm;      /* sqrt(sqnorm), binary64 */
  float clip_coef;  /* min(1, max_norm / (norm + 1e-6)) in binary32 */
  int32_t finite;   /* 1 if norm is finite; 0 means: skip this step */
} zero_norm_result;

/* AdamW hyper-parameters, binary64 as the user gives them. */
typedef struct zero_adamw_hparams {
  double lr;
  double beta1;
  double beta2;
  double eps;
  double weight_decay; /* 0: plain Adam as in the ZeRO page's step() */
} zero_adamw_hparams;

/* zero_shard_range -- host only.
 * The ZeRO page, section "ZeRO-1: 切分 Optimizer States",
 * ZeRO1Optimizer.__init__: chunk = ceil(total / world_size),
 * start = rank * chunk, end = min(start + chunk, total).  Where
 * rank * chunk > total (few elements, many ranks) the shard is the empty
 * range [total, total).  The flat buffer is never padded: the last shards
 * may be short or empty.
 * Errors: ZERO_EINVAL if start/end is NULL, total < 0, world_size < 1 or
 * rank is not in [0, world_size). */
zero_status zero_shard_range(int64_t total, int32_t world_size, int32_t rank, int64_t* start,
                             int64_t* end);

/* zero_tensor_table -- host only.
 * The FlatParameter layout (memory-ledger page, section "FSDP 的关键抽象：
 * FlatParameter"; the ZeRO page's _flatten_gradients / _apply_update): the
 * parameters are concatenated in list order, so tensor i starts at the sum
 * of the sizes of tensors 0..i-1.  Fills table[i] = {ptrs[i], numels[i],
 * offset_i} for i < n_tensors and *total = sum of numels.  ptrs may be NULL
 * (then every table[i].ptr is NULL) and any ptrs[i] may be NULL.  The
 * caller copies the table to device memory for zero_flatten_cast.
 * Errors: ZERO_EINVAL if table/total/numels is NULL with n_tensors > 0,
 * n_tensors < 0, a numel < 0, or the total overflows int64. */
zero_status zero_tensor_table(const void* const* ptrs, const int64_t* numels, int32_t n_tensors,
                              zero_tensor* table, int64_t* total);

/* zero_flatten_cast -- device.
 * The ZeRO page's _flatten_gradients (each grad viewed 1-D, cast to fp32,
 * concatenated), sliced to the rank's shard (ZeRO1Optimizer.step:
 * flat_grad[start:end]), scaled, and optionally accumulated over
 * micro-batches (the page's GradientAccumulator adds fp32 grads; the
 * gradient-accumulation page divides the loss by accum_steps).  For every
 * flat index k in [shard_start, shard_end), with x the grad element at k
 * (0 when its tensor has no grad):
 *   accumulate == 0:  d_dst[k - shard_start] = fl(scale * x)
 *   accumulate == 1:  d_dst[k - shard_start] = fl(d_dst[...] + fl(scale * x))
 *   accumulate == 2:  the values of accumulate == 1 are formed but not
 *                     stored (d_dst is only read): the norm workspace is
 *                     required and receives their partials.  For the last
 *                     micro-batch of a step whose AdamW adds it to the
 *                     accumulator itself (zero_adamw_step_tensors, d_acc).
 * d_table: device array of n_tensors entries as built by zero_tensor_table
 *   (sorted by flat_offset, contiguous, ending at `total`).
 * src_dtype: dtype of every grad in the table (F32, BF16 or F16).
 * d_dst: fp32, shard_end - shard_start elements; or NULL together with a
 *   norm workspace and accumulate == 0: then only the norm partials of the
 *   values are written (the grad is not materialized -- for a step without
 *   micro-batch accumulation whose update reads the grads through the table,
 *   see zero_adamw_step_tensors).
 * d_scale: NULL, or a device float read when the kernel runs and used in
 *   place of `scale` (the unscale factor of a loss scale kept on the device,
 *   zero_loss_scale_state.unscale, so that a step captured in a CUDA graph
 *   follows the scale's changes; `scale` must still be finite).
 * d_found_nonfinite: NULL, or a device int32 set to 1 when any
 *   fl(scale * x) is inf or NaN (never cleared by the call: zero it first).
 * d_norm_ws: NULL, or a device workspace of at least
 *   zero_grad_sqnorm_workspace_bytes(shard_end - shard_start) bytes
 *   (8-byte aligned).  When given, the same pass also writes the grad
 *   norm's per-tile partials of the values it writes to d_dst -- the very
 *   partials zero_grad_sqnorm would compute from d_dst, bit for bit -- so
 *   that zero_grad_sqnorm_finalize can produce the norm without reading the
 *   grad again.  Pass it on the last micro-batch only.
 * Errors: ZERO_EINVAL for n_tensors < 0, d_table NULL with n_tensors > 0,
 * shard bounds outside 0 <= shard_start <= shard_end <= total, d_dst NULL
 * on a non-empty shard (but for the norm-only pass above), a bad dtype,
 * accumulate not 0/1/2, accumulate == 2 on a non-empty shard without a
 * norm workspace, a non-finite scale, or a too-small / misaligned norm
 * workspace.  The table's contents
 * cannot be checked on the host: a table that does not match `total` or
 * points at too-small buffers is the caller's error and reads out of
 * bounds. */
zero_status zero_flatten_cast(const zero_tensor* d_table, int32_t n_tensors, int64_t total,
                              zero_dtype src_dtype, int64_t shard_start, int64_t shard_end,
                              float scale, const float* d_scale, int32_t accumulate, float* d_dst,
                              int32_t* d_found_nonfinite, void* d_norm_ws, size_t norm_ws_bytes,
                              void* stream);

/* zero_accum -- device.
 * Flat micro-batch accumulation and averaging (the ZeRO page's
 * GradientAccumulator.backward; flat_grad /= world_size; the gradient-
 * accumulation page's loss / accum_steps): for k in [0, n)
 *   accumulate == 0:  d_acc[k] = fl(scale * x[k])
 *   accumulate == 1:  d_acc[k] = fl(d_acc[k] + fl(scale * x[k]))
 * with x = d_src in src_dtype cast exactly to fp32.  This is the ZeRO-2/3
 * case, where the rank receives its shard's grads already flat.
 * d_scale, d_found_nonfinite and d_norm_ws (zero_grad_sqnorm_workspace_
 * bytes(n)) as for zero_flatten_cast.
 * Errors: ZERO_EINVAL for n < 0, NULL buffers with n > 0, a bad dtype,
 * accumulate not 0/1, a non-finite scale, or a too-small / misaligned norm
 * workspace. */
zero_status zero_accum(float* d_acc, const void* d_src, zero_dtype src_dtype, int64_t n, float scale,
                       const float* d_scale, int32_t accumulate, int32_t* d_found_nonfinite, void* d_norm_ws,
                       size_t norm_ws_bytes, void* stream);

/* zero_reduce_chunks -- device.
 * The local half of a ZeRO-2/3 reduce-scatter (the ZeRO page, section
 * "ZeRO-2: 附加切分梯度", ZeRO2Optimizer.reduce_gradients: the ranks' flat
 * grads are summed, each rank keeps its chunk, which is then divided by
 * world_size; the memory-ledger page, FSDP MixedPrecision: the reduction is
 * done in fp32 because summing in bf16 loses accuracy).  An all-to-all
 * exchange of the ranks' flat low-precision grads (padded to world_size
 * equal chunks) has placed, for this rank's shard, n_chunks blocks in
 * d_chunks, block r holding rank r's values; block r starts at element
 * r * chunk_stride.  For k in [0, n), in rank order r = 0 .. n_chunks-1:
 *   d_acc[k] = fl(d_acc[k] + fl(scale * x_r[k]))
 * where, for r == 0 and accumulate == 0, d_acc[k] = fl(scale * x_0[k])
 * instead (the accumulator's old contents are not read).  x_r is block r in
 * src_dtype cast exactly to fp32.  This is the rule of n_chunks successive
 * zero_accum calls, in one pass.  scale = 1 / world_size (times
 * 1 / accum_steps when each micro-batch is reduced and accumulated): for a
 * power-of-two world size scaling each term first is exactly the page's
 * sum-then-divide, summed in rank order in binary32.  Elements n ..
 * chunk_stride-1 of every block (the padding of a short last shard) are
 * never read.  d_scale, d_found_nonfinite and d_norm_ws (zero_grad_sqnorm_
 * workspace_bytes(n)) as for zero_flatten_cast: the norm partials are those
 * of the final d_acc values.
 * Layout: d_acc fp32 [n]; d_chunks [n_chunks][chunk_stride] of src_dtype.
 * Fast path: d_acc 32-byte aligned, d_chunks and chunk_stride * element
 * size 16-byte (16-bit) or 32-byte (fp32) aligned; otherwise a slower,
 * equally exact element path.
 * Errors: ZERO_EINVAL for n < 0, n_chunks < 1, chunk_stride < n, NULL
 * buffers with n > 0, a bad dtype, accumulate not 0/1, a non-finite scale,
 * a chunk array larger than 2^62 bytes, or a too-small / misaligned norm
 * workspace. */
zero_status zero_reduce_chunks(float* d_acc, const void* d_chunks, zero_dtype src_dtype, int32_t n_chunks,
                               int64_t chunk_stride, int64_t n, float scale, const float* d_scale,
                               int32_t accumulate, int32_t* d_found_nonfinite, void* d_norm_ws,
                               size_t norm_ws_bytes, void* stream);

/* zero_grad_sqnorm_workspace_bytes -- host only.
 * Device scratch that zero_grad_sqnorm needs for n elements: one binary64
 * partial per fixed tile of the grad buffer (8 bytes per 32768 elements).
 * Returns 0 for n <= 0. */
size_t zero_grad_sqnorm_workspace_bytes(int64_t n);

/* zero_grad_sqnorm -- device.
 * clip_grad_norm_(params, max_norm) as the ZeRO page's training loop
 * (section "组合策略") and the gradient-accumulation page call it after
 * accumulation and before the step, made deterministic:
 *   sqnorm = sum_k d_grad[k]^2 + extra_sqnorm
 *   norm   = sqrt(sqnorm)                                     (binary64)
 *   clip_coef = max_norm / (norm + 1e-6) if that is < 1, else 1 (binary32)
 *   finite = isfinite(norm)   -- the page skips the step when it is not
 * The squares are summed in fixed tiles of 32768 elements (exact squares
 * added into double-float binary32 pairs within a tile, binary64 across
 * tiles, relative error ~1e-14), so the result does not depend
 * on the GPU or the launch size and matches a binary64 sum to ~14 digits.
 * Squares beyond the binary32 range (|g| >= 2^64) give a non-finite norm.
 * extra_sqnorm is the other ranks' share of a global norm (0 for a norm over
 * this buffer alone).  max_norm = +inf turns clipping off (coefficient 1).
 * d_ws: device scratch of at least zero_grad_sqnorm_workspace_bytes(n)
 *   bytes, 8-byte aligned; overwritten.
 * d_out: device zero_norm_result, written by the call.
 * Errors: ZERO_EINVAL for n < 0, d_grad NULL with n > 0, d_out NULL, d_ws
 * NULL or smaller than required, a negative or NaN max_norm, or a
 * negative or non-finite extra_sqnorm. */
zero_status zero_grad_sqnorm(const float* d_grad, int64_t n, double extra_sqnorm, double max_norm,
                             void* d_ws, size_t ws_bytes, zero_norm_result* d_out, void* stream);

/* zero_grad_sqnorm_finalize -- device.
 * The second half of zero_grad_sqnorm: from the per-tile partials that a
 * zero_flatten_cast / zero_accum call with a norm workspace wrote for an
 * n-element grad buffer, add them in the fixed order, add extra_sqnorm and
 * write the zero_norm_result (norm, clip coefficient, finite flag) exactly
 * as zero_grad_sqnorm would for that buffer.  This fuses the grad-norm read
 * into the last micro-batch's pass (4 bytes per parameter saved).
 * Errors: ZERO_EINVAL for n < 0, d_out NULL, d_ws NULL or misaligned with
 * n > 0, a negative or NaN max_norm, or a negative or non-finite
 * extra_sqnorm. */
zero_status zero_grad_sqnorm_finalize(const void* d_ws, int64_t n, double extra_sqnorm, double max_norm,
                                      zero_norm_result* d_out, void* stream);

/* zero_grad_sqnorm_combine -- device.
 * The global norm of clip_grad_norm_ across data-parallel ranks (ZeRO-2/3:
 * each rank holds only its shard's grads).  d_sqnorms[r] is rank r's local
 * sum of squares (the `sqnorm` field of its zero_grad_sqnorm /
 * zero_grad_sqnorm_finalize result with extra_sqnorm = 0), gathered in rank
 * order -- the one exchange of the step, 8 bytes per rank.  The values are
 * added in index order in binary64, so every rank that combines the same
 * gathered vector gets the same norm and the same binary32 coefficient
 * (a tree all-reduce would not promise that).  Writes d_out like
 * zero_grad_sqnorm.
 * Errors: ZERO_EINVAL for n_parts < 1, NULL or misaligned pointers, or a
 * negative or NaN max_norm. */
zero_status zero_grad_sqnorm_combine(const double* d_sqnorms, int32_t n_parts, double max_norm,
                                     zero_norm_result* d_out, void* stream);

/* zero_adamw_step -- device.
 * The ZeRO page's ZeRO1Optimizer.step Adam update (bias_correction1/2 with
 * the step counter incremented before use; denom = sqrt(exp_avg_sq) /
 * sqrt(bias_correction2) + eps; update = exp_avg / denom * (-lr /
 * bias_correction1)), with AdamW's decoupled weight decay (the memory-ledger
 * page names "bf16 + AdamW" as the default) applied to the old master value,
 * the clip coefficient of zero_grad_sqnorm applied to the grad, and the
 * low-precision parameter copy written in the same pass (memory-ledger page:
 * 16 bytes/param = bf16 param + bf16 grad + 12 bytes fp32 state).  Per
 * element, each operation rounded to nearest even in binary32:
 *   g = grad * coef
 *   p = p * (1 - lr*wd)
 *   m = fma(1-beta1, g, m*beta1)
 *   v = fma((1-beta2)*g, g, v*beta2)
 *   d = sqrt(v) / sqrt(1-beta2^t) + eps
 *   p = p - (lr / (1-beta1^t)) * (m / d)
 *   lowp = round_to_nearest_even(p)
 * where the per-step scalars are computed in binary64 on the host and
 * rounded to binary32 once (zero_adamw_scalars).  d_master, d_exp_avg, d_exp_avg_sq (fp32, n,
 * updated in place), d_grad (fp32, n).  d_param_lowp: NULL or n elements of
 * lowp_dtype (BF16, or F16 for the ZeRO-3 page's fp16 local chunk); the
 * rank's slice of the full low-precision FlatParameter may start at any
 * element.  step: t >= 1, already incremented (the page's step_count).
 * d_clip: NULL (coefficient 1, no skip guard), or the device result of
 * zero_grad_sqnorm; when its `finite` is 0 the call changes nothing (the
 * device-side half of the page's skip-on-overflow policy; the caller should
 * then not advance t).
 * Errors: ZERO_EINVAL for n < 0, NULL state/grad buffers with n > 0, hp
 * NULL, step < 1, a bad lowp_dtype (F32 is not a low-precision copy), or
 * hyper-parameters outside lr >= 0, 0 <= beta < 1, eps > 0, wd >= 0 (all
 * finite). */
zero_status zero_adamw_step(float* d_master, float* d_exp_avg, float* d_exp_avg_sq,
                            const float* d_grad, void* d_param_lowp, zero_dtype lowp_dtype,
                            int64_t n, const zero_adamw_hparams* hp, int64_t step,
                            const zero_norm_result* d_clip, void* stream);

/* zero_grad_sqnorm_noalloc -- device.  No counterpart on the source pages:
 * a convenience of this library.
 * Computes exactly what zero_grad_sqnorm computes, for callers that cannot
 * allocate device memory for its workspace: code that runs inside another
 * framework's memory pool which owns all device memory, inside an allocator
 * hook, or in a loop that must not pay the implicit device synchronisation
 * that cudaMalloc/cudaFree can cause.  Instead of a caller workspace the
 * tile partials go to a fixed array inside the library: 4 MiB of device
 * memory on every GPU that loads the library, held until the process exits.
 * The caller still passes d_grad and d_out; the call itself allocates
 * nothing (no cudaMalloc, cudaFree or allocating library routine).
 * Limit: n <= 2^19 tiles * 32768 = 17,179,869,184 elements; a larger n
 * returns ZERO_EINVAL with a message that names the limit.
 * Set-up: the first call on each device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current; make that first
 * call before any stream capture begins.  The address is kept per device and
 * context (keyed on the context's process-unique ID): after cudaDeviceReset
 * the runtime's new context may hold the array elsewhere, so the first call
 * in it looks the address up again (and should also come before a capture).
 * Sharing: all calls on a device use the same array, which keeps the last
 * call's partials.  Calls whose work overlaps on the GPU (for example on two
 * streams at once) race on it; the caller must serialise them.  Nothing
 * needs clearing between calls: each call writes every partial it reads.
 * Errors: those of zero_grad_sqnorm without the workspace checks, the limit
 * above, and ZERO_ECUDA if the address lookup fails. */
zero_status zero_grad_sqnorm_noalloc(const float* d_grad, int64_t n, double extra_sqnorm,
                                     double max_norm, zero_norm_result* d_out, void* stream);

/* zero_loss_scale_update -- host only.
 * Dynamic loss scaling of mixed-precision training, as the ZeRO page's
 * Llama-7B recipe (section "组合策略：ZeRO-3 + 梯度累积 + 混合精度") configures
 * torch.cuda.amp.GradScaler(init_scale=2^16, growth_factor=2.0,
 * backoff_factor=0.5, growth_interval=2000) and skips the step on overflow.
 * After a step whose grads overflowed (found_inf != 0, e.g. the
 * d_found_nonfinite flag of zero_flatten_cast / zero_accum):
 * *scale *= backoff_factor and the count of good steps restarts at 0.
 * Otherwise the count grows; when it reaches growth_interval the scale is
 * multiplied by growth_factor (kept only if still finite) and the count
 * restarts.  Products are taken in binary64 and rounded to binary32.
 * The unscale itself is folded into the flatten / accumulate `scale`
 * argument: scale = 1 / (loss_scale * accum_steps), exact for the
 * power-of-two values used in practice.
 * Errors: ZERO_EINVAL for NULL pointers, growth_factor <= 1 or not finite,
 * backoff_factor outside (0, 1), growth_interval < 1. */
zero_status zero_loss_scale_update(float* scale, int32_t* growth_tracker, int32_t found_inf,
                                   double growth_factor, double backoff_factor,
                                   int32_t growth_interval);

/* The dynamic loss scale kept in device memory (zero_loss_scale_update_device),
 * for mixed-precision steps captured in a CUDA graph. */
typedef struct zero_loss_scale_state {
  float scale;             /* the loss scale S the next backward multiplies the loss by */
  int32_t growth_tracker;  /* good steps since the scale last changed */
  float unscale;           /* 1 / (S * accum_steps): the d_scale of the next step's grad passes */
  int32_t found_inf;       /* the grad passes' d_found_nonfinite; cleared by the update */
} zero_loss_scale_state;

/* zero_loss_scale_update_device -- device (one thread).
 * zero_loss_scale_update on a zero_loss_scale_state in device memory, read
 * and written when the kernel runs: the step overflowed when found_inf is
 * set, or when d_norm is given and its `finite` is 0 (a sum of squares that
 * overflowed).  The same binary64 products rounded to binary32 as the host
 * update, so host and device scales agree bit for bit.  Then unscale =
 * 1 / (scale * accum_steps) in binary64 rounded to binary32 (the value the
 * host path passes as `scale`) and found_inf = 0, ready for the next step.
 * The caller fills the initial state (scale, growth_tracker 0, its unscale,
 * found_inf 0).
 * Errors: ZERO_EINVAL for a NULL state, accum_steps < 1, or factors and
 * interval outside the ranges of zero_loss_scale_update. */
zero_status zero_loss_scale_update_device(zero_loss_scale_state* d_state, int32_t accum_steps,
                                          double growth_factor, double backoff_factor,
                                          int32_t growth_interval, const zero_norm_result* d_norm,
                                          void* stream);

/* zero_adamw_step_tensors -- device.
 * zero_adamw_step with the grad read straight from the per-tensor grads
 * through the FlatParameter table instead of from a materialized fp32 flat
 * grad: for k in [0, n) the grad is fl(grad_scale * x) where x is the grad
 * element at flat index shard_start + k (0 for a tensor without grad), cast
 * exactly to binary32 -- the value zero_flatten_cast(..., scale =
 * grad_scale, accumulate = 0) would have written -- and the update is then
 * the same operation sequence, so the result is bit-identical to flatten +
 * zero_adamw_step.  For a step without micro-batch accumulation this is the
 * whole flatten/cast row fused away: the step reads the bf16 grads twice
 * (norm pass with d_dst = NULL, then this) and never writes the 4-byte fp32
 * grad, 30 instead of 36 bytes per parameter, and the fp32 grad buffer
 * (4 bytes/param of HBM) is not needed at all.
 * d_grad_scale: NULL, or a device float read when the kernel runs and used
 *   in place of grad_scale (the unscale factor of a loss scale kept on the
 *   device, as d_scale of zero_flatten_cast; grad_scale must still be finite).
 * d_acc: NULL, or the fp32 sum of the step's earlier micro-batches (n
 *   elements, element k at flat index shard_start + k, as zero_flatten_cast
 *   or zero_accum left it): the grad is then fl(d_acc[k] + fl(grad_scale *
 *   x)), the value the last micro-batch's zero_flatten_cast(..., accumulate
 *   = 1) would have stored.  With the norm pass zero_flatten_cast(...,
 *   accumulate = 2), the last micro-batch is never written: 6 + 32 instead
 *   of 10 + 30 bytes per parameter for 16-bit grads.  Only read; it must not
 *   overlap the state.  Fast path: 32-byte aligned, like the state.
 * d_table / n_tensors / total / grad_dtype as for zero_flatten_cast; the
 * other arguments as for zero_adamw_step.
 * Errors: those of zero_adamw_step, plus a bad table, [shard_start,
 * shard_start + n) outside [0, total], a bad grad_dtype or a non-finite
 * grad_scale. */
zero_status zero_adamw_step_tensors(float* d_master, float* d_exp_avg, float* d_exp_avg_sq,
                                    const zero_tensor* d_table, int32_t n_tensors, int64_t total,
                                    zero_dtype grad_dtype, int64_t shard_start, float grad_scale,
                                    const float* d_grad_scale, const float* d_acc, void* d_param_lowp,
                                    zero_dtype lowp_dtype, int64_t n,
                                    const zero_adamw_hparams* hp, int64_t step,
                                    const zero_norm_result* d_clip, void* stream);

/* ---------------------------------------------------------------------
 * Graph-capturable steps.  No counterpart on the source pages: the pages'
 * loops keep the step count on the host and read the grad norm there to
 * decide on skipping.  These calls keep both on the device, so one whole
 * step (flatten / accumulate with the fused norm, finalize, prepare, AdamW)
 * can be captured once in a CUDA graph and replayed with no host work and
 * no device-to-host read per step.  The results are bit-identical to the
 * host-counter calls above.
 * --------------------------------------------------------------------- */

/* Device-resident step state of one optimizer (48 bytes, 8-byte aligned,
 * in device memory).  Zero it before the first step; `step` may be set to
 * resume from a checkpoint. */
typedef struct zero_adamw_device_state {
  int64_t step;     /* t: steps applied so far */
  int32_t apply;    /* written by zero_adamw_prepare_device: 1 = the prepared step
                       runs, 0 = it is skipped (non-finite norm or bad hparams) */
  int32_t status;   /* ZERO_OK, or ZERO_EINVAL when the hyper-parameters read on
                       the device were outside the ranges zero_adamw_step accepts */
  float scalars[8]; /* step_size, sqrt(1-beta2^t), 1-lr*wd, beta1, 1-beta1, beta2,
                       1-beta2, eps of the prepared step, each rounded once */
} zero_adamw_device_state;

/* zero_adamw_scalars -- host only.
 * The per-step scalars zero_adamw_step uses for step t (>= 1), in the order
 * of zero_adamw_device_state.scalars: bias corrections 1 - beta^t with
 * beta^t by binary powering in double-double (the correctly rounded power
 * but for near-ties), then lr / (1-beta1^t), sqrt(1-beta2^t), 1 - lr*wd in
 * binary64, each rounded to binary32 once.  out: 8 floats, host memory.
 * Errors: ZERO_EINVAL for NULL hp/out, step < 1, or hyper-parameters
 * outside the ranges of zero_adamw_step. */
zero_status zero_adamw_scalars(const zero_adamw_hparams* hp, int64_t step, float* out);

/* zero_adamw_prepare_device -- device (one thread).
 * The device half of the pages' skip policy and step counter: if d_clip is
 * NULL or its `finite` is 1, and the hyper-parameters at d_hp (device
 * memory, read when the kernel runs, so a schedule may rewrite them between
 * replays) are valid, then step += 1, the scalars of that step are stored
 * (the same bits zero_adamw_scalars gives) and apply = 1; otherwise apply =
 * 0 and step is unchanged (status = ZERO_EINVAL for bad hyper-parameters).
 * Errors (host): ZERO_EINVAL for NULL d_hp or d_state or a d_state that is
 * not 8-byte aligned; ZERO_ECUDA for a failed launch. */
zero_status zero_adamw_prepare_device(const zero_adamw_hparams* d_hp, const zero_norm_result* d_clip,
                                      zero_adamw_device_state* d_state, void* stream);

/* zero_adamw_step_device -- device.
 * zero_adamw_step with the scalars and the skip decision taken from
 * d_state, as the last zero_adamw_prepare_device on the stream left them:
 * nothing changes when apply is 0.  d_clip supplies the clip coefficient as
 * for zero_adamw_step (NULL: 1).
 * Errors: those of zero_adamw_step without the hyper-parameter checks, plus
 * NULL or misaligned d_state. */
zero_status zero_adamw_step_device(float* d_master, float* d_exp_avg, float* d_exp_avg_sq,
                                   const float* d_grad, void* d_param_lowp, zero_dtype lowp_dtype,
                                   int64_t n, const zero_adamw_device_state* d_state,
                                   const zero_norm_result* d_clip, void* stream);

/* zero_adamw_step_tensors_device -- device.
 * zero_adamw_step_tensors with the scalars and the skip decision from
 * d_state, as zero_adamw_step_device. */
zero_status zero_adamw_step_tensors_device(float* d_master, float* d_exp_avg, float* d_exp_avg_sq,
                                           const zero_tensor* d_table, int32_t n_tensors, int64_t total,
                                           zero_dtype grad_dtype, int64_t shard_start, float grad_scale,
                                           const float* d_grad_scale, const float* d_acc, void* d_param_lowp,
                                           zero_dtype lowp_dtype, int64_t n,
                                           const zero_adamw_device_state* d_state,
                                           const zero_norm_result* d_clip, void* stream);

/* ---------------------------------------------------------------------
 * Debug builds.  No counterpart on the source pages.  Built with
 * -DZERO_DEBUG (libzeroshard_debug.so), every kernel checks each global-
 * memory access site's index against the extent it must stay in and its
 * address against the alignment of its vector width before the access; a
 * violation is counted, the first one recorded, and the access skipped
 * (reported instead of faulting).  Release builds compile the checks away
 * and these two calls return ZERO_EINVAL.
 * --------------------------------------------------------------------- */

/* zero_debug_errors -- host (synchronises the device).
 * out[0] = violations since the last reset, out[1..3] = site, index and
 * block of the first one (0 when none); reset != 0 clears the record. */
zero_status zero_debug_errors(uint64_t* out, int32_t reset);

/* zero_debug_selftest -- device.
 * Records one violation at site 999 with the given index, touching no
 * memory: checks the reporting path of a debug build. */
zero_status zero_debug_selftest(int64_t index, void* stream);

/* Static text for a status code. */
const char* zero_status_string(zero_status status);

/* Message of the calling thread's last failed call ("" if none). */
const char* zero_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ZERO_SHARD_H_ */
