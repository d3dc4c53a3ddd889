// kernels.h -- launchers of the device kernels, called by the C-ABI entry
// points in api.cu after argument checking.  Internal; not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "zero_shard.h"

namespace zs {

// Per-step AdamW scalars, computed in binary64 and rounded to binary32 once
// (bias corrections of the ZeRO page's ZeRO1Optimizer.step; adam_scalars.cuh).
struct AdamScalars {
  float step_size;  // lr / (1 - beta1^t)
  float bc2_sqrt;   // sqrt(1 - beta2^t)
  float decay;      // 1 - lr * weight_decay
  float b1, omb1;   // beta1, 1 - beta1
  float b2, omb2;   // beta2, 1 - beta2
  float eps;
};

// Elements per binary64 partial of the grad-norm reduction.
constexpr int64_t kSqTile = 32768;

// `ds` (nullable): take the scalars and the skip decision from the device
// step state instead of `s` (graph-capturable steps).
zero_status launch_adamw(float* p, float* m, float* v, const float* g, void* lowp, int lowp_dtype, int64_t n,
                         const AdamScalars& s, const zero_adamw_device_state* ds, const zero_norm_result* clip,
                         cudaStream_t st);

// AdamW with the grad read through the tensor table (grad_scale * x at flat
// index shard_start + k) instead of a materialized fp32 grad; `acc`
// (nullable): the earlier micro-batches' fp32 sum, added first.
// `dscale` (nullable): read the grad scale from device memory when the kernel runs.
zero_status launch_adamw_table(float* p, float* m, float* v, const float* acc, const zero_tensor* table,
                               int n_tensors, int grad_dtype, int64_t shard_start, float gscale, const float* dscale,
                               void* lowp, int lowp_dtype, int64_t n, const AdamScalars& s,
                               const zero_adamw_device_state* ds, const zero_norm_result* clip, cudaStream_t st);
// Its other instances, each in a translation unit of its own (compiled in
// parallel): acc != NULL; one table search per four parts (long tables); both.
using AdamwTableInstance = zero_status(float* p, float* m, float* v, const float* acc, const zero_tensor* table,
                                       int n_tensors, int grad_dtype, int64_t shard_start, float gscale,
                                       const float* dscale, void* lowp, int lowp_dtype, int64_t n,
                                       const AdamScalars& s, const zero_adamw_device_state* ds,
                                       const zero_norm_result* clip, cudaStream_t st);
AdamwTableInstance launch_adamw_table_acc;
AdamwTableInstance launch_adamw_table_p4;
AdamwTableInstance launch_adamw_table_p4_acc;

// Debug builds (ZERO_DEBUG): each translation unit's violation record
// {count, first site, first index, first block}; reset clears it.
zero_status debug_read_adamw(unsigned long long* out, bool reset);
zero_status debug_read_adamw_table(unsigned long long* out, bool reset);
zero_status debug_read_adamw_table_acc(unsigned long long* out, bool reset);
zero_status debug_read_adamw_table_p4(unsigned long long* out, bool reset);
zero_status debug_read_adamw_table_p4_acc(unsigned long long* out, bool reset);
zero_status debug_read_adamw_device(unsigned long long* out, bool reset);
zero_status debug_read_flatten(unsigned long long* out, bool reset);
zero_status debug_read_sqnorm(unsigned long long* out, bool reset);
zero_status launch_debug_selftest(long long index, cudaStream_t st);

// One thread: the dynamic loss scale update on the device state.
zero_status launch_loss_scale_update(zero_loss_scale_state* state, int32_t accum_steps, double growth,
                                     double backoff, int32_t interval, const zero_norm_result* norm,
                                     cudaStream_t st);

// One thread: advance the device step state (see zero_adamw_prepare_device).
zero_status launch_adamw_prepare(const zero_adamw_hparams* hp, const zero_norm_result* clip,
                                 zero_adamw_device_state* state, cudaStream_t st);

// `partials` (nullable): also write the norm tiles' partial sums of squares
// of the values written (one binary64 per 32768 elements of dst / acc).
// launch_flatten's accumulate == 2: the values fl(dst + fl(scale * x)) are
// formed and their partials written, but dst is only read (partials required).
// `dscale` (nullable): read the scale from device memory when the kernel runs.
zero_status launch_flatten(const zero_tensor* table, int32_t n_tensors, int src_dtype, int64_t shard_start,
                           int64_t shard_end, float scale, const float* dscale, int accumulate, float* dst,
                           int32_t* flag, double* partials, cudaStream_t st);

zero_status launch_accum(float* acc, const void* src, int src_dtype, int64_t n, float scale, const float* dscale,
                         int accumulate, int32_t* flag, double* partials, cudaStream_t st);

// The ranks' received blocks of this rank's shard (n_chunks blocks, `stride`
// elements apart) added into acc in rank order, each scaled first.
zero_status launch_reduce_chunks(float* acc, const void* src, int src_dtype, int n_chunks, int64_t stride, int64_t n,
                                 float scale, const float* dscale, int accumulate, int32_t* flag, double* partials,
                                 cudaStream_t st);

zero_status launch_sqnorm(const float* g, int64_t n, double extra_sqnorm, double max_norm, double* partials,
                          zero_norm_result* out, cudaStream_t st);

// Norm result from already computed tile partials (ceil(n / kSqTile) of them).
zero_status launch_sqnorm_finalize(const double* partials, int64_t n, double extra_sqnorm, double max_norm,
                                   zero_norm_result* out, cudaStream_t st);

// Global norm from a device vector of per-rank sums of squares (rank order).
zero_status launch_sqnorm_combine(const double* sq, int n_parts, double max_norm, zero_norm_result* out,
                                  cudaStream_t st);

}  // namespace zs
