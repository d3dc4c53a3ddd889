// api.cu -- the C-ABI entry points of libzeroshard (declared in
// include/zero_shard.h): argument checking, per-step scalars, dispatch to the
// kernel launchers, and the per-thread error message.
#include <cmath>
#include <cstdarg>
#include <cstdio>

#include "adam_scalars.cuh"
#include "common.cuh"
#include "kernels.h"

namespace zs {

static thread_local char g_msg[512] = "";

zero_status fail(zero_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

zero_status check_launch(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(ZERO_ECUDA, "%s: %s", what, cudaGetErrorString(e));
  return ZERO_OK;
}

static bool valid_dtype(int d) { return d == ZERO_F32 || d == ZERO_BF16 || d == ZERO_F16; }

}  // namespace zs

using zs::fail;

extern "C" {

const char* zero_status_string(zero_status s) {
  switch (s) {
    case ZERO_OK: return "ZERO_OK";
    case ZERO_EINVAL: return "ZERO_EINVAL: invalid argument";
    case ZERO_ECUDA: return "ZERO_ECUDA: CUDA runtime error";
  }
  return "unknown zero_status";
}

const char* zero_last_error(void) { return zs::g_msg; }

zero_status zero_shard_range(int64_t total, int32_t world_size, int32_t rank, int64_t* start, int64_t* end) {
  if (start == nullptr || end == nullptr) return fail(ZERO_EINVAL, "zero_shard_range: NULL output");
  if (total < 0) return fail(ZERO_EINVAL, "zero_shard_range: total %lld < 0", (long long)total);
  if (world_size < 1) return fail(ZERO_EINVAL, "zero_shard_range: world_size %d < 1", world_size);
  if (rank < 0 || rank >= world_size)
    return fail(ZERO_EINVAL, "zero_shard_range: rank %d not in [0, %d)", rank, world_size);
  // chunk = ceil(total / world) without overflow for totals near INT64_MAX
  const int64_t chunk = total / world_size + (total % world_size != 0 ? 1 : 0);
  const int64_t s = (chunk != 0 && rank > (total / chunk)) ? total : static_cast<int64_t>(rank) * chunk;
  const int64_t lo = s < total ? s : total;
  const int64_t hi = (chunk > total - lo) ? total : lo + chunk;
  *start = lo;
  *end = hi;
  return ZERO_OK;
}

zero_status zero_tensor_table(const void* const* ptrs, const int64_t* numels, int32_t n_tensors,
                              zero_tensor* table, int64_t* total) {
  if (n_tensors < 0) return fail(ZERO_EINVAL, "zero_tensor_table: n_tensors %d < 0", n_tensors);
  if (total == nullptr) return fail(ZERO_EINVAL, "zero_tensor_table: NULL total");
  if (n_tensors > 0 && (numels == nullptr || table == nullptr))
    return fail(ZERO_EINVAL, "zero_tensor_table: NULL numels or table");
  int64_t acc = 0;
  for (int32_t i = 0; i < n_tensors; ++i) {
    if (numels[i] < 0) return fail(ZERO_EINVAL, "zero_tensor_table: numel[%d] = %lld < 0", i, (long long)numels[i]);
    if (numels[i] > INT64_MAX - acc) return fail(ZERO_EINVAL, "zero_tensor_table: total overflows int64");
    acc += numels[i];
  }
  int64_t off = 0;
  for (int32_t i = 0; i < n_tensors; ++i) {
    table[i].ptr = ptrs ? ptrs[i] : nullptr;
    table[i].numel = numels[i];
    table[i].flat_offset = off;
    off += numels[i];
  }
  *total = acc;
  return ZERO_OK;
}

// Optional fused-norm workspace of the flatten / accumulate calls: NULL, or
// room for one binary64 partial per 32768 output elements, 8-byte aligned.
static zero_status check_norm_ws(const char* who, const void* ws, size_t ws_bytes, int64_t n) {
  if (ws == nullptr) return ZERO_OK;
  const size_t need = zero_grad_sqnorm_workspace_bytes(n);
  if (ws_bytes < need) return fail(ZERO_EINVAL, "%s: norm workspace %zu bytes < %zu needed", who, ws_bytes, need);
  if (!zs::aligned(ws, 8)) return fail(ZERO_EINVAL, "%s: norm workspace not 8-byte aligned", who);
  return ZERO_OK;
}

zero_status zero_flatten_cast(const zero_tensor* d_table, int32_t n_tensors, int64_t total, zero_dtype src_dtype,
                              int64_t shard_start, int64_t shard_end, float scale, const float* d_scale,
                              int32_t accumulate, float* d_dst, int32_t* d_found_nonfinite, void* d_norm_ws,
                              size_t norm_ws_bytes, void* stream) {
  if (n_tensors < 0) return fail(ZERO_EINVAL, "zero_flatten_cast: n_tensors %d < 0", n_tensors);
  if (n_tensors > 0 && d_table == nullptr) return fail(ZERO_EINVAL, "zero_flatten_cast: NULL d_table");
  if (total < 0 || (n_tensors == 0 && total != 0))
    return fail(ZERO_EINVAL, "zero_flatten_cast: total %lld does not fit %d tensors", (long long)total, n_tensors);
  if (shard_start < 0 || shard_start > shard_end || shard_end > total)
    return fail(ZERO_EINVAL, "zero_flatten_cast: shard [%lld, %lld) outside [0, %lld]", (long long)shard_start,
                (long long)shard_end, (long long)total);
  if (!zs::valid_dtype(src_dtype)) return fail(ZERO_EINVAL, "zero_flatten_cast: bad src_dtype %d", (int)src_dtype);
  if (accumulate < 0 || accumulate > 2) return fail(ZERO_EINVAL, "zero_flatten_cast: accumulate must be 0, 1 or 2");
  if (!std::isfinite(scale)) return fail(ZERO_EINVAL, "zero_flatten_cast: non-finite scale");
  if (shard_end > shard_start && d_dst == nullptr && (d_norm_ws == nullptr || accumulate != 0))
    return fail(ZERO_EINVAL, "zero_flatten_cast: NULL d_dst needs a norm workspace and accumulate == 0");
  if (accumulate == 2 && shard_end > shard_start && d_norm_ws == nullptr)
    return fail(ZERO_EINVAL, "zero_flatten_cast: accumulate == 2 (norm of the sum only) needs a norm workspace");
  const zero_status w = check_norm_ws("zero_flatten_cast", d_norm_ws, norm_ws_bytes, shard_end - shard_start);
  if (w != ZERO_OK) return w;
  if (shard_end == shard_start) return ZERO_OK;
  return zs::launch_flatten(d_table, n_tensors, src_dtype, shard_start, shard_end, scale, d_scale, accumulate,
                            d_dst, d_found_nonfinite, static_cast<double*>(d_norm_ws), zs::as_stream(stream));
}

zero_status zero_accum(float* d_acc, const void* d_src, zero_dtype src_dtype, int64_t n, float scale,
                       const float* d_scale, int32_t accumulate, int32_t* d_found_nonfinite, void* d_norm_ws,
                       size_t norm_ws_bytes, void* stream) {
  if (n < 0) return fail(ZERO_EINVAL, "zero_accum: n %lld < 0", (long long)n);
  if (!zs::valid_dtype(src_dtype)) return fail(ZERO_EINVAL, "zero_accum: bad src_dtype %d", (int)src_dtype);
  if (accumulate != 0 && accumulate != 1) return fail(ZERO_EINVAL, "zero_accum: accumulate must be 0 or 1");
  if (!std::isfinite(scale)) return fail(ZERO_EINVAL, "zero_accum: non-finite scale");
  if (n > 0 && (d_acc == nullptr || d_src == nullptr)) return fail(ZERO_EINVAL, "zero_accum: NULL buffer");
  const zero_status w = check_norm_ws("zero_accum", d_norm_ws, norm_ws_bytes, n);
  if (w != ZERO_OK) return w;
  if (n == 0) return ZERO_OK;
  return zs::launch_accum(d_acc, d_src, src_dtype, n, scale, d_scale, accumulate, d_found_nonfinite,
                          static_cast<double*>(d_norm_ws), zs::as_stream(stream));
}

zero_status zero_reduce_chunks(float* d_acc, const void* d_chunks, zero_dtype src_dtype, int32_t n_chunks,
                               int64_t chunk_stride, int64_t n, float scale, const float* d_scale,
                               int32_t accumulate, int32_t* d_found_nonfinite, void* d_norm_ws,
                               size_t norm_ws_bytes, void* stream) {
  if (n < 0) return fail(ZERO_EINVAL, "zero_reduce_chunks: n %lld < 0", (long long)n);
  if (n_chunks < 1) return fail(ZERO_EINVAL, "zero_reduce_chunks: n_chunks %d < 1", (int)n_chunks);
  if (chunk_stride < n)
    return fail(ZERO_EINVAL, "zero_reduce_chunks: chunk_stride %lld < n %lld", (long long)chunk_stride,
                (long long)n);
  if (!zs::valid_dtype(src_dtype)) return fail(ZERO_EINVAL, "zero_reduce_chunks: bad src_dtype %d", (int)src_dtype);
  if (accumulate != 0 && accumulate != 1) return fail(ZERO_EINVAL, "zero_reduce_chunks: accumulate must be 0 or 1");
  if (!std::isfinite(scale)) return fail(ZERO_EINVAL, "zero_reduce_chunks: non-finite scale");
  if (n > 0 && (d_acc == nullptr || d_chunks == nullptr)) return fail(ZERO_EINVAL, "zero_reduce_chunks: NULL buffer");
  const int64_t es = (src_dtype == ZERO_F32) ? 4 : 2;
  if (chunk_stride > (int64_t(1) << 62) / es / n_chunks)
    return fail(ZERO_EINVAL, "zero_reduce_chunks: %d chunks of %lld elements exceed 2^62 bytes", (int)n_chunks,
                (long long)chunk_stride);
  const zero_status w = check_norm_ws("zero_reduce_chunks", d_norm_ws, norm_ws_bytes, n);
  if (w != ZERO_OK) return w;
  if (n == 0) return ZERO_OK;
  return zs::launch_reduce_chunks(d_acc, d_chunks, src_dtype, n_chunks, chunk_stride, n, scale, d_scale,
                                  accumulate, d_found_nonfinite, static_cast<double*>(d_norm_ws),
                                  zs::as_stream(stream));
}

size_t zero_grad_sqnorm_workspace_bytes(int64_t n) {
  if (n <= 0) return 0;
  return static_cast<size_t>((n + zs::kSqTile - 1) / zs::kSqTile) * sizeof(double);
}

zero_status zero_grad_sqnorm(const float* d_grad, int64_t n, double extra_sqnorm, double max_norm, void* d_ws,
                             size_t ws_bytes, zero_norm_result* d_out, void* stream) {
  if (n < 0) return fail(ZERO_EINVAL, "zero_grad_sqnorm: n %lld < 0", (long long)n);
  if (n > 0 && d_grad == nullptr) return fail(ZERO_EINVAL, "zero_grad_sqnorm: NULL d_grad");
  if (d_out == nullptr) return fail(ZERO_EINVAL, "zero_grad_sqnorm: NULL d_out");
  if (std::isnan(max_norm) || max_norm < 0.0) return fail(ZERO_EINVAL, "zero_grad_sqnorm: bad max_norm");
  if (!std::isfinite(extra_sqnorm) || extra_sqnorm < 0.0)
    return fail(ZERO_EINVAL, "zero_grad_sqnorm: bad extra_sqnorm");
  const size_t need = zero_grad_sqnorm_workspace_bytes(n);
  if (need > 0 && (d_ws == nullptr || ws_bytes < need))
    return fail(ZERO_EINVAL, "zero_grad_sqnorm: workspace %zu bytes < %zu needed", d_ws ? ws_bytes : 0, need);
  if (need > 0 && !zs::aligned(d_ws, 8)) return fail(ZERO_EINVAL, "zero_grad_sqnorm: workspace not 8-byte aligned");
  return zs::launch_sqnorm(d_grad, n, extra_sqnorm, max_norm, static_cast<double*>(d_ws), d_out,
                           zs::as_stream(stream));
}

zero_status zero_grad_sqnorm_finalize(const void* d_ws, int64_t n, double extra_sqnorm, double max_norm,
                                      zero_norm_result* d_out, void* stream) {
  if (n < 0) return fail(ZERO_EINVAL, "zero_grad_sqnorm_finalize: n %lld < 0", (long long)n);
  if (d_out == nullptr) return fail(ZERO_EINVAL, "zero_grad_sqnorm_finalize: NULL d_out");
  if (n > 0 && d_ws == nullptr) return fail(ZERO_EINVAL, "zero_grad_sqnorm_finalize: NULL d_ws");
  if (n > 0 && !zs::aligned(d_ws, 8)) return fail(ZERO_EINVAL, "zero_grad_sqnorm_finalize: d_ws not 8-byte aligned");
  if (std::isnan(max_norm) || max_norm < 0.0) return fail(ZERO_EINVAL, "zero_grad_sqnorm_finalize: bad max_norm");
  if (!std::isfinite(extra_sqnorm) || extra_sqnorm < 0.0)
    return fail(ZERO_EINVAL, "zero_grad_sqnorm_finalize: bad extra_sqnorm");
  return zs::launch_sqnorm_finalize(static_cast<const double*>(d_ws), n, extra_sqnorm, max_norm, d_out,
                                    zs::as_stream(stream));
}

zero_status zero_grad_sqnorm_combine(const double* d_sqnorms, int32_t n_parts, double max_norm,
                                    zero_norm_result* d_out, void* stream) {
  if (n_parts < 1) return fail(ZERO_EINVAL, "zero_grad_sqnorm_combine: n_parts %d < 1", n_parts);
  if (d_sqnorms == nullptr || d_out == nullptr) return fail(ZERO_EINVAL, "zero_grad_sqnorm_combine: NULL pointer");
  if (!zs::aligned(d_sqnorms, 8)) return fail(ZERO_EINVAL, "zero_grad_sqnorm_combine: d_sqnorms not 8-byte aligned");
  if (std::isnan(max_norm) || max_norm < 0.0) return fail(ZERO_EINVAL, "zero_grad_sqnorm_combine: bad max_norm");
  return zs::launch_sqnorm_combine(d_sqnorms, n_parts, max_norm, d_out, zs::as_stream(stream));
}

static zero_status check_loss_scale_policy(const char* who, double growth_factor, double backoff_factor,
                                           int32_t growth_interval) {
  if (!(growth_factor > 1.0) || !std::isfinite(growth_factor))
    return fail(ZERO_EINVAL, "%s: growth_factor must be > 1 and finite", who);
  if (!(backoff_factor > 0.0 && backoff_factor < 1.0))
    return fail(ZERO_EINVAL, "%s: backoff_factor must be in (0, 1)", who);
  if (growth_interval < 1) return fail(ZERO_EINVAL, "%s: growth_interval < 1", who);
  return ZERO_OK;
}

zero_status zero_loss_scale_update(float* scale, int32_t* growth_tracker, int32_t found_inf, double growth_factor,
                                   double backoff_factor, int32_t growth_interval) {
  if (scale == nullptr || growth_tracker == nullptr)
    return fail(ZERO_EINVAL, "zero_loss_scale_update: NULL scale or growth_tracker");
  const zero_status c = check_loss_scale_policy("zero_loss_scale_update", growth_factor, backoff_factor,
                                                growth_interval);
  if (c != ZERO_OK) return c;
  if (found_inf) {
    *scale = static_cast<float>(static_cast<double>(*scale) * backoff_factor);
    *growth_tracker = 0;
    return ZERO_OK;
  }
  const int32_t good = *growth_tracker + 1;
  if (good >= growth_interval) {
    const float grown = static_cast<float>(static_cast<double>(*scale) * growth_factor);
    if (std::isfinite(grown)) *scale = grown;
    *growth_tracker = 0;
  } else {
    *growth_tracker = good;
  }
  return ZERO_OK;
}

zero_status zero_loss_scale_update_device(zero_loss_scale_state* d_state, int32_t accum_steps, double growth_factor,
                                          double backoff_factor, int32_t growth_interval,
                                          const zero_norm_result* d_norm, void* stream) {
  if (d_state == nullptr) return fail(ZERO_EINVAL, "zero_loss_scale_update_device: NULL d_state");
  if (accum_steps < 1) return fail(ZERO_EINVAL, "zero_loss_scale_update_device: accum_steps < 1");
  const zero_status c = check_loss_scale_policy("zero_loss_scale_update_device", growth_factor, backoff_factor,
                                                growth_interval);
  if (c != ZERO_OK) return c;
  return zs::launch_loss_scale_update(d_state, accum_steps, growth_factor, backoff_factor, growth_interval, d_norm,
                                      zs::as_stream(stream));
}

static zero_status adamw_scalars(const char* who, const zero_adamw_hparams* hp, int64_t step, zs::AdamScalars* s) {
  if (hp == nullptr) return fail(ZERO_EINVAL, "%s: NULL hparams", who);
  if (step < 1) return fail(ZERO_EINVAL, "%s: step %lld < 1", who, (long long)step);
  const double lr = hp->lr, b1 = hp->beta1, b2 = hp->beta2, eps = hp->eps, wd = hp->weight_decay;
  if (!(std::isfinite(lr) && lr >= 0.0)) return fail(ZERO_EINVAL, "%s: bad lr", who);
  if (!(b1 >= 0.0 && b1 < 1.0 && b2 >= 0.0 && b2 < 1.0)) return fail(ZERO_EINVAL, "%s: bad betas", who);
  if (!(std::isfinite(eps) && eps > 0.0)) return fail(ZERO_EINVAL, "%s: bad eps", who);
  if (!(std::isfinite(wd) && wd >= 0.0)) return fail(ZERO_EINVAL, "%s: bad weight_decay", who);
  // per-step scalars in binary64, each rounded to binary32 once (the device
  // step state of graph-captured steps uses the same code)
  *s = zs::adam_scalars(lr, b1, b2, eps, wd, step);
  return ZERO_OK;
}

zero_status zero_adamw_scalars(const zero_adamw_hparams* hp, int64_t step, float* out) {
  if (out == nullptr) return fail(ZERO_EINVAL, "zero_adamw_scalars: NULL out");
  zs::AdamScalars s;
  const zero_status st = adamw_scalars("zero_adamw_scalars", hp, step, &s);
  if (st != ZERO_OK) return st;
  const float v[8] = {s.step_size, s.bc2_sqrt, s.decay, s.b1, s.omb1, s.b2, s.omb2, s.eps};
  for (int i = 0; i < 8; ++i) out[i] = v[i];
  return ZERO_OK;
}

zero_status zero_adamw_step(float* d_master, float* d_exp_avg, float* d_exp_avg_sq, const float* d_grad,
                            void* d_param_lowp, zero_dtype lowp_dtype, int64_t n, const zero_adamw_hparams* hp,
                            int64_t step, const zero_norm_result* d_clip, void* stream) {
  if (n < 0) return fail(ZERO_EINVAL, "zero_adamw_step: n %lld < 0", (long long)n);
  zs::AdamScalars s;
  const zero_status hs = adamw_scalars("zero_adamw_step", hp, step, &s);
  if (hs != ZERO_OK) return hs;
  if (n > 0 && (d_master == nullptr || d_exp_avg == nullptr || d_exp_avg_sq == nullptr || d_grad == nullptr))
    return fail(ZERO_EINVAL, "zero_adamw_step: NULL state or grad buffer");
  if (d_param_lowp != nullptr && lowp_dtype != ZERO_BF16 && lowp_dtype != ZERO_F16)
    return fail(ZERO_EINVAL, "zero_adamw_step: lowp_dtype must be BF16 or F16");
  if (n == 0) return ZERO_OK;
  return zs::launch_adamw(d_master, d_exp_avg, d_exp_avg_sq, d_grad, d_param_lowp, lowp_dtype, n, s, nullptr,
                          d_clip, zs::as_stream(stream));
}

zero_status zero_adamw_step_tensors(float* d_master, float* d_exp_avg, float* d_exp_avg_sq,
                                    const zero_tensor* d_table, int32_t n_tensors, int64_t total,
                                    zero_dtype grad_dtype, int64_t shard_start, float grad_scale,
                                    const float* d_grad_scale, const float* d_acc, void* d_param_lowp,
                                    zero_dtype lowp_dtype, int64_t n, const zero_adamw_hparams* hp, int64_t step,
                                    const zero_norm_result* d_clip, void* stream) {
  const char* who = "zero_adamw_step_tensors";
  if (n < 0) return fail(ZERO_EINVAL, "%s: n %lld < 0", who, (long long)n);
  zs::AdamScalars s;
  const zero_status hs = adamw_scalars(who, hp, step, &s);
  if (hs != ZERO_OK) return hs;
  if (n_tensors < 0 || (n_tensors > 0 && d_table == nullptr)) return fail(ZERO_EINVAL, "%s: bad table", who);
  if (total < 0 || (n_tensors == 0 && total != 0)) return fail(ZERO_EINVAL, "%s: total does not fit the table", who);
  if (shard_start < 0 || n > total - shard_start)
    return fail(ZERO_EINVAL, "%s: [%lld, %lld) outside [0, %lld]", who, (long long)shard_start,
                (long long)(shard_start + n), (long long)total);
  if (!zs::valid_dtype(grad_dtype)) return fail(ZERO_EINVAL, "%s: bad grad_dtype %d", who, (int)grad_dtype);
  if (!std::isfinite(grad_scale)) return fail(ZERO_EINVAL, "%s: non-finite grad_scale", who);
  if (n > 0 && (d_master == nullptr || d_exp_avg == nullptr || d_exp_avg_sq == nullptr))
    return fail(ZERO_EINVAL, "%s: NULL state buffer", who);
  if (d_param_lowp != nullptr && lowp_dtype != ZERO_BF16 && lowp_dtype != ZERO_F16)
    return fail(ZERO_EINVAL, "%s: lowp_dtype must be BF16 or F16", who);
  if (n == 0) return ZERO_OK;
  return zs::launch_adamw_table(d_master, d_exp_avg, d_exp_avg_sq, d_acc, d_table, n_tensors, grad_dtype,
                                shard_start, grad_scale, d_grad_scale, d_param_lowp, lowp_dtype, n, s, nullptr,
                                d_clip, zs::as_stream(stream));
}

// ------------------------------------------------------------- debug builds
zero_status zero_debug_errors(uint64_t* out, int32_t reset) {
  if (out == nullptr) return fail(ZERO_EINVAL, "zero_debug_errors: NULL out");
#ifdef ZERO_DEBUG
  zero_status (*const readers[])(unsigned long long*, bool) = {
      zs::debug_read_adamw,          zs::debug_read_adamw_table,        zs::debug_read_adamw_table_acc,
      zs::debug_read_adamw_table_p4, zs::debug_read_adamw_table_p4_acc, zs::debug_read_adamw_device,
      zs::debug_read_flatten,        zs::debug_read_sqnorm};
  uint64_t total = 0, first[3] = {0, 0, 0};
  for (auto rd : readers) {
    unsigned long long r[4];
    const zero_status st = rd(r, reset != 0);
    if (st != ZERO_OK) return st;
    if (r[0] != 0 && total == 0) {
      first[0] = r[1];
      first[1] = r[2];
      first[2] = r[3];
    }
    total += r[0];
  }
  out[0] = total;
  out[1] = first[0];
  out[2] = first[1];
  out[3] = first[2];
  return ZERO_OK;
#else
  (void)reset;
  return fail(ZERO_EINVAL, "zero_debug_errors: this library was built without ZERO_DEBUG");
#endif
}

zero_status zero_debug_selftest(int64_t index, void* stream) {
#ifdef ZERO_DEBUG
  return zs::launch_debug_selftest(index, zs::as_stream(stream));
#else
  (void)index;
  (void)stream;
  return fail(ZERO_EINVAL, "zero_debug_selftest: this library was built without ZERO_DEBUG");
#endif
}

// ------------------------------------------------------------- graph-capturable steps
static zero_status check_state(const char* who, const void* d_state) {
  if (d_state == nullptr) return fail(ZERO_EINVAL, "%s: NULL d_state", who);
  if (!zs::aligned(d_state, 8)) return fail(ZERO_EINVAL, "%s: d_state not 8-byte aligned", who);
  return ZERO_OK;
}

zero_status zero_adamw_prepare_device(const zero_adamw_hparams* d_hp, const zero_norm_result* d_clip,
                                      zero_adamw_device_state* d_state, void* stream) {
  const char* who = "zero_adamw_prepare_device";
  if (d_hp == nullptr) return fail(ZERO_EINVAL, "%s: NULL d_hp", who);
  if (!zs::aligned(d_hp, 8)) return fail(ZERO_EINVAL, "%s: d_hp not 8-byte aligned", who);
  const zero_status c = check_state(who, d_state);
  if (c != ZERO_OK) return c;
  return zs::launch_adamw_prepare(d_hp, d_clip, d_state, zs::as_stream(stream));
}

zero_status zero_adamw_step_device(float* d_master, float* d_exp_avg, float* d_exp_avg_sq, const float* d_grad,
                                   void* d_param_lowp, zero_dtype lowp_dtype, int64_t n,
                                   const zero_adamw_device_state* d_state, const zero_norm_result* d_clip,
                                   void* stream) {
  const char* who = "zero_adamw_step_device";
  if (n < 0) return fail(ZERO_EINVAL, "%s: n %lld < 0", who, (long long)n);
  const zero_status c = check_state(who, d_state);
  if (c != ZERO_OK) return c;
  if (n > 0 && (d_master == nullptr || d_exp_avg == nullptr || d_exp_avg_sq == nullptr || d_grad == nullptr))
    return fail(ZERO_EINVAL, "%s: NULL state or grad buffer", who);
  if (d_param_lowp != nullptr && lowp_dtype != ZERO_BF16 && lowp_dtype != ZERO_F16)
    return fail(ZERO_EINVAL, "%s: lowp_dtype must be BF16 or F16", who);
  if (n == 0) return ZERO_OK;
  return zs::launch_adamw(d_master, d_exp_avg, d_exp_avg_sq, d_grad, d_param_lowp, lowp_dtype, n, zs::AdamScalars{},
                          d_state, d_clip, zs::as_stream(stream));
}

zero_status zero_adamw_step_tensors_device(float* d_master, float* d_exp_avg, float* d_exp_avg_sq,
                                           const zero_tensor* d_table, int32_t n_tensors, int64_t total,
                                           zero_dtype grad_dtype, int64_t shard_start, float grad_scale,
                                           const float* d_grad_scale, const float* d_acc, void* d_param_lowp,
                                           zero_dtype lowp_dtype, int64_t n, const zero_adamw_device_state* d_state,
                                           const zero_norm_result* d_clip, void* stream) {
  const char* who = "zero_adamw_step_tensors_device";
  if (n < 0) return fail(ZERO_EINVAL, "%s: n %lld < 0", who, (long long)n);
  const zero_status c = check_state(who, d_state);
  if (c != ZERO_OK) return c;
  if (n_tensors < 0 || (n_tensors > 0 && d_table == nullptr)) return fail(ZERO_EINVAL, "%s: bad table", who);
  if (total < 0 || (n_tensors == 0 && total != 0)) return fail(ZERO_EINVAL, "%s: total does not fit the table", who);
  if (shard_start < 0 || n > total - shard_start)
    return fail(ZERO_EINVAL, "%s: [%lld, %lld) outside [0, %lld]", who, (long long)shard_start,
                (long long)(shard_start + n), (long long)total);
  if (!zs::valid_dtype(grad_dtype)) return fail(ZERO_EINVAL, "%s: bad grad_dtype %d", who, (int)grad_dtype);
  if (!std::isfinite(grad_scale)) return fail(ZERO_EINVAL, "%s: non-finite grad_scale", who);
  if (n > 0 && (d_master == nullptr || d_exp_avg == nullptr || d_exp_avg_sq == nullptr))
    return fail(ZERO_EINVAL, "%s: NULL state buffer", who);
  if (d_param_lowp != nullptr && lowp_dtype != ZERO_BF16 && lowp_dtype != ZERO_F16)
    return fail(ZERO_EINVAL, "%s: lowp_dtype must be BF16 or F16", who);
  if (n == 0) return ZERO_OK;
  return zs::launch_adamw_table(d_master, d_exp_avg, d_exp_avg_sq, d_acc, d_table, n_tensors, grad_dtype,
                                shard_start, grad_scale, d_grad_scale, d_param_lowp, lowp_dtype, n,
                                zs::AdamScalars{}, d_state, d_clip, zs::as_stream(stream));
}

}  // extern "C"
