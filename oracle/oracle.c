/*
 * oracle.c -- plain, slow, single-threaded CPU oracle of the flat-shard
 * optimizer step (ZeRO-1/2/3 and FSDP FlatParameter data-parallel hot path).
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check of
 * __graft_entry__ and the CPU-baseline leg of bench.py may load this file.
 * The CUDA library never links, includes or calls it, and it includes
 * nothing of the CUDA library: the two share no code, headers or tables.
 *
 * Build: gcc -O2 -ffp-contract=off -std=c11 -fPIC -shared (no -ffast-math).
 * -ffp-contract=off matters: without it GCC on aarch64 fuses a*b+c into an
 * fma, which would change the rounding of the steps below.  Every fma in
 * this file is written out explicitly with fmaf().
 *
 * Sources (four web pages on ZeRO / FSDP; each function names its passage):
 *   [ZeRO-NPU]   ai6s.net, "cann-recipes-train" ZeRO-1/2/3 on Ascend NPU
 *   [Mem-FSDP]   ybb.press, "大模型分布式训练并行与显存工程实战" (memory ledger,
 *                FSDP FlatParameter, MixedPrecision)
 *   [GradAcc]    ai6s.net, LLaMA-13B gradient accumulation + checkpointing
 *   [Infra]      cissy0802.github.io, "AI/ML 详解：训练基础设施"
 *
 * Every floating-point step is one IEEE-754 binary32 operation rounded to
 * nearest even, in the order the pages' torch code applies them, except the
 * grad norm, which is summed in binary64 with compensation (the squares of
 * binary32 values are exact in binary64).
 *
 * Pins: every function below is checked by the CPU test suite against
 * something other than itself (closed forms, invariants, library routines,
 * brute force on tiny inputs).  No function here is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1
#define ORC_F16 2

/* ------------------------------------------------------------------ dtypes */

/* bf16 -> f32: a bf16 value is the top 16 bits of the binary32 value. */
float orc_bf16_to_f32(uint16_t h) {
  uint32_t x = (uint32_t)h << 16;
  float f;
  memcpy(&f, &x, 4);
  return f;
}

/* f16 (IEEE binary16) -> f32, exact: value = (-1)^s * 2^(e-15) * (1 + m/1024),
 * subnormals 2^-14 * m/1024. */
float orc_f16_to_f32(uint16_t h) {
  uint32_t s = (h >> 15) & 1u, e = (h >> 10) & 0x1fu, m = h & 0x3ffu;
  float mag;
  if (e == 0)
    mag = ldexpf((float)m, -24);
  else if (e == 31)
    mag = m ? NAN : INFINITY;
  else
    mag = ldexpf((float)(m | 0x400u), (int)e - 25);
  return s ? -mag : mag;
}

/* f32 -> bf16, round to nearest, ties to even on the 16 dropped bits.
 * A carry out of the kept mantissa moves to the next binade (or to inf),
 * which is the correct rounding.  NaN stays NaN (quiet bit forced). */
uint16_t orc_bf16_rne(float f) {
  uint32_t x;
  memcpy(&x, &f, 4);
  if ((x & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((x >> 16) | 0x0040u);
  uint32_t hi = x >> 16, lo = x & 0xffffu;
  if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1u;
  return (uint16_t)hi;
}

/* Shift the integer significand sig right by sh bits, rounding to nearest even. */
static uint32_t rne_shift(uint32_t sig, int sh) {
  if (sh <= 0) return sig;
  if (sh > 31) return 0;
  uint32_t q = sig >> sh, r = sig & ((1u << sh) - 1u), half = 1u << (sh - 1);
  if (r > half || (r == half && (q & 1u))) q += 1u;
  return q;
}

/* f32 -> f16, round to nearest even; overflow to inf, gradual underflow. */
uint16_t orc_f16_rne(float f) {
  uint32_t x;
  memcpy(&x, &f, 4);
  uint16_t s = (uint16_t)((x >> 16) & 0x8000u);
  uint32_t ax = x & 0x7fffffffu;
  if (ax > 0x7f800000u) return (uint16_t)(s | 0x7e00u);  /* NaN */
  if (ax == 0x7f800000u) return (uint16_t)(s | 0x7c00u); /* inf */
  int e = (int)(ax >> 23) - 127;                          /* unbiased exponent */
  uint32_t sig = (ax & 0x7fffffu) | (ax >= 0x00800000u ? 0x800000u : 0u);
  if (ax < 0x00800000u) e = -126;                         /* binary32 subnormal */
  if (e >= -14) {
    /* normal binary16 range: keep 10 fraction bits; a carry bumps the exponent */
    uint32_t q = rne_shift(sig, 13);  /* 1.xxx in [2^10, 2^11] */
    uint32_t be = (uint32_t)(e + 15);
    if (q == 0x800u) { q = 0x400u; be += 1u; }
    if (be >= 31u) return (uint16_t)(s | 0x7c00u);
    return (uint16_t)(s | (be << 10) | (q & 0x3ffu));
  }
  /* subnormal binary16: value / 2^-24 = sig * 2^(e-23+24) */
  uint32_t q = rne_shift(sig, -(e + 1));
  return (uint16_t)(s | q); /* q == 0x400 becomes the smallest normal, correctly */
}

static float orc_load(const void* p, int dtype, int64_t j) {
  if (dtype == ORC_F32) return ((const float*)p)[j];
  if (dtype == ORC_BF16) return orc_bf16_to_f32(((const uint16_t*)p)[j]);
  return orc_f16_to_f32(((const uint16_t*)p)[j]);
}

/* -------------------------------------------------------------- shard range */

/* [ZeRO-NPU] section "ZeRO-1: 切分 Optimizer States", ZeRO1Optimizer.__init__:
 * chunk = ceil(total / world), start = rank * chunk,
 * end = min(start + chunk, total).  Where rank * chunk > total the page's
 * formula gives end < start; the reading taken here is the empty range
 * [total, total).  Returns 0, or 1 on invalid arguments. */
int orc_shard_range(int64_t total, int32_t world, int32_t rank, int64_t* start, int64_t* end) {
  if (total < 0 || world < 1 || rank < 0 || rank >= world) return 1;
  int64_t chunk = (total + world - 1) / world;
  int64_t s = (int64_t)rank * chunk;
  int64_t e = s + chunk;
  if (e > total) e = total;
  if (s > total) s = total;
  *start = s;
  *end = e;
  return 0;
}

/* ---------------------------------------------------------- FlatParameter */

/* [ZeRO-NPU] _flatten_gradients / _apply_update and [Mem-FSDP] section
 * "FSDP 的关键抽象：FlatParameter": the parameters are concatenated in list
 * order, so tensor i starts at the sum of the sizes of tensors 0..i-1.
 * offsets has n+1 entries; offsets[n] is the total. */
void orc_flat_offsets(const int64_t* numel, int32_t n, int64_t* offsets) {
  int64_t acc = 0;
  for (int32_t i = 0; i < n; ++i) {
    offsets[i] = acc;
    acc += numel[i];
  }
  offsets[n] = acc;
}

/* [ZeRO-NPU] _flatten_gradients (grad.view(-1).float(), zeros for a tensor
 * without grad, concatenated) restricted to the shard [s, e) of
 * ZeRO1Optimizer.step ("local_grad = flat_grad[start:end]"), with each value
 * multiplied by `scale` ([GradAcc] loss / accum_steps; [ZeRO-NPU]
 * flat_grad /= world_size) and, when `accumulate` is set, added to what dst
 * already holds ([ZeRO-NPU] GradientAccumulator.backward, fp32 add_).
 *   dst[k-s] = fl(scale * x)                 accumulate == 0
 *   dst[k-s] = fl(dst[k-s] + fl(scale * x))  accumulate == 1
 * *nonfinite is set to 1 if any fl(scale * x) is inf or NaN (it is never
 * cleared here). */
void orc_flatten(const void* const* srcs, const int64_t* numel, int32_t n, int dtype,
                 int64_t s, int64_t e, float scale, int accumulate, float* dst,
                 int32_t* nonfinite) {
  int64_t off = 0;
  for (int32_t i = 0; i < n; ++i) {
    int64_t lo = off > s ? off : s, hi = off + numel[i] < e ? off + numel[i] : e;
    for (int64_t k = lo; k < hi; ++k) {
      float x = srcs[i] ? orc_load(srcs[i], dtype, k - off) : 0.0f;
      float y = scale * x;
      if (!isfinite(y)) *nonfinite = 1;
      dst[k - s] = accumulate ? dst[k - s] + y : y;
    }
    off += numel[i];
  }
}

/* Flat micro-batch accumulation ([ZeRO-NPU] GradientAccumulator.backward;
 * [GradAcc] "loss / accum_steps", summed over the micro-batches): the same
 * rule as orc_flatten on an already-flat buffer of n values. */
void orc_accum(float* acc, const void* src, int dtype, int64_t n, float scale, int accumulate,
               int32_t* nonfinite) {
  for (int64_t k = 0; k < n; ++k) {
    float y = scale * orc_load(src, dtype, k);
    if (!isfinite(y)) *nonfinite = 1;
    acc[k] = accumulate ? acc[k] + y : y;
  }
}

/* The local half of a ZeRO-2/3 reduce-scatter ([ZeRO-NPU] section "ZeRO-2:
 * 附加切分梯度", ZeRO2Optimizer.reduce_gradients: the ranks' flat grads are
 * summed, each rank keeps its chunk, then divides it by world_size; [Mem-FSDP]
 * FSDP MixedPrecision: reduce_dtype fp32, because summing in bf16 loses
 * accuracy).  `chunks` holds n_chunks blocks of `stride` elements; block r is
 * rank r's grad values over this rank's shard, as an exchange delivers them.
 * The first n values of every block are added into acc in rank order, each
 * scaled first, with the orc_accum rule:
 *   acc = (accumulate ? acc : 0-free) + scale*x_0 + scale*x_1 + ...
 * With scale = 1/world_size (a power of two for the usual world sizes)
 * scaling each term first is exactly dividing the sum afterwards, away from
 * subnormals, so this is the page's sum-then-divide carried out in binary32
 * in rank order. */
void orc_reduce_chunks(float* acc, const void* chunks, int dtype, int32_t n_chunks, int64_t stride, int64_t n,
                       float scale, int accumulate, int32_t* nonfinite) {
  const size_t es = (dtype == ORC_F32) ? 4u : 2u;
  for (int32_t r = 0; r < n_chunks; ++r)
    orc_accum(acc, (const char*)chunks + (size_t)r * (size_t)stride * es, dtype, n, scale, accumulate || r > 0,
              nonfinite);
}

/* ------------------------------------------------------------- grad norm */

/* Sum of squares of n binary32 values (clip_grad_norm_ in [ZeRO-NPU] section
 * "组合策略" and [GradAcc]; the L2 norm is its square root).  Each square is
 * exact in binary64; the squares are added in index order with Neumaier's
 * compensated summation.  NaN in -> NaN out; otherwise inf in -> inf out. */
double orc_sqnorm(const float* g, int64_t n) {
  double s = 0.0, c = 0.0;
  int has_nan = 0, has_inf = 0;
  for (int64_t k = 0; k < n; ++k) {
    double x = (double)g[k];
    if (isnan(x)) { has_nan = 1; continue; }
    if (isinf(x)) { has_inf = 1; continue; }
    double q = x * x;
    double t = s + q;
    if (fabs(s) >= fabs(q))
      c += (s - t) + q;
    else
      c += (q - t) + s;
    s = t;
  }
  if (has_nan) return NAN;
  if (has_inf) return INFINITY;
  return s + c;
}

/* Global-norm clipping as clip_grad_norm_(params, max_norm) is used in
 * [ZeRO-NPU] section "组合策略" and [GradAcc]: norm = sqrt(sum of squares over
 * everything the rank holds plus `extra_sqnorm`, the other ranks' share);
 * coefficient = max_norm / (norm + 1e-6), clamped to at most 1; a non-finite
 * norm means the step is skipped ([ZeRO-NPU]: "if not isfinite(grad_norm)").
 * max_norm = +inf means no clipping (coefficient 1). */
void orc_clip(double sq_local, double extra_sqnorm, double max_norm, double* sqnorm,
              double* norm, float* coef, int32_t* finite) {
  double sq = sq_local + extra_sqnorm;
  double nv = sqrt(sq);
  double q = max_norm / (nv + 1e-6);
  *sqnorm = sq;
  *norm = nv;
  *finite = isfinite(nv) ? 1 : 0;
  *coef = (q < 1.0) ? (float)q : 1.0f;
}

/* --------------------------------------------------------------- AdamW */

/* Per-step scalars, computed in binary64 and rounded to binary32 once.
 * [ZeRO-NPU] ZeRO1Optimizer.step: step_count is incremented before use,
 * bias_correction1 = 1 - beta1^t, bias_correction2 = 1 - beta2^t,
 * step_size = lr / bias_correction1, the denominator divides by
 * bias_correction2 ** 0.5.  AdamW ([Mem-FSDP] section "一、显存账本", "bf16 +
 * AdamW" named as the default; no formula on the pages): decoupled decay
 * p <- p * (1 - lr * weight_decay) on the old p, before the Adam term.
 * out = {step_size, bc2_sqrt, decay, beta1, 1-beta1, beta2, 1-beta2, eps}. */
void orc_adamw_scalars(double lr, double beta1, double beta2, double eps, double wd, int64_t t,
                       float* out) {
  double bc1 = 1.0 - pow(beta1, (double)t);
  double bc2 = 1.0 - pow(beta2, (double)t);
  out[0] = (float)(lr / bc1);
  out[1] = (float)sqrt(bc2);
  out[2] = (float)(1.0 - lr * wd);
  out[3] = (float)beta1;
  out[4] = (float)(1.0 - beta1);
  out[5] = (float)beta2;
  out[6] = (float)(1.0 - beta2);
  out[7] = (float)eps;
}

/* One AdamW step over n elements of the rank's flat shard, element by
 * element, in the order of [ZeRO-NPU] ZeRO1Optimizer.step:
 *   g = grad * coef                      (clip_grad_norm_ scaling)
 *   p = p * decay                        (AdamW decoupled decay, old p)
 *   m = fma(1-b1, g, m*b1)               (exp_avg.mul_(b1).add_(g, alpha=1-b1))
 *   v = fma((1-b2)*g, g, v*b2)           (exp_avg_sq.mul_(b2).addcmul_(g, g, value=1-b2))
 *   d = sqrt(v) / bc2_sqrt + eps         (denom)
 *   p = p - step_size * (m / d)          (p += exp_avg / denom * (-step_size))
 *   lowp = round-to-nearest-even(p)      ([Mem-FSDP] bf16 param copy; f16 for the
 *                                         ZeRO-3 local chunk of [ZeRO-NPU])
 * State m, v start at 0 ([ZeRO-NPU] torch.zeros exp_avg / exp_avg_sq).
 * lowp may be NULL (no low-precision copy). */
void orc_adamw(float* p, float* m, float* v, const float* grad, uint16_t* lowp, int lowp_dtype,
               int64_t n, const float* sc, float coef) {
  const float step_size = sc[0], bc2_sqrt = sc[1], decay = sc[2];
  const float b1 = sc[3], omb1 = sc[4], b2 = sc[5], omb2 = sc[6], eps = sc[7];
  for (int64_t k = 0; k < n; ++k) {
    float g = grad[k] * coef;
    float pk = p[k] * decay;
    float mk = fmaf(omb1, g, m[k] * b1);
    float vk = fmaf(omb2 * g, g, v[k] * b2);
    float d = sqrtf(vk) / bc2_sqrt + eps;
    float u = mk / d;
    pk = pk - step_size * u;
    p[k] = pk;
    m[k] = mk;
    v[k] = vk;
    if (lowp) lowp[k] = (lowp_dtype == ORC_F16) ? orc_f16_rne(pk) : orc_bf16_rne(pk);
  }
}

/* Element-wise array conversions, for the tests' pins of the casts. */
void orc_bf16_rne_array(const float* x, uint16_t* y, int64_t n) {
  for (int64_t k = 0; k < n; ++k) y[k] = orc_bf16_rne(x[k]);
}
void orc_f16_rne_array(const float* x, uint16_t* y, int64_t n) {
  for (int64_t k = 0; k < n; ++k) y[k] = orc_f16_rne(x[k]);
}
void orc_to_f32_array(const void* x, int dtype, float* y, int64_t n) {
  for (int64_t k = 0; k < n; ++k) y[k] = orc_load(x, dtype, k);
}

/* ----------------------------------------------------- dynamic loss scale */

/* [ZeRO-NPU] section "组合策略": torch.cuda.amp.GradScaler(init_scale=2^16,
 * growth_interval=2000, backoff_factor=0.5, growth_factor=2.0); after a step
 * with overflowed grads the scale backs off and the good-step count
 * restarts, and after growth_interval good steps in a row the scale grows
 * (kept only if it stays finite).  Products in binary64, rounded to binary32. */
void orc_loss_scale_update(float* scale, int32_t* good_steps, int32_t found_inf, double growth,
                           double backoff, int32_t interval) {
  if (found_inf) {
    *scale = (float)((double)*scale * backoff);
    *good_steps = 0;
    return;
  }
  *good_steps += 1;
  if (*good_steps >= interval) {
    float g = (float)((double)*scale * growth);
    if (isfinite(g)) *scale = g;
    *good_steps = 0;
  }
}
