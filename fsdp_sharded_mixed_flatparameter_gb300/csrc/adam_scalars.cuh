// adam_scalars.cuh -- the per-step AdamW scalars (bias corrections of the
// ZeRO page's ZeRO1Optimizer.step) from the step count t, in binary64,
// rounded to binary32 once.  Compiled for the host (api.cu: the step count
// is a host argument) and for the device (adamw_device.cu: the step count
// lives in device memory, so a step can be captured in a CUDA graph); every
// operation is correctly rounded on both, so both give the same bits.
// Internal; not part of the C ABI.
#pragma once

#include <math.h>
#include <stdint.h>

#include "kernels.h"

namespace zs {

// Correctly rounded binary64 operations: the device intrinsics, or the plain
// host operators (the host code is compiled without fp contraction).
__host__ __device__ __forceinline__ double dmul(double a, double b) {
#ifdef __CUDA_ARCH__
  return __dmul_rn(a, b);
#else
  return a * b;
#endif
}
__host__ __device__ __forceinline__ double dadd(double a, double b) {
#ifdef __CUDA_ARCH__
  return __dadd_rn(a, b);
#else
  return a + b;
#endif
}
__host__ __device__ __forceinline__ double dsub(double a, double b) {
#ifdef __CUDA_ARCH__
  return __dsub_rn(a, b);
#else
  return a - b;
#endif
}
__host__ __device__ __forceinline__ double ddiv(double a, double b) {
#ifdef __CUDA_ARCH__
  return __ddiv_rn(a, b);
#else
  return a / b;
#endif
}
__host__ __device__ __forceinline__ double dsqrt(double a) {
#ifdef __CUDA_ARCH__
  return __dsqrt_rn(a);
#else
  return sqrt(a);
#endif
}
__host__ __device__ __forceinline__ double dfma(double a, double b, double c) {
#ifdef __CUDA_ARCH__
  return __fma_rn(a, b, c);
#else
  return fma(a, b, c);
#endif
}
__host__ __device__ __forceinline__ float to_f32(double a) {
#ifdef __CUDA_ARCH__
  return __double2float_rn(a);
#else
  return static_cast<float>(a);
#endif
}

// (h, l) <- (h, l) * (bh, bl) in double-double: the head product's rounding
// error is taken exactly by an fma, the cross terms are added to it, and the
// pair is renormalised.  Relative error ~2^-104 per product.
__host__ __device__ __forceinline__ void dd_mul(double& h, double& l, double bh, double bl) {
  const double p = dmul(h, bh);
  double e = dfma(h, bh, -p);
  e = dadd(e, dadd(dmul(h, bl), dmul(l, bh)));
  const double s = dadd(p, e);
  l = dsub(e, dsub(s, p));
  h = s;
}

// beta^t (t >= 1) by binary powering in double-double, rounded to binary64
// once: the correctly rounded power unless it lies within ~1e-29 (relative)
// of a rounding tie.  Pure arithmetic, so the host and the device agree.
__host__ __device__ __forceinline__ double pow_step(double beta, int64_t t) {
  double rh = 1.0, rl = 0.0, bh = beta, bl = 0.0;
  while (t > 0) {
    if (t & 1) dd_mul(rh, rl, bh, bl);
    t >>= 1;
    if (t > 0) dd_mul(bh, bl, bh, bl);
  }
  return dadd(rh, rl);
}

// The hyper-parameters the step accepts: lr >= 0, 0 <= beta < 1, eps > 0,
// weight_decay >= 0, all finite.
__host__ __device__ __forceinline__ bool adam_hparams_ok(double lr, double b1, double b2, double eps, double wd) {
  return isfinite(lr) && lr >= 0.0 && b1 >= 0.0 && b1 < 1.0 && b2 >= 0.0 && b2 < 1.0 && isfinite(eps) &&
         eps > 0.0 && isfinite(wd) && wd >= 0.0;
}

// Scalars of step t (t >= 1, already incremented).
__host__ __device__ __forceinline__ AdamScalars adam_scalars(double lr, double b1, double b2, double eps, double wd,
                                                            int64_t t) {
  const double bc1 = dsub(1.0, pow_step(b1, t));
  const double bc2 = dsub(1.0, pow_step(b2, t));
  AdamScalars s;
  s.step_size = to_f32(ddiv(lr, bc1));
  s.bc2_sqrt = to_f32(dsqrt(bc2));
  s.decay = to_f32(dsub(1.0, dmul(lr, wd)));
  s.b1 = to_f32(b1);
  s.omb1 = to_f32(dsub(1.0, b1));
  s.b2 = to_f32(b2);
  s.omb2 = to_f32(dsub(1.0, b2));
  s.eps = to_f32(eps);
  return s;
}

}  // namespace zs
