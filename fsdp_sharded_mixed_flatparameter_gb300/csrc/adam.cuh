// adam.cuh -- the per-element AdamW update shared by the flat-grad kernel
// (adamw.cu) and the kernel that reads the grads through the tensor table
// (adamw_table.cu).  Internal; not part of the C ABI.
//
// The operation order is the ZeRO page's ZeRO1Optimizer.step (ai6s.net
// "cann-recipes-train" ZeRO, section "ZeRO-1: 切分 Optimizer States"), with the
// clip coefficient applied to the grad and AdamW's decoupled decay applied to
// the old master value; every step is an explicitly rounded binary32
// intrinsic, so the compiler cannot contract or reorder it.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace zs {

__device__ __forceinline__ void adam_update(float& p, float& m, float& v, float g, float coef,
                                            const AdamScalars& s) {
  g = __fmul_rn(g, coef);
  p = __fmul_rn(p, s.decay);
  m = __fmaf_rn(s.omb1, g, __fmul_rn(m, s.b1));
  v = __fmaf_rn(__fmul_rn(s.omb2, g), g, __fmul_rn(v, s.b2));
  const float d = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), s.bc2_sqrt), s.eps);
  const float u = __fdiv_rn(m, d);
  p = __fsub_rn(p, __fmul_rn(s.step_size, u));
}

// The scalars of the step a kernel applies: the host-computed ones, or
// (DEVS) those zero_adamw_prepare_device left in device memory, where
// apply == 0 means the step is skipped (returns false).
template <bool DEVS>
__device__ __forceinline__ bool step_scalars(const AdamScalars& hs, const zero_adamw_device_state* ds,
                                             AdamScalars& s) {
  if (!DEVS) {
    s = hs;
    return true;
  }
  if (!ds->apply) return false;
  s.step_size = ds->scalars[0];
  s.bc2_sqrt = ds->scalars[1];
  s.decay = ds->scalars[2];
  s.b1 = ds->scalars[3];
  s.omb1 = ds->scalars[4];
  s.b2 = ds->scalars[5];
  s.omb2 = ds->scalars[6];
  s.eps = ds->scalars[7];
  return true;
}

}  // namespace zs
