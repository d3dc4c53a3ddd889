// adamw_device.cu -- the device half of the step counter and skip policy,
// for steps captured in a CUDA graph.
//
// The ZeRO page's loop increments step_count on the host before each step
// and skips the step (without incrementing) when the grad norm is not
// finite.  Here one thread does the same on the device: it reads the norm
// result the finalize kernel wrote, advances the step count in the
// caller's zero_adamw_device_state only for a finite norm, and stores the
// step's binary32 scalars computed by the same code as the host path
// (adam_scalars.cuh), so the AdamW kernel that follows reads them and the
// result is bit-identical to a host-driven step.  With both the count and the
// decision on the device, a whole step needs no host work and no
// device-to-host read, and can be replayed from a graph.  The dynamic loss
// scale of mixed-precision steps can live on the device as well.
#include "adam_scalars.cuh"
#include "common.cuh"
#include "kernels.h"

namespace zs {

__global__ void adamw_prepare_kernel(const zero_adamw_hparams* __restrict__ hp,
                                     const zero_norm_result* __restrict__ clip,
                                     zero_adamw_device_state* __restrict__ state) {
  if (blockIdx.x != 0 || threadIdx.x != 0) return;
  const double lr = hp->lr, b1 = hp->beta1, b2 = hp->beta2, eps = hp->eps, wd = hp->weight_decay;
  if (!adam_hparams_ok(lr, b1, b2, eps, wd)) {
    state->apply = 0;
    state->status = ZERO_EINVAL;
    return;
  }
  state->status = ZERO_OK;
  if (clip != nullptr && !clip->finite) {  // skip: the step count stays
    state->apply = 0;
    return;
  }
  const int64_t t = state->step + 1;
  const AdamScalars s = adam_scalars(lr, b1, b2, eps, wd, t);
  state->scalars[0] = s.step_size;
  state->scalars[1] = s.bc2_sqrt;
  state->scalars[2] = s.decay;
  state->scalars[3] = s.b1;
  state->scalars[4] = s.omb1;
  state->scalars[5] = s.b2;
  state->scalars[6] = s.omb2;
  state->scalars[7] = s.eps;
  state->step = t;
  state->apply = 1;
}

// The dynamic loss scale on the device (zero_loss_scale_update_device): the
// host update's rule and roundings -- binary64 products rounded to binary32,
// a grown scale kept only if finite -- then the grad passes' next unscale
// factor 1 / (scale * accum_steps), rounded once, and the overflow flag cleared.
__global__ void loss_scale_update_kernel(zero_loss_scale_state* __restrict__ st, int32_t accum_steps,
                                         double growth, double backoff, int32_t interval,
                                         const zero_norm_result* __restrict__ norm) {
  if (blockIdx.x != 0 || threadIdx.x != 0) return;
  const bool found = st->found_inf != 0 || (norm != nullptr && !norm->finite);
  if (found) {
    st->scale = __double2float_rn(__dmul_rn(static_cast<double>(st->scale), backoff));
    st->growth_tracker = 0;
  } else {
    const int32_t good = st->growth_tracker + 1;
    if (good >= interval) {
      const float grown = __double2float_rn(__dmul_rn(static_cast<double>(st->scale), growth));
      if (isfinite(grown)) st->scale = grown;
      st->growth_tracker = 0;
    } else {
      st->growth_tracker = good;
    }
  }
  st->unscale = __double2float_rn(__ddiv_rn(1.0, __dmul_rn(static_cast<double>(st->scale),
                                                            static_cast<double>(accum_steps))));
  st->found_inf = 0;
}

// One thread that records a violation on purpose without touching memory: the
// debug build's self-test of its own reporting (release builds: a no-op).
__global__ void debug_selftest_kernel(long long index) {
  if (blockIdx.x == 0 && threadIdx.x == 0) (void)ZS_CHECK(false, 999, index);
}

zero_status launch_debug_selftest(long long index, cudaStream_t st) {
  debug_selftest_kernel<<<1, 32, 0, st>>>(index);
  return check_launch("debug_selftest_kernel");
}

ZS_DEBUG_UNIT(adamw_device)

zero_status launch_loss_scale_update(zero_loss_scale_state* state, int32_t accum_steps, double growth,
                                     double backoff, int32_t interval, const zero_norm_result* norm,
                                     cudaStream_t st) {
  loss_scale_update_kernel<<<1, 32, 0, st>>>(state, accum_steps, growth, backoff, interval, norm);
  return check_launch("loss_scale_update_kernel");
}

zero_status launch_adamw_prepare(const zero_adamw_hparams* hp, const zero_norm_result* clip,
                                 zero_adamw_device_state* state, cudaStream_t st) {
  adamw_prepare_kernel<<<1, 32, 0, st>>>(hp, clip, state);
  return check_launch("adamw_prepare_kernel");
}

}  // namespace zs
