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
// device-to-host read, and can be replayed from a graph.
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

zero_status launch_adamw_prepare(const zero_adamw_hparams* hp, const zero_norm_result* clip,
                                 zero_adamw_device_state* state, cudaStream_t st) {
  adamw_prepare_kernel<<<1, 32, 0, st>>>(hp, clip, state);
  return check_launch("adamw_prepare_kernel");
}

}  // namespace zs
