// adamw.cu -- fused bias-corrected AdamW over one rank's flat shard.
//
// One HBM pass: reads grad, master, exp_avg, exp_avg_sq (4 x 4 B) and writes
// master, exp_avg, exp_avg_sq (3 x 4 B) plus the low-precision copy (2 B):
// 30 bytes per parameter.  The per-element operation order is the ZeRO
// page's ZeRO1Optimizer.step (ai6s.net "cann-recipes-train" ZeRO, section
// "ZeRO-1: 切分 Optimizer States"), with the clip coefficient applied to the
// grad and AdamW's decoupled decay applied to the old master value; every
// step is an explicitly rounded binary32 intrinsic, so the compiler cannot
// contract or reorder it and the result is the same on every run.
//
// Work split: one pass, one thread per group of 8 consecutive elements
// (256 groups per block, as many blocks as groups need); each group is four
// 32-byte loads, three 32-byte stores and one store of 8 packed 16-bit
// values.  Up to 7 leading elements (to reach 32-byte alignment) and 7
// trailing ones are done by single threads of the same launch.
#include "adam.cuh"
#include "common.cuh"
#include "kernels.h"

namespace zs {

template <int LOWP>
__device__ __forceinline__ void adam_scalar(int64_t k, int64_t n, float* __restrict__ p, float* __restrict__ m,
                                            float* __restrict__ v, const float* __restrict__ g,
                                            void* __restrict__ lowp, float coef, const AdamScalars& s) {
  if (!ZS_CHECK(k >= 0 && k < n, 1, k)) return;
  float pk = p[k], mk = m[k], vk = v[k];
  adam_update(pk, mk, vk, g[k], coef, s);
  p[k] = pk;
  m[k] = mk;
  v[k] = vk;
  if (LOWP != 0) static_cast<unsigned short*>(lowp)[k] = round1_rn<LOWP>(pk);
}

// LOWP: 0 (no copy), ZERO_BF16 or ZERO_F16.  LW: widest store (bytes) the
// low-precision pointer's alignment allows for a group of 8: 16, 8, 4 or 2.
// DEVS: scalars and skip decision from the device step state `ds` (graph-
// capturable steps) instead of the host-computed `hs`.
template <int LOWP, int LW, bool DEVS>
__global__ void __launch_bounds__(256) adamw_v8_kernel(float* __restrict__ p, float* __restrict__ m,
                                                       float* __restrict__ v, const float* __restrict__ g,
                                                       void* __restrict__ lowp, int64_t head, int64_t nvec,
                                                       int64_t n, AdamScalars hs,
                                                       const zero_adamw_device_state* __restrict__ ds,
                                                       const zero_norm_result* __restrict__ clip) {
  AdamScalars s;
  if (!step_scalars<DEVS>(hs, ds, s)) return;  // the prepared step is skipped
  float coef = 1.0f;
  if (clip != nullptr) {
    if (!clip->finite) return;  // non-finite grad norm: the step is skipped
    coef = clip->clip_coef;
  }
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t body_end = head + 8 * nvec;
  if (tid < head) adam_scalar<LOWP>(tid, n, p, m, v, g, lowp, coef, s);
  if (tid < n - body_end) adam_scalar<LOWP>(body_end + tid, n, p, m, v, g, lowp, coef, s);

  for (int64_t i = tid; i < nvec; i += stride) {
    const int64_t k = head + 8 * i;
    if (!ZS_CHECK(k >= 0 && k + 8 <= n && aligned(p + k, 32) && aligned(m + k, 32) && aligned(v + k, 32) &&
                      aligned(g + k, 32) && (LOWP == 0 || aligned(static_cast<char*>(lowp) + 2 * k, LW)),
                  2, k))
      continue;
    float gr[8], pr[8], mr[8], vr[8];
    ld8_ro(g + k, gr);
    ld8_rw(p + k, pr);
    ld8_rw(m + k, mr);
    ld8_rw(v + k, vr);
#pragma unroll
    for (int j = 0; j < 8; ++j) adam_update(pr[j], mr[j], vr[j], gr[j], coef, s);
    st8(p + k, pr);
    st8(m + k, mr);
    st8(v + k, vr);
    if (LOWP != 0) {
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = pack2_rn<LOWP>(pr[2 * j], pr[2 * j + 1]);
      char* dst = static_cast<char*>(lowp) + 2 * k;
      if (LW == 16) {
        st16(dst, make_uint4(w[0], w[1], w[2], w[3]));
      } else if (LW == 8) {
        reinterpret_cast<uint2*>(dst)[0] = make_uint2(w[0], w[1]);
        reinterpret_cast<uint2*>(dst)[1] = make_uint2(w[2], w[3]);
      } else if (LW == 4) {
#pragma unroll
        for (int j = 0; j < 4; ++j) reinterpret_cast<uint32_t*>(dst)[j] = w[j];
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          reinterpret_cast<unsigned short*>(dst)[2 * j] = static_cast<unsigned short>(w[j] & 0xffffu);
          reinterpret_cast<unsigned short*>(dst)[2 * j + 1] = static_cast<unsigned short>(w[j] >> 16);
        }
      }
    }
  }
}

// Any alignment: one element per thread per iteration.
template <int LOWP, bool DEVS>
__global__ void __launch_bounds__(256) adamw_scalar_kernel(float* __restrict__ p, float* __restrict__ m,
                                                           float* __restrict__ v, const float* __restrict__ g,
                                                           void* __restrict__ lowp, int64_t n, AdamScalars hs,
                                                           const zero_adamw_device_state* __restrict__ ds,
                                                           const zero_norm_result* __restrict__ clip) {
  AdamScalars s;
  if (!step_scalars<DEVS>(hs, ds, s)) return;
  float coef = 1.0f;
  if (clip != nullptr) {
    if (!clip->finite) return;
    coef = clip->clip_coef;
  }
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < n; k += stride)
    adam_scalar<LOWP>(k, n, p, m, v, g, lowp, coef, s);
}

template <int LOWP, int LW>
static zero_status launch_v8(float* p, float* m, float* v, const float* g, void* lowp, int64_t head,
                             int64_t nvec, int64_t n, const AdamScalars& s, const zero_adamw_device_state* ds,
                             const zero_norm_result* clip, cudaStream_t st) {
  if (ds != nullptr)
    adamw_v8_kernel<LOWP, LW, true><<<one_pass_blocks(nvec, 256), 256, 0, st>>>(p, m, v, g, lowp, head, nvec, n, s,
                                                                                 ds, clip);
  else
    adamw_v8_kernel<LOWP, LW, false><<<one_pass_blocks(nvec, 256), 256, 0, st>>>(p, m, v, g, lowp, head, nvec, n, s,
                                                                                  nullptr, clip);
  return check_launch("adamw_v8_kernel");
}

template <int LOWP>
static zero_status launch_lowp(float* p, float* m, float* v, const float* g, void* lowp, int64_t n,
                               const AdamScalars& s, const zero_adamw_device_state* ds, const zero_norm_result* clip,
                               cudaStream_t st) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p) % 32;
  const bool coaligned = (a % 4 == 0) && reinterpret_cast<uintptr_t>(m) % 32 == a &&
                         reinterpret_cast<uintptr_t>(v) % 32 == a && reinterpret_cast<uintptr_t>(g) % 32 == a &&
                         (LOWP == 0 || reinterpret_cast<uintptr_t>(lowp) % 2 == 0);
  if (!coaligned) {
    if (ds != nullptr)
      adamw_scalar_kernel<LOWP, true><<<one_pass_blocks(n, 256), 256, 0, st>>>(p, m, v, g, lowp, n, s, ds, clip);
    else
      adamw_scalar_kernel<LOWP, false><<<one_pass_blocks(n, 256), 256, 0, st>>>(p, m, v, g, lowp, n, s, nullptr, clip);
    return check_launch("adamw_scalar_kernel");
  }
  int64_t head = static_cast<int64_t>((32 - a) % 32) / 4;
  if (head > n) head = n;
  const int64_t nvec = (n - head) / 8;
  if (LOWP == 0) return launch_v8<0, 16>(p, m, v, g, lowp, head, nvec, n, s, ds, clip, st);
  const uintptr_t la = (reinterpret_cast<uintptr_t>(lowp) + 2 * static_cast<uintptr_t>(head)) % 16;
  if (la == 0) return launch_v8<LOWP, 16>(p, m, v, g, lowp, head, nvec, n, s, ds, clip, st);
  if (la % 8 == 0) return launch_v8<LOWP, 8>(p, m, v, g, lowp, head, nvec, n, s, ds, clip, st);
  if (la % 4 == 0) return launch_v8<LOWP, 4>(p, m, v, g, lowp, head, nvec, n, s, ds, clip, st);
  return launch_v8<LOWP, 2>(p, m, v, g, lowp, head, nvec, n, s, ds, clip, st);
}

ZS_DEBUG_UNIT(adamw)

zero_status launch_adamw(float* p, float* m, float* v, const float* g, void* lowp, int lowp_dtype, int64_t n,
                         const AdamScalars& s, const zero_adamw_device_state* ds, const zero_norm_result* clip,
                         cudaStream_t st) {
  if (lowp == nullptr) return launch_lowp<0>(p, m, v, g, nullptr, n, s, ds, clip, st);
  if (lowp_dtype == ZERO_BF16) return launch_lowp<ZERO_BF16>(p, m, v, g, lowp, n, s, ds, clip, st);
  return launch_lowp<ZERO_F16>(p, m, v, g, lowp, n, s, ds, clip, st);
}

}  // namespace zs
