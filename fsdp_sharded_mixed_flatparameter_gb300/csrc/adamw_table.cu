// adamw_table.cu -- AdamW with the grad read straight from the FlatParameter
// tensor table (the direct path of a step without micro-batch accumulation).
#include "adam.cuh"
#include "common.cuh"
#include "kernels.h"
#include "table.cuh"

namespace zs {

// AdamW with the grad read straight from the FlatParameter tensor table (no
// materialized fp32 flat grad): g = fl(grad_scale * x) for the grad element x
// at flat index shard_start + k, then the same update as above -- so the
// result is bit-identical to flatten (scale) + adamw_v8_kernel, while the
// step moves 2 + 28 instead of 6 + 30 bytes per parameter when there is no
// micro-batch accumulation.  A block owns 2048 consecutive shard elements;
// inside one co-aligned tensor each thread loads its 8 grads directly,
// otherwise the block stages its grads in shared memory through the table
// (source-aligned loads, tensors without grad read as zeros) and updates
// the state with coalesced scalar accesses.
constexpr int kAtBlock = 2048;

// Stores of one group of 8 updated parameters (thread t: elements k .. k+7):
// the fp32 state and the packed low-precision copy.
template <int LOWP, int LW>
__device__ __forceinline__ void store_group(float* __restrict__ p, float* __restrict__ m, float* __restrict__ v,
                                            void* __restrict__ lowp, int64_t k, const float (&pr)[8],
                                            const float (&mr)[8], const float (&vr)[8]) {
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

// A full block (2048 elements, state 32-byte aligned): thread t owns the
// group of elements k0 + 8t .. k0 + 8t + 7.  Its state loads do not depend
// on the tensor table, so they are issued first and the table lookup's
// dependent loads run while they are in flight; the grads then come straight
// from the tensor (inside one co-aligned tensor) or from the block's staged
// copy in shared memory.  A partial last block or unaligned state goes
// element by element through the staged copy.
template <int DT, int LOWP, int LW, bool DEVS>
__global__ void __launch_bounds__(256, DT == ZERO_F32 ? 3 : 4) adamw_table_kernel(float* __restrict__ p, float* __restrict__ m,
                                                             float* __restrict__ v,
                                                             const zero_tensor* __restrict__ table, int n_tensors,
                                                             int64_t shard_start, int64_t n, float gscale,
                                                             void* __restrict__ lowp, bool state_vec, AdamScalars hs,
                                                             const zero_adamw_device_state* __restrict__ ds,
                                                             const zero_norm_result* __restrict__ clip) {
  __shared__ float stage[kAtBlock + kAtBlock / 8];
  AdamScalars s;
  if (!step_scalars<DEVS>(hs, ds, s)) return;  // the prepared step is skipped
  float coef = 1.0f;
  if (clip != nullptr) {
    if (!clip->finite) return;  // non-finite grad norm: the step is skipped
    coef = clip->clip_coef;
  }
  constexpr int es = SrcTraits<DT>::esize;
  constexpr int vb = (DT == ZERO_F32) ? 32 : 16;
  const int64_t nblk = (n + kAtBlock - 1) / kAtBlock;
  // stage_range also reports non-finite grads; here that flag is unused: the
  // norm pass of this step (K1 without output) raises d_found_nonfinite, and a
  // non-finite norm has already made this kernel return above
  bool unused_flag = false;
  for (int64_t b = blockIdx.x; b < nblk; b += gridDim.x) {
    const int64_t k0 = b * kAtBlock;
    const int blen = static_cast<int>((n - k0 < kAtBlock) ? (n - k0) : kAtBlock);
    const int64_t f0 = shard_start + k0;
    const bool full = state_vec && blen == kAtBlock;  // block-uniform
    const int64_t k = k0 + 8 * threadIdx.x;
    float pr[8], mr[8], vr[8];
    bool ok = full && ZS_CHECK(k + 8 <= n && aligned(p + k, 32) && aligned(m + k, 32) && aligned(v + k, 32), 10, k);
    if (ok) {
      ld8_rw(p + k, pr);
      ld8_rw(m + k, mr);
      ld8_rw(v + k, vr);
    }
    const int ti = find_tensor_warp(table, n_tensors, f0);
    const void* tptr = table[ti].ptr;
    const int64_t toff = __ldg(&table[ti].flat_offset), tnum = __ldg(&table[ti].numel);
    const char* tsrc = tptr ? static_cast<const char*>(tptr) + es * (f0 - toff) : nullptr;
    const bool direct = full && tsrc != nullptr && toff <= f0 && f0 + kAtBlock <= toff + tnum &&
                        reinterpret_cast<uintptr_t>(tsrc) % vb == 0;  // block-uniform
    if (full) {
      float gr[8];
      if (direct) {
        ok = ok && ZS_CHECK(f0 - toff + 8 * threadIdx.x + 8 <= tnum && aligned(tsrc + es * 8 * threadIdx.x, vb) &&
                                (LOWP == 0 || aligned(static_cast<char*>(lowp) + 2 * k, LW)),
                            11, k);
        if (ok) {
          load8_src<DT>(tsrc + es * 8 * threadIdx.x, gr);
#pragma unroll
          for (int j = 0; j < 8; ++j) gr[j] = __fmul_rn(gscale, gr[j]);
        }
      } else {
        stage_range<DT>(table, n_tensors, ti, f0, f0 + kAtBlock, gscale, stage, unused_flag);
        __syncthreads();
#pragma unroll
        for (int j = 0; j < 8; ++j) gr[j] = stage[stage_idx(8 * threadIdx.x + j)];  // stride 9: no bank conflict
        __syncthreads();  // the stage is refilled by the next block
      }
      if (ok) {
#pragma unroll
        for (int j = 0; j < 8; ++j) adam_update(pr[j], mr[j], vr[j], gr[j], coef, s);
        store_group<LOWP, LW>(p, m, v, lowp, k, pr, mr, vr);
      }
    } else {
      stage_range<DT>(table, n_tensors, ti, f0, f0 + blen, gscale, stage, unused_flag);
      __syncthreads();
      for (int q = threadIdx.x; q < blen; q += blockDim.x) {
        const int64_t kq = k0 + q;
        if (!ZS_CHECK(kq < n && q < kAtBlock, 12, kq)) continue;
        float pk = p[kq], mk = m[kq], vk = v[kq];
        adam_update(pk, mk, vk, stage[stage_idx(q)], coef, s);
        p[kq] = pk;
        m[kq] = mk;
        v[kq] = vk;
        if (LOWP != 0) static_cast<unsigned short*>(lowp)[kq] = round1_rn<LOWP>(pk);
      }
      __syncthreads();
    }
  }
}

ZS_DEBUG_UNIT(adamw_table)

template <int DT, int LOWP, int LW>
static zero_status launch_table_t(float* p, float* m, float* v, const zero_tensor* table, int n_tensors,
                                  int64_t shard_start, int64_t n, float gscale, void* lowp, bool state_vec,
                                  const AdamScalars& s, const zero_adamw_device_state* ds,
                                  const zero_norm_result* clip, cudaStream_t st) {
  if (ds != nullptr)
    adamw_table_kernel<DT, LOWP, LW, true><<<one_pass_blocks(n, kAtBlock), 256, 0, st>>>(
        p, m, v, table, n_tensors, shard_start, n, gscale, lowp, state_vec, s, ds, clip);
  else
    adamw_table_kernel<DT, LOWP, LW, false><<<one_pass_blocks(n, kAtBlock), 256, 0, st>>>(
        p, m, v, table, n_tensors, shard_start, n, gscale, lowp, state_vec, s, nullptr, clip);
  return check_launch("adamw_table_kernel");
}

template <int DT, int LOWP>
static zero_status launch_table_lw(float* p, float* m, float* v, const zero_tensor* table, int n_tensors,
                                   int64_t shard_start, int64_t n, float gscale, void* lowp, const AdamScalars& s,
                                   const zero_adamw_device_state* ds, const zero_norm_result* clip, cudaStream_t st) {
  const bool sv = aligned(p, 32) && aligned(m, 32) && aligned(v, 32);
  const uintptr_t la = reinterpret_cast<uintptr_t>(lowp) % 16;
  if (LOWP == 0 || la == 0)
    return launch_table_t<DT, LOWP, 16>(p, m, v, table, n_tensors, shard_start, n, gscale, lowp, sv, s, ds, clip, st);
  if (la % 8 == 0)
    return launch_table_t<DT, LOWP, 8>(p, m, v, table, n_tensors, shard_start, n, gscale, lowp, sv, s, ds, clip, st);
  if (la % 4 == 0)
    return launch_table_t<DT, LOWP, 4>(p, m, v, table, n_tensors, shard_start, n, gscale, lowp, sv, s, ds, clip, st);
  return launch_table_t<DT, LOWP, 2>(p, m, v, table, n_tensors, shard_start, n, gscale, lowp, sv, s, ds, clip, st);
}

template <int DT>
static zero_status launch_table_dt(float* p, float* m, float* v, const zero_tensor* table, int n_tensors,
                                   int64_t shard_start, int64_t n, float gscale, void* lowp, int lowp_dtype,
                                   const AdamScalars& s, const zero_adamw_device_state* ds,
                                   const zero_norm_result* clip, cudaStream_t st) {
  if (lowp == nullptr)
    return launch_table_lw<DT, 0>(p, m, v, table, n_tensors, shard_start, n, gscale, nullptr, s, ds, clip, st);
  if (lowp_dtype == ZERO_BF16)
    return launch_table_lw<DT, ZERO_BF16>(p, m, v, table, n_tensors, shard_start, n, gscale, lowp, s, ds, clip, st);
  return launch_table_lw<DT, ZERO_F16>(p, m, v, table, n_tensors, shard_start, n, gscale, lowp, s, ds, clip, st);
}

zero_status launch_adamw_table(float* p, float* m, float* v, const zero_tensor* table, int n_tensors, int grad_dtype,
                               int64_t shard_start, float gscale, void* lowp, int lowp_dtype, int64_t n,
                               const AdamScalars& s, const zero_adamw_device_state* ds,
                               const zero_norm_result* clip, cudaStream_t st) {
  if (grad_dtype == ZERO_F32)
    return launch_table_dt<ZERO_F32>(p, m, v, table, n_tensors, shard_start, n, gscale, lowp, lowp_dtype, s, ds, clip,
                                     st);
  if (grad_dtype == ZERO_BF16)
    return launch_table_dt<ZERO_BF16>(p, m, v, table, n_tensors, shard_start, n, gscale, lowp, lowp_dtype, s, ds, clip,
                                      st);
  return launch_table_dt<ZERO_F16>(p, m, v, table, n_tensors, shard_start, n, gscale, lowp, lowp_dtype, s, ds, clip, st);
}

}  // namespace zs
