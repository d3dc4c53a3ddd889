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
#include "common.cuh"
#include "kernels.h"
#include "table.cuh"

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

template <int LOWP>
__device__ __forceinline__ void adam_scalar(int64_t k, float* __restrict__ p, float* __restrict__ m,
                                            float* __restrict__ v, const float* __restrict__ g,
                                            void* __restrict__ lowp, float coef, const AdamScalars& s) {
  float pk = p[k], mk = m[k], vk = v[k];
  adam_update(pk, mk, vk, g[k], coef, s);
  p[k] = pk;
  m[k] = mk;
  v[k] = vk;
  if (LOWP != 0) static_cast<unsigned short*>(lowp)[k] = round1_rn<LOWP>(pk);
}

// LOWP: 0 (no copy), ZERO_BF16 or ZERO_F16.  LW: widest store (bytes) the
// low-precision pointer's alignment allows for a group of 8: 16, 8, 4 or 2.
template <int LOWP, int LW>
__global__ void __launch_bounds__(256) adamw_v8_kernel(float* __restrict__ p, float* __restrict__ m,
                                                       float* __restrict__ v, const float* __restrict__ g,
                                                       void* __restrict__ lowp, int64_t head, int64_t nvec,
                                                       int64_t n, AdamScalars s,
                                                       const zero_norm_result* __restrict__ clip) {
  float coef = 1.0f;
  if (clip != nullptr) {
    if (!clip->finite) return;  // non-finite grad norm: the step is skipped
    coef = clip->clip_coef;
  }
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t body_end = head + 8 * nvec;
  if (tid < head) adam_scalar<LOWP>(tid, p, m, v, g, lowp, coef, s);
  if (tid < n - body_end) adam_scalar<LOWP>(body_end + tid, p, m, v, g, lowp, coef, s);

  for (int64_t i = tid; i < nvec; i += stride) {
    const int64_t k = head + 8 * i;
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
template <int LOWP>
__global__ void __launch_bounds__(256) adamw_scalar_kernel(float* __restrict__ p, float* __restrict__ m,
                                                           float* __restrict__ v, const float* __restrict__ g,
                                                           void* __restrict__ lowp, int64_t n, AdamScalars s,
                                                           const zero_norm_result* __restrict__ clip) {
  float coef = 1.0f;
  if (clip != nullptr) {
    if (!clip->finite) return;
    coef = clip->clip_coef;
  }
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < n; k += stride)
    adam_scalar<LOWP>(k, p, m, v, g, lowp, coef, s);
}

// ------------------------------------------------------------------------
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

template <int DT, int LOWP, int LW>
__global__ void __launch_bounds__(256) adamw_table_kernel(float* __restrict__ p, float* __restrict__ m,
                                                          float* __restrict__ v, const zero_tensor* __restrict__ table,
                                                          int n_tensors, int64_t shard_start, int64_t n, float gscale,
                                                          void* __restrict__ lowp, bool state_vec, AdamScalars s,
                                                          const zero_norm_result* __restrict__ clip) {
  __shared__ float stage[kAtBlock + kAtBlock / 8];
  float coef = 1.0f;
  if (clip != nullptr) {
    if (!clip->finite) return;  // non-finite grad norm: the step is skipped
    coef = clip->clip_coef;
  }
  constexpr int es = SrcTraits<DT>::esize;
  constexpr int vb = (DT == ZERO_F32) ? 32 : 16;
  const int64_t nblk = (n + kAtBlock - 1) / kAtBlock;
  bool bad = false;  // the flatten pass of this step reports non-finite grads
  for (int64_t b = blockIdx.x; b < nblk; b += gridDim.x) {
    const int64_t k0 = b * kAtBlock;
    const int blen = static_cast<int>((n - k0 < kAtBlock) ? (n - k0) : kAtBlock);
    const int64_t f0 = shard_start + k0;
    const int ti = find_tensor(table, n_tensors, f0);
    const void* tptr = table[ti].ptr;
    const int64_t toff = __ldg(&table[ti].flat_offset), tnum = __ldg(&table[ti].numel);
    const char* tsrc = static_cast<const char*>(tptr) + es * (f0 - toff);
    const bool direct = state_vec && blen == kAtBlock && tptr != nullptr && toff <= f0 &&
                        f0 + kAtBlock <= toff + tnum && reinterpret_cast<uintptr_t>(tsrc) % vb == 0;
    if (direct) {
      const int64_t k = k0 + 8 * threadIdx.x;
      float gr[8], pr[8], mr[8], vr[8];
      load8_src<DT>(tsrc + es * 8 * threadIdx.x, gr);
      ld8_rw(p + k, pr);
      ld8_rw(m + k, mr);
      ld8_rw(v + k, vr);
#pragma unroll
      for (int j = 0; j < 8; ++j) adam_update(pr[j], mr[j], vr[j], __fmul_rn(gscale, gr[j]), coef, s);
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
    } else {
      stage_range<DT>(table, n_tensors, ti, f0, f0 + blen, gscale, stage, bad);
      __syncthreads();
      for (int q = threadIdx.x; q < blen; q += blockDim.x) {
        const int64_t k = k0 + q;
        float pk = p[k], mk = m[k], vk = v[k];
        adam_update(pk, mk, vk, stage[stage_idx(q)], coef, s);
        p[k] = pk;
        m[k] = mk;
        v[k] = vk;
        if (LOWP != 0) static_cast<unsigned short*>(lowp)[k] = round1_rn<LOWP>(pk);
      }
      __syncthreads();
    }
  }
}

template <int DT, int LOWP, int LW>
static zero_status launch_table_t(float* p, float* m, float* v, const zero_tensor* table, int n_tensors,
                                  int64_t shard_start, int64_t n, float gscale, void* lowp, bool state_vec,
                                  const AdamScalars& s, const zero_norm_result* clip, cudaStream_t st) {
  adamw_table_kernel<DT, LOWP, LW><<<one_pass_blocks(n, kAtBlock), 256, 0, st>>>(
      p, m, v, table, n_tensors, shard_start, n, gscale, lowp, state_vec, s, clip);
  return check_launch("adamw_table_kernel");
}

template <int DT, int LOWP>
static zero_status launch_table_lw(float* p, float* m, float* v, const zero_tensor* table, int n_tensors,
                                   int64_t shard_start, int64_t n, float gscale, void* lowp, const AdamScalars& s,
                                   const zero_norm_result* clip, cudaStream_t st) {
  const bool state_vec = aligned(p, 32) && aligned(m, 32) && aligned(v, 32);
  if (LOWP == 0)
    return launch_table_t<DT, 0, 16>(p, m, v, table, n_tensors, shard_start, n, gscale, lowp, state_vec, s, clip, st);
  const uintptr_t la = reinterpret_cast<uintptr_t>(lowp) % 16;
  if (la == 0)
    return launch_table_t<DT, LOWP, 16>(p, m, v, table, n_tensors, shard_start, n, gscale, lowp, state_vec, s, clip,
                                        st);
  if (la % 8 == 0)
    return launch_table_t<DT, LOWP, 8>(p, m, v, table, n_tensors, shard_start, n, gscale, lowp, state_vec, s, clip, st);
  if (la % 4 == 0)
    return launch_table_t<DT, LOWP, 4>(p, m, v, table, n_tensors, shard_start, n, gscale, lowp, state_vec, s, clip, st);
  return launch_table_t<DT, LOWP, 2>(p, m, v, table, n_tensors, shard_start, n, gscale, lowp, state_vec, s, clip, st);
}

template <int DT>
static zero_status launch_table_dt(float* p, float* m, float* v, const zero_tensor* table, int n_tensors,
                                   int64_t shard_start, int64_t n, float gscale, void* lowp, int lowp_dtype,
                                   const AdamScalars& s, const zero_norm_result* clip, cudaStream_t st) {
  if (lowp == nullptr)
    return launch_table_lw<DT, 0>(p, m, v, table, n_tensors, shard_start, n, gscale, nullptr, s, clip, st);
  if (lowp_dtype == ZERO_BF16)
    return launch_table_lw<DT, ZERO_BF16>(p, m, v, table, n_tensors, shard_start, n, gscale, lowp, s, clip, st);
  return launch_table_lw<DT, ZERO_F16>(p, m, v, table, n_tensors, shard_start, n, gscale, lowp, s, clip, st);
}

zero_status launch_adamw_table(float* p, float* m, float* v, const zero_tensor* table, int n_tensors, int grad_dtype,
                               int64_t shard_start, float gscale, void* lowp, int lowp_dtype, int64_t n,
                               const AdamScalars& s, const zero_norm_result* clip, cudaStream_t st) {
  if (grad_dtype == ZERO_F32)
    return launch_table_dt<ZERO_F32>(p, m, v, table, n_tensors, shard_start, n, gscale, lowp, lowp_dtype, s, clip,
                                     st);
  if (grad_dtype == ZERO_BF16)
    return launch_table_dt<ZERO_BF16>(p, m, v, table, n_tensors, shard_start, n, gscale, lowp, lowp_dtype, s, clip,
                                      st);
  return launch_table_dt<ZERO_F16>(p, m, v, table, n_tensors, shard_start, n, gscale, lowp, lowp_dtype, s, clip, st);
}

template <int LOWP, int LW>
static zero_status launch_v8(float* p, float* m, float* v, const float* g, void* lowp, int64_t head,
                             int64_t nvec, int64_t n, const AdamScalars& s, const zero_norm_result* clip,
                             cudaStream_t st) {
  adamw_v8_kernel<LOWP, LW><<<one_pass_blocks(nvec, 256), 256, 0, st>>>(p, m, v, g, lowp, head, nvec, n, s, clip);
  return check_launch("adamw_v8_kernel");
}

template <int LOWP>
static zero_status launch_lowp(float* p, float* m, float* v, const float* g, void* lowp, int64_t n,
                               const AdamScalars& s, const zero_norm_result* clip, cudaStream_t st) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p) % 32;
  const bool coaligned = (a % 4 == 0) && reinterpret_cast<uintptr_t>(m) % 32 == a &&
                         reinterpret_cast<uintptr_t>(v) % 32 == a && reinterpret_cast<uintptr_t>(g) % 32 == a &&
                         (LOWP == 0 || reinterpret_cast<uintptr_t>(lowp) % 2 == 0);
  if (!coaligned) {
    adamw_scalar_kernel<LOWP><<<one_pass_blocks(n, 256), 256, 0, st>>>(p, m, v, g, lowp, n, s, clip);
    return check_launch("adamw_scalar_kernel");
  }
  int64_t head = static_cast<int64_t>((32 - a) % 32) / 4;
  if (head > n) head = n;
  const int64_t nvec = (n - head) / 8;
  if (LOWP == 0) return launch_v8<0, 16>(p, m, v, g, lowp, head, nvec, n, s, clip, st);
  const uintptr_t la = (reinterpret_cast<uintptr_t>(lowp) + 2 * static_cast<uintptr_t>(head)) % 16;
  if (la == 0) return launch_v8<LOWP, 16>(p, m, v, g, lowp, head, nvec, n, s, clip, st);
  if (la % 8 == 0) return launch_v8<LOWP, 8>(p, m, v, g, lowp, head, nvec, n, s, clip, st);
  if (la % 4 == 0) return launch_v8<LOWP, 4>(p, m, v, g, lowp, head, nvec, n, s, clip, st);
  return launch_v8<LOWP, 2>(p, m, v, g, lowp, head, nvec, n, s, clip, st);
}

zero_status launch_adamw(float* p, float* m, float* v, const float* g, void* lowp, int lowp_dtype, int64_t n,
                         const AdamScalars& s, const zero_norm_result* clip, cudaStream_t st) {
  if (lowp == nullptr) return launch_lowp<0>(p, m, v, g, nullptr, n, s, clip, st);
  if (lowp_dtype == ZERO_BF16) return launch_lowp<ZERO_BF16>(p, m, v, g, lowp, n, s, clip, st);
  return launch_lowp<ZERO_F16>(p, m, v, g, lowp, n, s, clip, st);
}

}  // namespace zs
