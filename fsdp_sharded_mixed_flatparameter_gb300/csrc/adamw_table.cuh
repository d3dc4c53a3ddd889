// adamw_table.cuh -- AdamW with the grad read straight from the FlatParameter
// tensor table (the direct path: no materialized fp32 flat grad for the last
// micro-batch).  Internal.  The kernel template is instantiated in four
// translation units, so that they compile in parallel: ACC = false (the grad
// is the last micro-batch alone: adamw_table.cu, adamw_table_p4.cu) or true
// (the earlier micro-batches' fp32 sum is added first: adamw_table_acc.cu,
// adamw_table_p4_acc.cu), with one table search per block of one part or of
// four (PARTS, below).
#pragma once

#include "adam.cuh"
#include "common.cuh"
#include "kernels.h"
#include "table.cuh"

namespace zs {

// g = fl(grad_scale * x) for the grad element x at flat index shard_start + k
// -- with ACC, g = fl(acc[k] + fl(grad_scale * x)), the value the
// accumulating flatten pass would have stored -- then the update of
// adamw.cu.  So the result is bit-identical to flatten (scale, accumulate)
// + adamw_v8_kernel, while the last micro-batch's pass writes no fp32 grad:
// without accumulation the step moves 2 + 28 instead of 6 + 30 bytes per
// parameter, with it (6 + 32 instead of 10 + 30).  A block owns 2048
// consecutive shard elements; inside one tensor each thread loads its 8
// grads directly (realigned in registers when a 16-bit source is off the
// 16-byte grid), otherwise the block stages its grads in shared memory
// through the table (source-aligned loads, tensors without grad read as
// zeros) and updates the state with coalesced scalar accesses.
constexpr int kAtBlock = 2048;

// PARTS: 2048-element parts one block updates one after the other, searching
// the table once: 4 for a table of more than 32 x 32 tensors, whose search
// takes a third round of dependent reads, else 1.  Measured on GB300: a third
// round made the update 15 % slower (a Llama list plus 3,000 small tensors:
// 2.24 against 1.94 ms); four parts per search took the 376M-element ragged
// shard (20,000 tensors) from 1.95 to 1.58 ms, but slowed Llama-7B (291
// tensors, two rounds) from 26.5 to 27.4 ms, where one block per part keeps
// more loads in flight -- and a part count read at run time cost Llama-7B 1 %,
// hence a template parameter.
inline bool table_four_parts(int n_tensors) { return n_tensors > 1024; }

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

// A full part (2048 elements, state -- and with ACC the accumulator --
// 32-byte aligned): thread t owns the group of elements k0 + 8t .. k0 + 8t + 7.
// Its state (and accumulator) loads do not depend on the tensor table, so
// they are issued first and the table lookup's dependent loads run while they
// are in flight; the grads then come straight from the tensor (inside one
// tensor, realigned in registers when needed) or from the block's staged
// copy in shared memory.  A partial last part or unaligned state goes
// element by element through the staged copy.  ACC holds 8 more values per
// thread across the lookup, so it runs 3 blocks per SM, like the fp32-grad
// variant, instead of 4 (fp32 grads with ACC: 2, which at 3 spilled).
template <int DT, int LOWP, int LW, bool DEVS, bool ACC, int PARTS>
__global__ void __launch_bounds__(256, (DT == ZERO_F32 && ACC) ? 2 : (DT == ZERO_F32 || ACC) ? 3 : 4)
    adamw_table_kernel(float* __restrict__ p, float* __restrict__ m, float* __restrict__ v,
                       const float* __restrict__ acc, const zero_tensor* __restrict__ table, int n_tensors,
                       int64_t shard_start, int64_t n, float gscale, const float* __restrict__ dscale,
                       void* __restrict__ lowp, bool state_vec, AdamScalars hs,
                       const zero_adamw_device_state* __restrict__ ds, const zero_norm_result* __restrict__ clip) {
  __shared__ float stage[kAtBlock + kAtBlock / 8];
  AdamScalars s;
  if (!step_scalars<DEVS>(hs, ds, s)) return;  // the prepared step is skipped
  if (dscale != nullptr) gscale = *dscale;  // a scale kept on the device (graph-captured mixed precision)
  float coef = 1.0f;
  if (clip != nullptr) {
    if (!clip->finite) return;  // non-finite grad norm: the step is skipped
    coef = clip->clip_coef;
  }
  constexpr int es = SrcTraits<DT>::esize;
  constexpr int vb = (DT == ZERO_F32) ? 32 : 16;
  constexpr int64_t kSpan = static_cast<int64_t>(kAtBlock) * PARTS;
  const int64_t nblk = (n + kSpan - 1) / kSpan;
  // stage_range also reports non-finite grads; here that flag is unused: the
  // norm pass of this step (K1 without output) raises d_found_nonfinite, and a
  // non-finite norm has already made this kernel return above
  bool unused_flag = false;
  for (int64_t b = blockIdx.x; b < nblk; b += gridDim.x) {
    int ti = -1;
#pragma unroll 1
    for (int part = 0; part < PARTS; ++part) {
      const int64_t k0 = b * kSpan + static_cast<int64_t>(part) * kAtBlock;
      if (k0 >= n) break;  // block-uniform: the ragged end
      const int blen = static_cast<int>((n - k0 < kAtBlock) ? (n - k0) : kAtBlock);
      const int64_t f0 = shard_start + k0;
      const bool full = state_vec && blen == kAtBlock;  // block-uniform
      const int64_t k = k0 + 8 * threadIdx.x;
      float pr[8], mr[8], vr[8], ar[8];
      bool ok = full && ZS_CHECK(k + 8 <= n && aligned(p + k, 32) && aligned(m + k, 32) && aligned(v + k, 32) &&
                                     (!ACC || aligned(acc + k, 32)),
                                 10, k);
      if (ok) {
        ld8_rw(p + k, pr);
        ld8_rw(m + k, mr);
        ld8_rw(v + k, vr);
        if (ACC) ld8_ro(acc + k, ar);
      }
      // the block's first part searches the table (dependent rounds of reads, whose latency adds to the
      // grad load's); the next parts walk forward from the tensor found, usually not moving at all
      if (ti < 0)
        ti = find_tensor_warp(table, n_tensors, f0);
      else
        while (ti + 1 < n_tensors && __ldg(&table[ti + 1].flat_offset) <= f0) ++ti;
      const void* tptr = table[ti].ptr;
      const int64_t toff = __ldg(&table[ti].flat_offset), tnum = __ldg(&table[ti].numel);
      const char* tsrc = tptr ? static_cast<const char*>(tptr) + es * (f0 - toff) : nullptr;
      // block-uniform: the block's grads lie inside one tensor, co-aligned with the state (direct) or a
      // 16-bit source off its 16-byte grid with a vector of the tensor on either side (shifted: realigned
      // in registers, as the flatten kernel does for flat offsets that are not multiples of 8)
      const bool inside = full && tsrc != nullptr && toff <= f0 && f0 + kAtBlock <= toff + tnum;
      const bool direct = inside && reinterpret_cast<uintptr_t>(tsrc) % vb == 0;
      const bool shifted = DT != ZERO_F32 && inside && !direct && f0 - toff >= 8 && f0 + kAtBlock + 8 <= toff + tnum &&
                           ZS_CHECK(aligned(tsrc, es), 13, k);
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
        } else if (shifted) {
          ok = ok && ZS_CHECK(LOWP == 0 || aligned(static_cast<char*>(lowp) + 2 * k, LW), 14, k);
          float xs[1][8];
          load8_shifted<DT, 1>(tsrc, xs);  // every lane (warp shuffles); the reads stay inside the tensor
#pragma unroll
          for (int j = 0; j < 8; ++j) gr[j] = __fmul_rn(gscale, xs[0][j]);
        } else {
          stage_range<DT>(table, n_tensors, ti, f0, f0 + kAtBlock, gscale, stage, unused_flag);
          __syncthreads();
#pragma unroll
          for (int j = 0; j < 8; ++j) gr[j] = stage[stage_idx(8 * threadIdx.x + j)];  // stride 9: no bank conflict
          __syncthreads();  // the stage is refilled by the next part
        }
        if (ok) {
          if (ACC) {
#pragma unroll
            for (int j = 0; j < 8; ++j) gr[j] = __fadd_rn(ar[j], gr[j]);
          }
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
          const float gq = ACC ? __fadd_rn(acc[kq], stage[stage_idx(q)]) : stage[stage_idx(q)];
          adam_update(pk, mk, vk, gq, coef, s);
          p[kq] = pk;
          m[kq] = mk;
          v[kq] = vk;
          if (LOWP != 0) static_cast<unsigned short*>(lowp)[kq] = round1_rn<LOWP>(pk);
        }
        __syncthreads();
      }
    }
  }
}

// The launch arguments shared by every level below.
struct TableArgs {
  float *p, *m, *v;
  const float* acc;
  const zero_tensor* table;
  int n_tensors;
  int64_t shard_start, n;
  float gscale;
  const float* dscale;
  void* lowp;
  const AdamScalars* s;
  const zero_adamw_device_state* ds;
  const zero_norm_result* clip;
  cudaStream_t st;
};

template <int DT, int LOWP, int LW, bool ACC, int PARTS>
static zero_status launch_table_t(const TableArgs& a, bool state_vec) {
  const unsigned grid = one_pass_blocks(a.n, static_cast<int64_t>(kAtBlock) * PARTS);
  if (a.ds != nullptr)
    adamw_table_kernel<DT, LOWP, LW, true, ACC, PARTS><<<grid, 256, 0, a.st>>>(
        a.p, a.m, a.v, a.acc, a.table, a.n_tensors, a.shard_start, a.n, a.gscale, a.dscale, a.lowp, state_vec, *a.s,
        a.ds, a.clip);
  else
    adamw_table_kernel<DT, LOWP, LW, false, ACC, PARTS><<<grid, 256, 0, a.st>>>(
        a.p, a.m, a.v, a.acc, a.table, a.n_tensors, a.shard_start, a.n, a.gscale, a.dscale, a.lowp, state_vec, *a.s,
        nullptr, a.clip);
  return check_launch("adamw_table_kernel");
}

template <int DT, int LOWP, bool ACC, int PARTS>
static zero_status launch_table_lw(const TableArgs& a) {
  const bool sv = aligned(a.p, 32) && aligned(a.m, 32) && aligned(a.v, 32) && (!ACC || aligned(a.acc, 32));
  const uintptr_t la = reinterpret_cast<uintptr_t>(a.lowp) % 16;
  if (LOWP == 0 || la == 0) return launch_table_t<DT, LOWP, 16, ACC, PARTS>(a, sv);
  if (la % 8 == 0) return launch_table_t<DT, LOWP, 8, ACC, PARTS>(a, sv);
  if (la % 4 == 0) return launch_table_t<DT, LOWP, 4, ACC, PARTS>(a, sv);
  return launch_table_t<DT, LOWP, 2, ACC, PARTS>(a, sv);
}

template <int DT, bool ACC, int PARTS>
static zero_status launch_table_dt(const TableArgs& a, int lowp_dtype) {
  if (a.lowp == nullptr) return launch_table_lw<DT, 0, ACC, PARTS>(a);
  if (lowp_dtype == ZERO_BF16) return launch_table_lw<DT, ZERO_BF16, ACC, PARTS>(a);
  return launch_table_lw<DT, ZERO_F16, ACC, PARTS>(a);
}

// Every grad dtype of one (ACC, PARTS) instance.
template <bool ACC, int PARTS>
static zero_status launch_table_instance(float* p, float* m, float* v, const float* acc, const zero_tensor* table,
                                         int n_tensors, int grad_dtype, int64_t shard_start, float gscale,
                                         const float* dscale, void* lowp, int lowp_dtype, int64_t n,
                                         const AdamScalars& s, const zero_adamw_device_state* ds,
                                         const zero_norm_result* clip, cudaStream_t st) {
  const TableArgs a{p, m, v, acc, table, n_tensors, shard_start, n, gscale, dscale, lowp, &s, ds, clip, st};
  if (grad_dtype == ZERO_F32) return launch_table_dt<ZERO_F32, ACC, PARTS>(a, lowp_dtype);
  if (grad_dtype == ZERO_BF16) return launch_table_dt<ZERO_BF16, ACC, PARTS>(a, lowp_dtype);
  return launch_table_dt<ZERO_F16, ACC, PARTS>(a, lowp_dtype);
}

}  // namespace zs
