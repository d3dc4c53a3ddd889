// flatten.cu -- gradient flatten/cast into the FlatParameter layout (K1),
// flat micro-batch accumulation (K2) and the local reduction of a ZeRO-2/3
// reduce-scatter (K2r).
//
// K1 implements the ZeRO page's _flatten_gradients (grad.view(-1).float(),
// zeros for a tensor without grad, concatenated in list order) restricted to
// the rank's shard, scaled by 1/accum_steps (LLaMA-13B gradient-accumulation
// page) or 1/world_size, optionally added to the fp32 accumulator.  The
// tensors are given as a device table {ptr, numel, flat_offset} sorted by
// flat offset, so thousands of tensors take one launch (the memory-ledger
// page's point about FlatParameter: one big operation instead of hundreds of
// small ones with microsecond launch costs each).
//
// Work split: the shard's destination range is cut into tiles of 8192
// elements, one block per tile (one pass); each block finds its first tensor
// in the table (L1/L2-resident) and walks forward.  A tile that lies inside
// one tensor whose source address is co-aligned with the destination is
// copied directly with 16- or 32-byte loads and 32-byte stores.  A tile inside
// one 16-bit tensor whose source is not co-aligned (flat offsets need not be
// multiples of 8) is realigned in registers: aligned source vectors, the next
// one from the neighbouring lane, a funnel shift (load8_shifted).  Any other
// tile (tensor boundaries inside it, a NULL grad, the first and last tile of
// a misaligned tensor, fp32 sources misaligned relative to the destination)
// is staged: the block reads each source segment with loads aligned to the
// SOURCE, writes the scaled binary32 values to shared memory, and then
// writes the destination with loads/stores aligned to the DESTINATION.  The
// staging buffer is padded by one word per 8 (index q -> q + q/8) so that
// both phases are free of shared-memory bank conflicts.
//
// Fused grad norm (NORM = true, used on the last micro-batch): a block then
// owns four consecutive tiles = one 32768-element norm tile and adds the
// squares of the values it writes in the order of the norm tile contract
// (reduce.cuh), so its partial equals bit for bit what the separate norm
// kernel would compute from the written buffer -- without reading it again.
//
// Norm of the sum only (STORE = false, with ACC and NORM): the last
// micro-batch of a step whose AdamW adds it to the accumulator itself
// (zero_adamw_step_tensors with d_acc) needs the norm of acc + scale * x but
// not its flat copy: the same pass, reading the accumulator and writing only
// the partials (6 instead of 10 bytes per element for 16-bit grads).
//
// Norm only (K1n, normonly_kernel below): the direct AdamW path without
// accumulation needs the norm of the grads but not the flat copy; that pass
// has its own kernel.
#include <string.h>

#include "common.cuh"
#include "kernels.h"
#include "reduce.cuh"
#include "table.cuh"

namespace zs {

template <int DT, bool ACC, bool NORM, bool STORE>
__global__ void __launch_bounds__(kFlThreads) flatten_kernel(const zero_tensor* __restrict__ table, int n_tensors,
                                                             int64_t shard_start, int64_t len, int64_t ntiles,
                                                             float* __restrict__ dst, bool dst_vec, float scale,
                                                             const float* __restrict__ dscale,
                                                             int32_t* __restrict__ flag,
                                                             double* __restrict__ partials) {
  __shared__ float stage[kFlStage];
  if (dscale != nullptr) scale = *dscale;  // a scale kept on the device (graph-captured mixed precision)
  __shared__ float2 red[kFlThreads / 32];
  constexpr int es = SrcTraits<DT>::esize;
  constexpr int vb = (DT == ZERO_F32) ? 32 : 16;
  constexpr int kPerBlock = NORM ? static_cast<int>(kSqTile / kFlTile) : 1;  // tiles per block
  static_assert(!NORM || kFlThreads == kSqThreads, "norm tile contract");
  static_assert(STORE || (ACC && NORM), "a pass that stores nothing is the norm of the accumulated sum");
  const int64_t nblocks_work = (ntiles + kPerBlock - 1) / kPerBlock;
  bool bad = false;

  for (int64_t wb = blockIdx.x; wb < nblocks_work; wb += gridDim.x) {
    const int64_t t0 = wb * kPerBlock;
    const int64_t t1 = (t0 + kPerBlock < ntiles) ? t0 + kPerBlock : ntiles;
    const int64_t k_first = shard_start + t0 * kFlTile;
    // the block's first tensor: a warp-cooperative search (a few rounds of independent loads), except for
    // the writing pass with the fused norm over a short table, where the per-thread binary search measured
    // faster (291 tensors: 5.91 vs 6.02 ms; 20,000 tensors: the warp search 1.9 % faster)
    int ti = (NORM && n_tensors <= 1024) ? find_tensor(table, n_tensors, k_first)
                                         : find_tensor_warp(table, n_tensors, k_first);
    NormAcc nacc;  // this thread's share of the norm tile
    for (int64_t tile = t0; tile < t1; ++tile) {
      const int64_t base = tile * kFlTile;
      const int tlen = static_cast<int>((len - base < kFlTile) ? (len - base) : kFlTile);
      const int64_t klo = shard_start + base, khi = klo + tlen;
      while (ti + 1 < n_tensors && __ldg(&table[ti + 1].flat_offset) <= klo) ++ti;
      const void* tptr = table[ti].ptr;
      const int64_t toff = __ldg(&table[ti].flat_offset), tnum = __ldg(&table[ti].numel);
      const char* tsrc = tptr ? static_cast<const char*>(tptr) + es * (klo - toff) : nullptr;

      const bool inside = tlen == kFlTile && dst_vec && tsrc != nullptr && toff <= klo && khi <= toff + tnum;
      const bool direct = inside && reinterpret_cast<uintptr_t>(tsrc) % vb == 0;
      // a 16-bit source inside one tensor but not co-aligned with the destination, with
      // a vector of the tensor on either side of the tile: realigned in registers
      const bool shifted = DT != ZERO_F32 && inside && !direct && klo - toff >= 8 && khi + 8 <= toff + tnum;
      if (!ZS_CHECK(!direct || (klo - toff + kFlTile <= tnum && aligned(tsrc, vb) &&
                                aligned(dst + base, 32) && base + kFlTile <= len),
                    20, tile))
        continue;
      if (!ZS_CHECK(!shifted || (klo - toff >= 8 && klo - toff + kFlTile + 8 <= tnum && aligned(tsrc, es) &&
                                 aligned(dst + base, 32) && base + kFlTile <= len),
                    53, tile))
        continue;
      if (direct || shifted) {
        // 1024 groups of 8; thread t takes groups t + 256 r, r = 0..3, all loads first
        float x[4][8];
        if (direct) {
#pragma unroll
          for (int r = 0; r < 4; ++r) load8_src<DT>(tsrc + es * 8 * (threadIdx.x + r * kFlThreads), x[r]);
        } else {
          load8_shifted<DT, 4>(tsrc, x);
        }
        float a[4][8];
        if (ACC) {
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            if (STORE)
              ld8_rw(dst + base + 8 * (threadIdx.x + r * kFlThreads), a[r]);
            else
              ld8_ro(dst + base + 8 * (threadIdx.x + r * kFlThreads), a[r]);  // read-only in this pass
          }
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float y = __fmul_rn(scale, x[r][i]);
            bad |= !finite_f(y);
            x[r][i] = ACC ? __fadd_rn(a[r][i], y) : y;
          }
          if (NORM) nacc.add8(x[r]);
          if (STORE) st8(dst + base + 8 * (threadIdx.x + r * kFlThreads), x[r]);
        }
        continue;
      }

      // staged tile: walk the tensors that overlap [klo, khi)
      stage_range<DT>(table, n_tensors, ti, klo, khi, scale, stage, bad);
      __syncthreads();
      const int ngroups = (tlen + 7) / 8;
      for (int u = threadIdx.x; u < ngroups; u += kFlThreads) {
        float y[8];
        const int64_t d = base + 8 * u;
        if (!ZS_CHECK(d < len && (!dst_vec || 8 * u + 8 > tlen || aligned(dst + d, 32)), 21, d)) continue;
        if (dst_vec && 8 * u + 8 <= tlen) {
#pragma unroll
          for (int i = 0; i < 8; ++i) y[i] = stage[stage_idx(8 * u + i)];
          if (ACC) {
            float a[8];
            if (STORE)
              ld8_rw(dst + d, a);
            else
              ld8_ro(dst + d, a);
#pragma unroll
            for (int i = 0; i < 8; ++i) y[i] = __fadd_rn(a[i], y[i]);
          }
          if (NORM) nacc.add8(y);
          if (STORE) st8(dst + d, y);
        } else {
          for (int i = 0; i < 8 && 8 * u + i < tlen; ++i) {
            const float si = stage[stage_idx(8 * u + i)];
            const float yi = ACC ? __fadd_rn(dst[d + i], si) : si;
            if (NORM) nacc.add1(i, yi);
            if (STORE) dst[d + i] = yi;
          }
        }
      }
      __syncthreads();
    }
    if (NORM) {
      const double bs = block_sum_norm<kFlThreads>(nacc, red);
      if (threadIdx.x == 0 && ZS_CHECK(wb < nblocks_work, 22, wb)) partials[wb] = bs;
    }
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0 && flag != nullptr) atomicOr(flag, 1);
}

// ------------------------------------------------------------------- K1n
// Norm only (the direct AdamW path needs the norm of the grads, not their
// flat fp32 copy): reads the grads through the table and writes only the
// norm tiles' partials, 2 bytes per element for 16-bit grads.  With so few
// bytes per element the pass is bound by instructions, not DRAM, so it has
// its own kernel with no staging buffer (small shared-memory footprint, so
// more blocks per SM) and no per-8192-element tile bookkeeping:
//  * one block per 32768-element norm tile (the tile contract of reduce.cuh);
//  * a tile that lies inside one tensor with a 16-byte aligned (32-byte for
//    fp32) source -- all but a few tiles per tensor boundary -- is read with
//    16-byte loads, eight per thread in flight (no L2 bulk prefetch: measured
//    on GB300 at 6.74B bf16 grads, a 64 KB prefetch per tile racing these
//    loads took 2.87 ms, none 1.85 ms = 7.27 TB/s; with the prefetch, four
//    loads in flight measured the same as eight and sixteen were slower at
//    152 registers);
//  * any other tile (tensor boundaries, a tensor without grad, misaligned
//    sources, the ragged end) is staged in shared memory part by part with
//    source-aligned vector loads, as the flatten kernel stages its tiles.
//    (Walking the table element by element instead cost about 50 pure tiles'
//    time per such tile: 0.88 ms for the 376M-element ragged shard of 20,000
//    tensors, against 0.26 ms staged);
//  * for 16-bit grads with a power-of-two scale (EXACT = 1; 2 when the scale
//    is 1 and the multiply goes away) every value fl(scale * w) has a square
//    with no rounding residual, so NormAcc::add2_exact gives the general
//    accumulator's bits with fewer instructions, and the non-finite flag needs
//    no per-element test: an inf or NaN value leaves the thread's sum
//    non-finite, and only then does the thread re-read its groups to decide
//    (a finite value whose square overflows binary32 gives the same sum but
//    no flag).
// The partials equal bit for bit those of the separate norm kernel over the
// flattened values, and those of the writing flatten pass with the fused norm.
// Registers: the exact-square variants are held to 64 (4 blocks per SM, no
// spills); the general one is left to the compiler's choice (46-54, no
// spills -- held to 64 it spilled).
template <int DT, int EXACT>
__global__ void __launch_bounds__(kSqThreads, EXACT ? 4 : 0)
    normonly_kernel(const zero_tensor* __restrict__ table, int n_tensors, int64_t shard_start, int64_t len,
                    int64_t ntiles, float scale, const float* __restrict__ dscale, int32_t* __restrict__ flag,
                    double* __restrict__ partials) {
  __shared__ float2 red[kSqThreads / 32];
  __shared__ float stage[kFlStage];  // tiles with tensor boundaries (37 KB: still 4 blocks per SM)
  constexpr int es = SrcTraits<DT>::esize;
  constexpr int vb = (DT == ZERO_F32) ? 32 : 16;
  static_assert(!EXACT || DT != ZERO_F32, "exact squares: 16-bit grads only");
  if (dscale != nullptr) scale = *dscale;  // (EXACT is 0 then: the host cannot check the value)
  const unsigned long long scale2 = f2_pack(scale, scale);
  bool bad = false;
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t base = tile * kSqTile;
    const int64_t k0 = shard_start + base;
    const int64_t tlen = (len - base < kSqTile) ? len - base : kSqTile;
    const int ti = find_tensor_warp(table, n_tensors, k0);
    const void* tptr = table[ti].ptr;
    const int64_t toff = __ldg(&table[ti].flat_offset), tnum = __ldg(&table[ti].numel);
    const char* tsrc = tptr ? static_cast<const char*>(tptr) + es * (k0 - toff) : nullptr;
    const bool pure = tlen == kSqTile && tsrc != nullptr && toff <= k0 && k0 + kSqTile <= toff + tnum &&
                      reinterpret_cast<uintptr_t>(tsrc) % vb == 0;  // block-uniform
    NormAcc nacc;
    if (pure && ZS_CHECK(k0 - toff + kSqTile <= tnum && aligned(tsrc, vb), 50, tile)) {
#pragma unroll
      for (int round = 0; round < 2; ++round) {
        if (DT == ZERO_F32) {
          float x[8][8];
#pragma unroll
          for (int r = 0; r < 8; ++r) ld8_ro(reinterpret_cast<const float*>(tsrc) +
                                                 8 * ((round * 8 + r) * kSqThreads + threadIdx.x), x[r]);
#pragma unroll
          for (int r = 0; r < 8; ++r) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              x[r][i] = __fmul_rn(scale, x[r][i]);
              bad |= !finite_f(x[r][i]);
            }
            nacc.add8(x[r]);
          }
        } else {
          uint4 w[8];
#pragma unroll
          for (int r = 0; r < 8; ++r) w[r] = ld16_ro(tsrc + 16 * ((round * 8 + r) * kSqThreads + threadIdx.x));
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const uint32_t ws[4] = {w[r].x, w[r].y, w[r].z, w[r].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float lo = half_bits_to_f32<DT>(ws[j] & 0xffffu), hi = half_bits_to_f32<DT>(ws[j] >> 16);
              if (EXACT) {
                const unsigned long long w2 = f2_pack(lo, hi);
                nacc.add2_exact(EXACT == 2 ? w2 : f2_mul(w2, scale2));
              } else {
                const float y0 = __fmul_rn(scale, lo), y1 = __fmul_rn(scale, hi);
                bad |= !finite_f(y0) || !finite_f(y1);
                nacc.add2(y0, y1);
              }
            }
          }
        }
      }
      if (EXACT) {  // the flag, decided only where the thread's sum went non-finite
        float h0, h1;
        f2_unpack(nacc.h, h0, h1);
        if (!finite_f(h0) || !finite_f(h1)) {
          for (int r = 0; r < kSqVecPerThread; ++r) {
            const uint4 w = ld16_ro(tsrc + 16 * (r * kSqThreads + threadIdx.x));
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
            for (int j = 0; j < 4; ++j) {
              bad |= !finite_f(__fmul_rn(scale, half_bits_to_f32<DT>(ws[j] & 0xffffu)));
              bad |= !finite_f(__fmul_rn(scale, half_bits_to_f32<DT>(ws[j] >> 16)));
            }
          }
        }
      }
    } else {
      // four 8192-element parts, each thread adding its groups of the part -- groups
      // 4 * part + r of the contract, r = 0..3, so the parts in order give the
      // contract's order.  A part inside one tensor is read straight from it (16-byte
      // loads, realigned in registers when the source is off the 16-byte grid);
      // any other is staged: the block reads each source segment of the part with
      // loads aligned to that source (stage_range) into shared memory
      int j = ti;
#pragma unroll 1
      for (int part = 0; part < static_cast<int>(kSqTile / kFlTile); ++part) {
        const int64_t plo = base + static_cast<int64_t>(part) * kFlTile;
        if (plo >= len) break;  // block-uniform: the ragged end
        const int plen = static_cast<int>((len - plo < kFlTile) ? (len - plo) : kFlTile);
        const int64_t klo = shard_start + plo;
        while (j + 1 < n_tensors && __ldg(&table[j + 1].flat_offset) <= klo) ++j;
        const void* pptr = table[j].ptr;
        const int64_t poff = __ldg(&table[j].flat_offset), pnum = __ldg(&table[j].numel);
        const char* psrc = pptr ? static_cast<const char*>(pptr) + es * (klo - poff) : nullptr;
        // block-uniform
        const bool pin = plen == kFlTile && psrc != nullptr && poff <= klo && klo + kFlTile <= poff + pnum;
        const bool pdirect = pin && reinterpret_cast<uintptr_t>(psrc) % vb == 0;
        const bool pshift = DT != ZERO_F32 && pin && !pdirect && klo - poff >= 8 && klo + kFlTile + 8 <= poff + pnum &&
                            ZS_CHECK(aligned(psrc, es), 54, klo);
        if (pdirect || pshift) {
          float x[4][8];
          if (pdirect) {
#pragma unroll
            for (int r = 0; r < 4; ++r) load8_src<DT>(psrc + es * 8 * (r * kSqThreads + threadIdx.x), x[r]);
          } else {
            load8_shifted<DT, 4>(psrc, x);  // every lane (warp shuffles); the reads stay inside the tensor
          }
#pragma unroll
          for (int r = 0; r < 4; ++r) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              x[r][i] = __fmul_rn(scale, x[r][i]);
              bad |= !finite_f(x[r][i]);
            }
            nacc.add8(x[r]);
          }
          continue;
        }
        stage_range<DT>(table, n_tensors, j, klo, klo + plen, scale, stage, bad);
        __syncthreads();
#pragma unroll 1
        for (int r = 0; r < static_cast<int>(kFlTile / (8 * kSqThreads)); ++r) {
          const int g = 8 * (r * kSqThreads + static_cast<int>(threadIdx.x));
          if (g + 8 <= plen) {
            float y[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) y[i] = stage[stage_idx(g + i)];
            nacc.add8(y);
          } else {
            for (int i = 0; i < 8 && g + i < plen; ++i) nacc.add1(i, stage[stage_idx(g + i)]);
          }
        }
        __syncthreads();  // the stage is refilled by the next part
      }
    }
    const double bs = block_sum_norm<kSqThreads>(nacc, red);
    if (threadIdx.x == 0 && ZS_CHECK(tile < ntiles, 52, tile)) partials[tile] = bs;
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0 && flag != nullptr) atomicOr(flag, 1);
}

// A normal binary32 power of two (either sign): fl(scale * w) then keeps the
// significand of a 16-bit w.
static bool pow2_scale(float scale) {
  uint32_t b;
  memcpy(&b, &scale, sizeof b);
  const uint32_t ex = (b >> 23) & 0xffu;
  return (b & 0x7fffffu) == 0u && ex != 0u && ex != 0xffu;
}

template <int DT, bool ACC, bool NORM, bool STORE = true>
static zero_status launch_flatten_t(const zero_tensor* table, int32_t n_tensors, int64_t s, int64_t e, float scale,
                                    const float* dscale, float* dst, int32_t* flag, double* partials,
                                    cudaStream_t st) {
  const int64_t len = e - s;
  const int64_t ntiles = (len + kFlTile - 1) / kFlTile;
  const int64_t per = NORM ? kSqTile / kFlTile : 1;
  const unsigned grid = one_pass_blocks(ntiles, per);
  const bool dst_vec = aligned(dst, 32);
  flatten_kernel<DT, ACC, NORM, STORE><<<grid, kFlThreads, 0, st>>>(table, n_tensors, s, len, ntiles, dst, dst_vec,
                                                                    scale, dscale, flag, partials);
  return check_launch("flatten_kernel");
}

template <int DT>
static zero_status launch_normonly(const zero_tensor* table, int32_t n_tensors, int64_t s, int64_t e, float scale,
                                   const float* dscale, int32_t* flag, double* partials, cudaStream_t st) {
  const int64_t len = e - s;
  const int64_t ntiles = (len + kSqTile - 1) / kSqTile;
  const unsigned grid = one_pass_blocks(ntiles, 1);
  if constexpr (DT != ZERO_F32) {
    if (dscale == nullptr && scale == 1.0f) {
      normonly_kernel<DT, 2><<<grid, kSqThreads, 0, st>>>(table, n_tensors, s, len, ntiles, scale, nullptr, flag,
                                                           partials);
      return check_launch("normonly_kernel");
    }
    if (dscale == nullptr && pow2_scale(scale)) {
      normonly_kernel<DT, 1><<<grid, kSqThreads, 0, st>>>(table, n_tensors, s, len, ntiles, scale, nullptr, flag,
                                                           partials);
      return check_launch("normonly_kernel");
    }
  }
  normonly_kernel<DT, 0><<<grid, kSqThreads, 0, st>>>(table, n_tensors, s, len, ntiles, scale, dscale, flag,
                                                       partials);
  return check_launch("normonly_kernel");
}

template <int DT, bool ACC>
static zero_status launch_flatten_n(const zero_tensor* table, int32_t n_tensors, int64_t s, int64_t e, float scale,
                                    const float* dscale, bool store, float* dst, int32_t* flag, double* partials,
                                    cudaStream_t st) {
  if (!store) {  // the norm of dst + the values, dst only read (ACC, dst and partials checked by the caller)
    if (!ACC || dst == nullptr || partials == nullptr) return ZERO_EINVAL;
    return launch_flatten_t<DT, true, true, false>(table, n_tensors, s, e, scale, dscale, dst, flag, partials, st);
  }
  if (dst == nullptr) {  // norm partials only: the grad is not written (ACC is rejected by the caller)
    if (ACC) return ZERO_EINVAL;
    return launch_normonly<DT>(table, n_tensors, s, e, scale, dscale, flag, partials, st);
  }
  if (partials != nullptr)
    return launch_flatten_t<DT, ACC, true>(table, n_tensors, s, e, scale, dscale, dst, flag, partials, st);
  return launch_flatten_t<DT, ACC, false>(table, n_tensors, s, e, scale, dscale, dst, flag, nullptr, st);
}

template <int DT>
static zero_status launch_flatten_dt(const zero_tensor* table, int32_t n_tensors, int64_t s, int64_t e, float scale,
                                     const float* dscale, int accumulate, float* dst, int32_t* flag,
                                     double* partials, cudaStream_t st) {
  const bool store = accumulate != 2;  // 2: the norm of the accumulated sum, nothing stored
  if (accumulate != 0)
    return launch_flatten_n<DT, true>(table, n_tensors, s, e, scale, dscale, store, dst, flag, partials, st);
  return launch_flatten_n<DT, false>(table, n_tensors, s, e, scale, dscale, store, dst, flag, partials, st);
}

zero_status launch_flatten(const zero_tensor* table, int32_t n_tensors, int src_dtype, int64_t s, int64_t e,
                           float scale, const float* dscale, int accumulate, float* dst, int32_t* flag,
                           double* partials, cudaStream_t st) {
  if (e <= s) return ZERO_OK;
  if (src_dtype == ZERO_F32)
    return launch_flatten_dt<ZERO_F32>(table, n_tensors, s, e, scale, dscale, accumulate, dst, flag, partials, st);
  if (src_dtype == ZERO_BF16)
    return launch_flatten_dt<ZERO_BF16>(table, n_tensors, s, e, scale, dscale, accumulate, dst, flag, partials, st);
  return launch_flatten_dt<ZERO_F16>(table, n_tensors, s, e, scale, dscale, accumulate, dst, flag, partials, st);
}

// ------------------------------------------------------------------- K2
// acc[k] = (ACC ? acc[k] : 0-free) + fl(scale * x[k]); groups of 8 with one
// 32-byte accumulator load/store and one 16/32-byte source load.
template <int DT, bool ACC>
__device__ __forceinline__ void accum_scalar(int64_t k, int64_t n, float* __restrict__ acc,
                                             const void* __restrict__ src, float scale, bool& bad) {
  if (!ZS_CHECK(k >= 0 && k < n, 23, k)) return;
  const float y = __fmul_rn(scale, load_elem<DT>(src, k));
  bad |= !finite_f(y);
  acc[k] = ACC ? __fadd_rn(acc[k], y) : y;
}

template <int DT, bool ACC>
__global__ void __launch_bounds__(256) accum_kernel(float* __restrict__ acc, const void* __restrict__ src,
                                                    int64_t head, int64_t nvec, int64_t n, float scale,
                                                    const float* __restrict__ dscale, int32_t* __restrict__ flag) {
  constexpr int es = SrcTraits<DT>::esize;
  if (dscale != nullptr) scale = *dscale;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t body_end = head + 8 * nvec;
  bool bad = false;
  if (tid < head) accum_scalar<DT, ACC>(tid, n, acc, src, scale, bad);
  if (tid < n - body_end) accum_scalar<DT, ACC>(body_end + tid, n, acc, src, scale, bad);
  const char* s8 = static_cast<const char*>(src);
  for (int64_t i = tid; i < nvec; i += stride) {
    const int64_t k = head + 8 * i;
    if (!ZS_CHECK(k + 8 <= n && aligned(acc + k, 32) && aligned(s8 + es * k, DT == ZERO_F32 ? 32 : 16), 24, k))
      continue;
    float x[8], a[8];
    load8_src<DT>(s8 + es * k, x);
    if (ACC) ld8_rw(acc + k, a);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float y = __fmul_rn(scale, x[j]);
      bad |= !finite_f(y);
      x[j] = ACC ? __fadd_rn(a[j], y) : y;
    }
    st8(acc + k, x);
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0 && flag != nullptr) atomicOr(flag, 1);
}

template <int DT, bool ACC>
__global__ void __launch_bounds__(256) accum_scalar_kernel(float* __restrict__ acc, const void* __restrict__ src,
                                                           int64_t n, float scale, const float* __restrict__ dscale,
                                                           int32_t* __restrict__ flag) {
  if (dscale != nullptr) scale = *dscale;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  bool bad = false;
  for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < n; k += stride)
    accum_scalar<DT, ACC>(k, n, acc, src, scale, bad);
  if (__syncthreads_or(bad) && threadIdx.x == 0 && flag != nullptr) atomicOr(flag, 1);
}

// K2 with the fused grad norm: one block per 32768-element norm tile, thread
// t handles groups r * 256 + t (r = 0..15) of the tile, four at a time with
// their loads first, and adds the squares of the values it writes in the
// norm tile contract's order.  `vec`: acc is 32-byte aligned and src is
// aligned for its 8-element vector; otherwise every element goes scalar.
template <int DT, bool ACC>
__global__ void __launch_bounds__(kSqThreads) accum_norm_kernel(float* __restrict__ acc, const void* __restrict__ src,
                                                                int64_t n, int64_t ntiles, bool vec, float scale,
                                                                const float* __restrict__ dscale,
                                                                int32_t* __restrict__ flag,
                                                                double* __restrict__ partials) {
  __shared__ float2 red[kSqThreads / 32];
  constexpr int es = SrcTraits<DT>::esize;
  if (dscale != nullptr) scale = *dscale;
  const char* s8 = static_cast<const char*>(src);
  bool bad = false;
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    NormAcc nacc;
    const int64_t base = tile * kSqTile;
#pragma unroll 1
    for (int r0 = 0; r0 < kSqVecPerThread; r0 += 4) {
      float x[4][8], a[4][8];
      bool full[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int64_t k = base + (static_cast<int64_t>(r0 + q) * kSqThreads + threadIdx.x) * 8;
        full[q] = vec && k + 8 <= n;
        if (full[q] && !ZS_CHECK(aligned(acc + k, 32) && aligned(s8 + es * k, DT == ZERO_F32 ? 32 : 16), 25, k))
          full[q] = false;  // (debug build) treated as a ragged group: element accesses only
        if (full[q]) {
          load8_src<DT>(s8 + es * k, x[q]);
          if (ACC) ld8_rw(acc + k, a[q]);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int64_t k = base + (static_cast<int64_t>(r0 + q) * kSqThreads + threadIdx.x) * 8;
        if (full[q]) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float y = __fmul_rn(scale, x[q][i]);
            bad |= !finite_f(y);
            x[q][i] = ACC ? __fadd_rn(a[q][i], y) : y;
          }
          nacc.add8(x[q]);
          st8(acc + k, x[q]);
        } else {
          for (int i = 0; i < 8 && k + i < n; ++i) {
            const float y = __fmul_rn(scale, load_elem<DT>(src, k + i));
            bad |= !finite_f(y);
            const float o = ACC ? __fadd_rn(acc[k + i], y) : y;
            nacc.add1(i, o);
            acc[k + i] = o;
          }
        }
      }
    }
    const double bs = block_sum_norm<kSqThreads>(nacc, red);
    if (threadIdx.x == 0 && ZS_CHECK(tile < ntiles, 26, tile)) partials[tile] = bs;
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0 && flag != nullptr) atomicOr(flag, 1);
}

// ------------------------------------------------------------------- K2r
// The local half of a ZeRO-2/3 reduce-scatter (the ZeRO page's ZeRO-2
// reduce_gradients: the ranks' flat grads summed, each rank keeping its
// chunk, divided by world_size; the memory-ledger page: reduce in fp32).
// An all-to-all exchange has brought every rank's values of this rank's
// shard here as n_chunks blocks `stride_bytes` apart (block r = rank r's);
// they are added into the fp32 accumulator in rank order, each scaled
// first (scale = 1/world_size, times 1/accum_steps when micro-batches are
// reduced one by one):
//     acc = (ACC ? acc : first term) + s*x_0 + s*x_1 + ...
// exactly the rule of n_chunks accumulate passes, but in one pass: every
// block is read once (2 bytes per element and rank for 16-bit grads) and
// the accumulator is read (ACC) and written once.  The exchange moves the
// grads in their own 16-bit type; only the sum is binary32.
// Work split and fused norm as accum_norm_kernel: one block per 32768-
// element norm tile; in a tile that is whole and vector-aligned, thread t
// takes its groups r*256 + t two at a time and loads up to four ranks'
// blocks of them together (eight 16/32-byte loads in flight per thread)
// before adding them in rank order; the ragged last tile goes element by
// element.  NORM adds the squares of the final values in the norm tile
// contract's order (add8 and add1 give the same bits).
constexpr int kRcGroups = 2;  // groups of 8 elements a thread carries at a time

template <int DT, int B>
__device__ __forceinline__ void reduce_batch(float (&a)[kRcGroups][8], const char* __restrict__ src,
                                             int64_t stride_bytes, const int64_t (&k)[kRcGroups], float scale,
                                             bool first_is_set, bool& bad) {
  constexpr int es = SrcTraits<DT>::esize;
  float x[B][kRcGroups][8];
#pragma unroll
  for (int u = 0; u < B; ++u)
#pragma unroll
    for (int q = 0; q < kRcGroups; ++q) load8_src<DT>(src + u * stride_bytes + es * k[q], x[u][q]);
#pragma unroll
  for (int u = 0; u < B; ++u) {
    const bool set = first_is_set && u == 0;  // the first rank's value starts the sum (no add: -0 stays -0)
#pragma unroll
    for (int q = 0; q < kRcGroups; ++q) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float y = __fmul_rn(scale, x[u][q][i]);
        bad |= !finite_f(y);
        a[q][i] = set ? y : __fadd_rn(a[q][i], y);
      }
    }
  }
}

template <int DT, bool ACC, bool NORM>
__global__ void __launch_bounds__(kSqThreads) reduce_chunks_kernel(float* __restrict__ acc,
                                                                   const char* __restrict__ src, int n_chunks,
                                                                   int64_t stride_bytes, int64_t n, int64_t ntiles,
                                                                   bool vec, float scale,
                                                                   const float* __restrict__ dscale,
                                                                   int32_t* __restrict__ flag,
                                                                   double* __restrict__ partials) {
  __shared__ float2 red[kSqThreads / 32];
  [[maybe_unused]] constexpr int es = SrcTraits<DT>::esize;  // (the debug build's alignment checks)
  [[maybe_unused]] constexpr int vb = (DT == ZERO_F32) ? 32 : 16;
  if (dscale != nullptr) scale = *dscale;
  bool bad = false;
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    NormAcc nacc;
    const int64_t base = tile * kSqTile;
    if (vec && base + kSqTile <= n) {  // block-uniform: every group of the tile is a full vector group
#pragma unroll 1
      for (int r0 = 0; r0 < kSqVecPerThread; r0 += kRcGroups) {
        float a[kRcGroups][8];
        int64_t k[kRcGroups];
        bool ok = true;
#pragma unroll
        for (int q = 0; q < kRcGroups; ++q) {
          k[q] = base + (static_cast<int64_t>(r0 + q) * kSqThreads + threadIdx.x) * 8;
          ok = ok && ZS_CHECK(k[q] + 8 <= n && aligned(acc + k[q], 32) && aligned(src + es * k[q], vb), 27, k[q]);
        }
        if (!ok) continue;  // (debug build only)
#pragma unroll
        for (int q = 0; q < kRcGroups; ++q) {
          if (ACC) {
            ld8_rw(acc + k[q], a[q]);
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) a[q][i] = 0.0f;
          }
        }
        int c = 0;
#pragma unroll 1
        for (; c + 4 <= n_chunks; c += 4)
          reduce_batch<DT, 4>(a, src + c * stride_bytes, stride_bytes, k, scale, !ACC && c == 0, bad);
        if (c + 2 <= n_chunks) {
          reduce_batch<DT, 2>(a, src + c * stride_bytes, stride_bytes, k, scale, !ACC && c == 0, bad);
          c += 2;
        }
        if (c < n_chunks) reduce_batch<DT, 1>(a, src + c * stride_bytes, stride_bytes, k, scale, !ACC && c == 0, bad);
#pragma unroll
        for (int q = 0; q < kRcGroups; ++q) {
          if (NORM) nacc.add8(a[q]);
          st8(acc + k[q], a[q]);
        }
      }
    } else {  // the ragged last tile, or buffers without the vector alignment: element by element
      for (int r = 0; r < kSqVecPerThread; ++r) {
        const int64_t k = base + (static_cast<int64_t>(r) * kSqThreads + threadIdx.x) * 8;
        for (int i = 0; i < 8 && k + i < n; ++i) {
          const int64_t j = k + i;
          if (!ZS_CHECK(j >= 0 && j < n, 28, j)) continue;
          float o = ACC ? acc[j] : 0.0f;
          for (int c = 0; c < n_chunks; ++c) {
            const float y = __fmul_rn(scale, load_elem<DT>(src + c * stride_bytes, j));
            bad |= !finite_f(y);
            o = (!ACC && c == 0) ? y : __fadd_rn(o, y);
          }
          if (NORM) nacc.add1(i, o);
          acc[j] = o;
        }
      }
    }
    if (NORM) {
      const double bs = block_sum_norm<kSqThreads>(nacc, red);
      if (threadIdx.x == 0 && ZS_CHECK(tile < ntiles, 29, tile)) partials[tile] = bs;
    }
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0 && flag != nullptr) atomicOr(flag, 1);
}

ZS_DEBUG_UNIT(flatten)

template <int DT, bool ACC>
static zero_status launch_accum_t(float* acc, const void* src, int64_t n, float scale, const float* dscale,
                                  int32_t* flag, cudaStream_t st) {
  constexpr int es = SrcTraits<DT>::esize;
  constexpr uintptr_t vb = (DT == ZERO_F32) ? 32 : 16;
  const uintptr_t aa = reinterpret_cast<uintptr_t>(acc) % 32;
  int64_t head = (aa % 4 == 0) ? static_cast<int64_t>((32 - aa) % 32) / 4 : -1;
  if (head > n) head = n;
  const bool vec = head >= 0 && reinterpret_cast<uintptr_t>(src) % es == 0 &&
                   (reinterpret_cast<uintptr_t>(src) + es * static_cast<uintptr_t>(head)) % vb == 0;
  if (!vec) {
    accum_scalar_kernel<DT, ACC><<<one_pass_blocks(n, 256), 256, 0, st>>>(acc, src, n, scale, dscale, flag);
    return check_launch("accum_scalar_kernel");
  }
  const int64_t nvec = (n - head) / 8;
  accum_kernel<DT, ACC><<<one_pass_blocks(nvec, 256), 256, 0, st>>>(acc, src, head, nvec, n, scale, dscale,
                                                                                      flag);
  return check_launch("accum_kernel");
}

template <int DT, bool ACC>
static zero_status launch_accum_n(float* acc, const void* src, int64_t n, float scale, const float* dscale,
                                  int32_t* flag, double* partials, cudaStream_t st) {
  if (partials == nullptr) return launch_accum_t<DT, ACC>(acc, src, n, scale, dscale, flag, st);
  constexpr uintptr_t vb = (DT == ZERO_F32) ? 32 : 16;
  const bool vec = aligned(acc, 32) && aligned(src, vb);
  const int64_t ntiles = (n + kSqTile - 1) / kSqTile;
  accum_norm_kernel<DT, ACC><<<one_pass_blocks(ntiles, 1), kSqThreads, 0, st>>>(acc, src, n, ntiles, vec, scale, dscale,
                                                                               flag, partials);
  return check_launch("accum_norm_kernel");
}

zero_status launch_accum(float* acc, const void* src, int src_dtype, int64_t n, float scale, const float* dscale,
                         int accumulate, int32_t* flag, double* partials, cudaStream_t st) {
  if (n <= 0) return ZERO_OK;
  switch (src_dtype * 2 + (accumulate ? 1 : 0)) {
    case ZERO_F32 * 2: return launch_accum_n<ZERO_F32, false>(acc, src, n, scale, dscale, flag, partials, st);
    case ZERO_F32 * 2 + 1: return launch_accum_n<ZERO_F32, true>(acc, src, n, scale, dscale, flag, partials, st);
    case ZERO_BF16 * 2: return launch_accum_n<ZERO_BF16, false>(acc, src, n, scale, dscale, flag, partials, st);
    case ZERO_BF16 * 2 + 1: return launch_accum_n<ZERO_BF16, true>(acc, src, n, scale, dscale, flag, partials, st);
    case ZERO_F16 * 2: return launch_accum_n<ZERO_F16, false>(acc, src, n, scale, dscale, flag, partials, st);
    default: return launch_accum_n<ZERO_F16, true>(acc, src, n, scale, dscale, flag, partials, st);
  }
}

template <int DT, bool ACC, bool NORM>
static zero_status launch_reduce_chunks_t(float* acc, const void* src, int n_chunks, int64_t stride, int64_t n,
                                          float scale, const float* dscale, int32_t* flag, double* partials,
                                          cudaStream_t st) {
  constexpr int64_t es = SrcTraits<DT>::esize;
  constexpr uintptr_t vb = (DT == ZERO_F32) ? 32 : 16;
  const int64_t stride_bytes = stride * es;
  const bool vec = aligned(acc, 32) && aligned(src, vb) && stride_bytes % static_cast<int64_t>(vb) == 0;
  const int64_t ntiles = (n + kSqTile - 1) / kSqTile;
  reduce_chunks_kernel<DT, ACC, NORM><<<one_pass_blocks(ntiles, 1), kSqThreads, 0, st>>>(
      acc, static_cast<const char*>(src), n_chunks, stride_bytes, n, ntiles, vec, scale, dscale, flag, partials);
  return check_launch("reduce_chunks_kernel");
}

template <int DT, bool ACC>
static zero_status launch_reduce_chunks_n(float* acc, const void* src, int n_chunks, int64_t stride, int64_t n,
                                          float scale, const float* dscale, int32_t* flag, double* partials,
                                          cudaStream_t st) {
  if (partials != nullptr)
    return launch_reduce_chunks_t<DT, ACC, true>(acc, src, n_chunks, stride, n, scale, dscale, flag, partials, st);
  return launch_reduce_chunks_t<DT, ACC, false>(acc, src, n_chunks, stride, n, scale, dscale, flag, nullptr, st);
}

zero_status launch_reduce_chunks(float* acc, const void* src, int src_dtype, int n_chunks, int64_t stride, int64_t n,
                                 float scale, const float* dscale, int accumulate, int32_t* flag, double* partials,
                                 cudaStream_t st) {
  if (n <= 0) return ZERO_OK;
  // one block (one rank, or one FSDP unit on one rank) is the accumulate rule itself: the K2
  // kernels keep four groups' loads in flight where this one would hold two (measured on
  // Llama-7B as 34 units: 6.04 TB/s here against K2's ~7.1)
  if (n_chunks == 1) return launch_accum(acc, src, src_dtype, n, scale, dscale, accumulate, flag, partials, st);
  switch (src_dtype * 2 + (accumulate ? 1 : 0)) {
    case ZERO_F32 * 2:
      return launch_reduce_chunks_n<ZERO_F32, false>(acc, src, n_chunks, stride, n, scale, dscale, flag, partials, st);
    case ZERO_F32 * 2 + 1:
      return launch_reduce_chunks_n<ZERO_F32, true>(acc, src, n_chunks, stride, n, scale, dscale, flag, partials, st);
    case ZERO_BF16 * 2:
      return launch_reduce_chunks_n<ZERO_BF16, false>(acc, src, n_chunks, stride, n, scale, dscale, flag, partials, st);
    case ZERO_BF16 * 2 + 1:
      return launch_reduce_chunks_n<ZERO_BF16, true>(acc, src, n_chunks, stride, n, scale, dscale, flag, partials, st);
    case ZERO_F16 * 2:
      return launch_reduce_chunks_n<ZERO_F16, false>(acc, src, n_chunks, stride, n, scale, dscale, flag, partials, st);
    default:
      return launch_reduce_chunks_n<ZERO_F16, true>(acc, src, n_chunks, stride, n, scale, dscale, flag, partials, st);
  }
}

}  // namespace zs
