// sqnorm.cu -- deterministic global L2 grad norm and clip coefficient.
//
// clip_grad_norm_ as the ZeRO page's training loop (section "组合策略") and
// the LLaMA-13B gradient-accumulation page call it, in two launches:
//
//  1. sqnorm_tiles_kernel: the grad buffer is cut into fixed tiles of
//     kSqTile = 32768 elements.  A block reduces one tile at a time: each of
//     its 256 threads squares 128 elements (16 x 32-byte loads, two rounds of
//     eight) and sums them by a fixed binary tree in binary32 (depth 7), the
//     256 thread sums are added in binary64 by a fixed shuffle/shared-memory
//     tree, and the tile's binary64 partial is stored.  A persistent grid
//     strides over the tiles, so the partial of a tile does not depend on
//     which block computed it or how many blocks ran.
//  2. sqnorm_finalize_kernel: one block adds the partials in a fixed order
//     (binary64), adds the other ranks' share, takes the square root and the
//     clip coefficient, and writes the zero_norm_result.
//
// Accuracy: each square is one rounding, the tree adds at most 7 more per
// path, so the relative error of the sum of squares is below ~8 * 2^-24
// (< 5e-7; about 2.5e-7 on the norm), far inside the 1e-5 the step needs.
// No atomics: the result is bit-identical from run to run and GPU to GPU.
#include "common.cuh"
#include "kernels.h"

namespace zs {

constexpr int kSqThreads = 256;
constexpr int kSqVecPerThread = 16;  // 16 x 8 = 128 elements per thread per tile
static_assert(kSqThreads * kSqVecPerThread * 8 == kSqTile, "tile size");

__device__ __forceinline__ float sum8_sq(const float (&x)[8]) {
  float q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) q[i] = __fmul_rn(x[i], x[i]);
  return __fadd_rn(__fadd_rn(__fadd_rn(q[0], q[1]), __fadd_rn(q[2], q[3])),
                   __fadd_rn(__fadd_rn(q[4], q[5]), __fadd_rn(q[6], q[7])));
}

__device__ __forceinline__ float tree8(const float (&s)[8]) {
  return __fadd_rn(__fadd_rn(__fadd_rn(s[0], s[1]), __fadd_rn(s[2], s[3])),
                   __fadd_rn(__fadd_rn(s[4], s[5]), __fadd_rn(s[6], s[7])));
}

// Block-wide binary64 sum in a fixed order; the result is valid in thread 0.
template <int THREADS>
__device__ __forceinline__ double block_sum(double x, double* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_down_sync(0xffffffffu, x, off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = x;
  __syncthreads();
  double r = 0.0;
  if (threadIdx.x == 0) {
#pragma unroll
    for (int w = 0; w < THREADS / 32; ++w) r += red[w];
  }
  __syncthreads();  // red[] may be reused by the caller's next round
  return r;
}

// Element e of a tile belongs to thread t, vector slot r, lane i where
// e = ((r * 256) + t) * 8 + i: each 32-byte load of a warp covers 1 KiB.
template <bool VEC>
__device__ __forceinline__ float thread_tile_sum(const float* __restrict__ g, int64_t base, int64_t n) {
  float rs[2];
#pragma unroll
  for (int round = 0; round < 2; ++round) {
    float x[8][8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int64_t e = base + ((static_cast<int64_t>(round * 8 + r) * kSqThreads) + threadIdx.x) * 8;
      if (VEC) {
        ld8_ro(g + e, x[r]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) x[r][i] = (e + i < n) ? __ldg(g + e + i) : 0.0f;
      }
    }
    float s[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) s[r] = sum8_sq(x[r]);
    rs[round] = tree8(s);
  }
  return __fadd_rn(rs[0], rs[1]);
}

__global__ void __launch_bounds__(kSqThreads) sqnorm_tiles_kernel(const float* __restrict__ g, int64_t n,
                                                                  int64_t ntiles, bool vec_ok,
                                                                  double* __restrict__ partials) {
  __shared__ double red[kSqThreads / 32];
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t base = tile * kSqTile;
    float ts;
    if (vec_ok && base + kSqTile <= n)
      ts = thread_tile_sum<true>(g, base, n);
    else
      ts = thread_tile_sum<false>(g, base, n);
    const double bs = block_sum<kSqThreads>(static_cast<double>(ts), red);
    if (threadIdx.x == 0) partials[tile] = bs;
  }
}

constexpr int kFinThreads = 1024;

__global__ void __launch_bounds__(kFinThreads) sqnorm_finalize_kernel(const double* __restrict__ partials,
                                                                      int64_t ntiles, double extra_sqnorm,
                                                                      double max_norm,
                                                                      zero_norm_result* __restrict__ out) {
  __shared__ double red[kFinThreads / 32];
  double acc = 0.0;
  for (int64_t j = threadIdx.x; j < ntiles; j += kFinThreads) acc += partials[j];
  const double local = block_sum<kFinThreads>(acc, red);
  if (threadIdx.x == 0) {
    const double sq = local + extra_sqnorm;
    const double norm = __dsqrt_rn(sq);
    const double q = __ddiv_rn(max_norm, __dadd_rn(norm, 1e-6));
    zero_norm_result r;
    r.sqnorm = sq;
    r.norm = norm;
    r.clip_coef = (q < 1.0) ? __double2float_rn(q) : 1.0f;
    r.finite = isfinite(norm) ? 1 : 0;
    *out = r;
  }
}

zero_status launch_sqnorm(const float* g, int64_t n, double extra_sqnorm, double max_norm, double* partials,
                          zero_norm_result* out, cudaStream_t st) {
  const int64_t ntiles = (n + kSqTile - 1) / kSqTile;
  if (ntiles > 0) {
    const void* fn = reinterpret_cast<const void*>(&sqnorm_tiles_kernel);
    int64_t blocks = persistent_blocks(fn, kSqThreads, 0);
    if (ntiles < blocks) blocks = ntiles;
    sqnorm_tiles_kernel<<<static_cast<unsigned>(blocks), kSqThreads, 0, st>>>(g, n, ntiles, aligned(g, 32),
                                                                             partials);
    zero_status s = check_launch("sqnorm_tiles_kernel");
    if (s != ZERO_OK) return s;
  }
  sqnorm_finalize_kernel<<<1, kFinThreads, 0, st>>>(partials, ntiles, extra_sqnorm, max_norm, out);
  return check_launch("sqnorm_finalize_kernel");
}

}  // namespace zs
