// reduce.cuh -- the grad-norm reduction pieces shared by the norm kernel
// and the kernels that fuse the norm into their last pass (flatten,
// accumulate).  Internal; not part of the C ABI.
//
// Tile contract (what makes fused and separate norms agree bit for bit):
// the flat grad buffer is cut into tiles of kSqTile = 32768 elements,
// indexed from the buffer's element 0; one block of kSqThreads = 256
// threads owns a tile; thread t owns the 16 groups of 8 elements
//     e = tile * 32768 + (r * 256 + t) * 8 + i,   r = 0..15, i = 0..7,
// and adds their squares with df_add_square in (r, i) order; elements past
// the end add nothing.  The 256 thread sums go through block_sum in binary64
// and the result is the tile's partial.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace zs {

constexpr int kSqThreads = 256;
constexpr int kSqVecPerThread = 16;  // 16 x 8 = 128 elements per thread per tile
static_assert(kSqThreads * kSqVecPerThread * 8 == kSqTile, "tile size");

// hi + lo += x*x, error-free except for the rounding of lo itself
__device__ __forceinline__ void df_add_square(float& hi, float& lo, float x) {
  const float p = __fmul_rn(x, x);
  const float e = __fmaf_rn(x, x, -p);  // x*x == p + e exactly
  const float s = __fadd_rn(hi, p);     // TwoSum(hi, p) = s + t exactly
  const float bp = __fsub_rn(s, hi);
  const float t = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(p, bp));
  hi = s;
  lo = __fadd_rn(lo, __fadd_rn(t, e));
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

}  // namespace zs
