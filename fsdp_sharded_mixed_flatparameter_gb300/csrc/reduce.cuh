// reduce.cuh -- the grad-norm reduction pieces shared by the norm kernel
// and the kernels that fuse the norm into their pass (flatten, accumulate,
// norm-only).  Internal; not part of the C ABI.
//
// Tile contract (what makes fused and separate norms agree bit for bit):
// the flat grad buffer is cut into tiles of kSqTile = 32768 elements,
// indexed from the buffer's element 0; one block of kSqThreads = 256
// threads owns a tile; thread t owns the 16 groups of 8 elements
//     e = tile * 32768 + (r * 256 + t) * 8 + i,   r = 0..15, i = 0..7,
// and adds their squares into a NormAcc: even i into lane 0, odd i into
// lane 1, each lane in increasing (r, i) order; elements past the end add
// nothing.  The thread's value is NormAcc::value(), lane 0 + lane 1 as a
// double-float; block_sum_norm adds the 256 thread values in double-float
// (a shuffle tree down each warp, then the 8 warp values in warp order) and
// the tile's partial is the binary64 sum of the result's two words.
//
// Everything up to the partial runs on the FP32 pipes: binary64 arithmetic
// is a small fraction of the binary32 rate on GB300, and a per-thread
// binary64 reduction was measured to keep that pipe ~40 % busy in the
// norm-only pass.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace zs {

constexpr int kSqThreads = 256;
constexpr int kSqVecPerThread = 16;  // 16 x 8 = 128 elements per thread per tile
static_assert(kSqThreads * kSqVecPerThread * 8 == kSqTile, "tile size");

// Packed pair arithmetic (sm_100+): one instruction applies the IEEE
// round-to-nearest operation to two binary32 lanes, so every lane gets
// exactly the bits the scalar operation would give.
__device__ __forceinline__ unsigned long long f2_pack(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long f2_sub(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// A double-float: the unevaluated sum h + l of two binary32 values.
struct DF {
  float h, l;
};

// Two double-float accumulators (lane 0: even elements, lane 1: odd ones),
// each an unevaluated sum h + l of two binary32 values.  Adding x*x: the
// square is split exactly as x*x = p + e (one fma); p joins h by an
// error-free TwoSum, s + t = h + p exactly; t and e go into l.  The relative
// error of a lane is ~n * 2^-48 -- about 1e-14 here -- and non-finite inputs
// make the total non-finite.  Lanes are updated in pairs with packed
// instructions (half the instructions of scalar code); add1 does the same
// arithmetic on one lane for ragged groups, giving the same bits.
struct NormAcc {
  unsigned long long h = 0ull, l = 0ull;  // lane 0 in the low word

  __device__ __forceinline__ void add2(float x0, float x1) {
    const unsigned long long x = f2_pack(x0, x1);
    const unsigned long long p = f2_mul(x, x);
    const unsigned long long e = f2_fma(x, x, p ^ 0x8000000080000000ull);  // x*x - p, exact
    const unsigned long long s = f2_add(h, p);
    const unsigned long long bp = f2_sub(s, h);
    const unsigned long long t = f2_add(f2_sub(h, f2_sub(s, bp)), f2_sub(p, bp));
    h = s;
    l = f2_add(l, f2_add(t, e));
  }
  __device__ __forceinline__ void add8(const float (&x)[8]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) add2(x[2 * j], x[2 * j + 1]);
  }
  // add2 for a packed pair whose squares leave no residual: e = x*x - p
  // rounds to a zero in both lanes.  That holds for every fl(s * w) with w a
  // bf16 or f16 value and s a power of two: the square of a significand of
  // at most 11 bits fits binary32's 24 exactly, and where it underflows the
  // residual is at most half of the smallest subnormal, which rounds to a
  // zero (the tie goes to the even 0).  t + e then differs from t at most
  // in the sign of a zero, and l -- +0 at the start, never -0 after, since a
  // sum is -0 only when both terms are -- gets the same l + (t + e) = l + t.
  // So this gives exactly add2's bits with three fewer instructions.  (An
  // ordered Fast2Sum in place of TwoSum gives the same error term with fewer
  // FMA-pipe operations, but needs scalar max/min and repacking; it measured
  // no faster.)
  __device__ __forceinline__ void add2_exact(unsigned long long x) {
    const unsigned long long p = f2_mul(x, x);
    const unsigned long long s = f2_add(h, p);
    const unsigned long long bp = f2_sub(s, h);
    const unsigned long long t = f2_add(f2_sub(h, f2_sub(s, bp)), f2_sub(p, bp));
    h = s;
    l = f2_add(l, t);
  }
  // element i (0..7) of a group alone, e.g. the ragged end of a buffer
  __device__ __forceinline__ void add1(int i, float x) {
    float h0, h1, l0, l1;
    f2_unpack(h, h0, h1);
    f2_unpack(l, l0, l1);
    float& hh = (i & 1) ? h1 : h0;
    float& ll = (i & 1) ? l1 : l0;
    const float p = __fmul_rn(x, x);
    const float e = __fmaf_rn(x, x, -p);
    const float s = __fadd_rn(hh, p);
    const float bp = __fsub_rn(s, hh);
    const float t = __fadd_rn(__fsub_rn(hh, __fsub_rn(s, bp)), __fsub_rn(p, bp));
    hh = s;
    ll = __fadd_rn(ll, __fadd_rn(t, e));
    h = f2_pack(h0, h1);
    l = f2_pack(l0, l1);
  }
  __device__ __forceinline__ DF value() const;
};

// s + e = a + b exactly, s = fl(a + b) (TwoSum: no condition on a, b).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bp = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

// (a.h + a.l) + (b.h + b.l): the heads by TwoSum, the tails and its error
// added, then renormalised by Fast2Sum (the head sum dominates the tail
// sum).  For sums of squares (no cancellation) the relative error is a few
// units of 2^-48; an inf or NaN anywhere makes the result non-finite.
__device__ __forceinline__ DF df_add(DF a, DF b) {
  float s, e;
  two_sum(a.h, b.h, s, e);
  const float t = __fadd_rn(__fadd_rn(a.l, b.l), e);
  const float hh = __fadd_rn(s, t);
  return DF{hh, __fsub_rn(t, __fsub_rn(hh, s))};
}

__device__ __forceinline__ DF NormAcc::value() const {
  float h0, h1, l0, l1;
  f2_unpack(h, h0, h1);
  f2_unpack(l, l0, l1);
  return df_add(DF{h0, l0}, DF{h1, l1});
}

// The tile partial of the tile contract: the block's 256 NormAcc values in
// double-float, in a fixed order, rounded once to binary64.  Valid in
// thread 0; every thread of the block must call it.
template <int THREADS>
__device__ __forceinline__ double block_sum_norm(const NormAcc& acc, float2* red) {
  DF x = acc.value();
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const DF y{__shfl_down_sync(0xffffffffu, x.h, off), __shfl_down_sync(0xffffffffu, x.l, off)};
    x = df_add(x, y);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = make_float2(x.h, x.l);
  __syncthreads();
  double r = 0.0;
  if (threadIdx.x == 0) {
    DF a{red[0].x, red[0].y};
#pragma unroll
    for (int w = 1; w < THREADS / 32; ++w) a = df_add(a, DF{red[w].x, red[w].y});
    r = static_cast<double>(a.h) + static_cast<double>(a.l);
  }
  __syncthreads();  // red[] may be reused by the caller's next round
  return r;
}

// Block-wide binary64 sum in a fixed order (the finalize over tile
// partials); the result is valid in thread 0.
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
