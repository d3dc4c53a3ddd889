// sqnorm.cu -- deterministic global L2 grad norm and clip coefficient.
//
// clip_grad_norm_ as the ZeRO page's training loop (section "组合策略") and
// the LLaMA-13B gradient-accumulation page call it, in two launches:
//
//  1. sqnorm_tiles_kernel: the grad buffer is cut into fixed tiles of
//     kSqTile = 32768 elements.  A block reduces one tile at a time: each of
//     its 256 threads takes 128 elements (16 x 32-byte loads, two rounds of
//     eight) and adds their squares into two double-float accumulators
//     (unevaluated sums h + l of two binary32 values, even and odd elements,
//     updated together by packed f32x2 instructions): every square is split
//     exactly into x*x = p + e with one fma, p is added to h with an
//     error-free TwoSum, and the two error terms go into l (reduce.cuh).  The
//     256 thread sums are added in double-float by a fixed shuffle/shared-
//     memory tree and the tile's partial is stored rounded to binary64.  One
//     block per tile (the grid loop
//     only covers grids beyond the hardware limit), so the partial of a tile
//     does not depend on which block computed it or how many blocks ran.
//  2. sqnorm_finalize_kernel: a cluster of 8 blocks adds the partials in a
//     fixed order (binary64), adds the other ranks' share, takes the square
//     root and the clip coefficient, and writes the zero_norm_result.
//
// Accuracy: the double-float sums carry about 48 significant bits, so the
// relative error of the sum of squares is ~1e-14 (binary64 beyond the
// tile level), about as good as the compensated binary64 sum of the CPU
// oracle.  (The accumulation order and helpers live in reduce.cuh, shared
// with the kernels that fuse the norm into their pass.)  That is what makes the binary32 clip coefficient -- and with it
// the whole AdamW step -- agree bit for bit with the oracle in practice: a
// coarser norm would move the coefficient by an ulp now and then, and where
// p*(1-lr*wd) and the Adam update nearly cancel, that ulp is a large
// relative error of the new parameter.  The extra arithmetic (~5 packed
// instructions per element) hides under the 4 bytes/element memory stream.
// Limits: squares outside the binary32 range (|g| >= 2^64 overflows to a
// non-finite norm, |g| < 2^-75 underflows toward 0) are where the result can
// differ from the binary64 oracle; gradients never come near either.
// No atomics: the result is bit-identical from run to run and GPU to GPU.
#include <cooperative_groups.h>
#include <cuda.h>

#include <cmath>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "reduce.cuh"

namespace zs {

namespace cg = cooperative_groups;


// Element e of a tile belongs to thread t, vector slot r, lane i where
// e = ((r * 256) + t) * 8 + i: each 32-byte load of a warp covers 1 KiB.
// The thread adds its 128 squares in that (r, i) order.
template <bool VEC>
__device__ __forceinline__ NormAcc thread_tile_sum(const float* __restrict__ g, int64_t base, int64_t n) {
  NormAcc acc;
#pragma unroll
  for (int round = 0; round < 2; ++round) {
    float x[8][8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const int64_t e = base + ((static_cast<int64_t>(round * 8 + r) * kSqThreads) + threadIdx.x) * 8;
      if (VEC) {
        if (ZS_CHECK(e + 8 <= n && aligned(g + e, 32), 30, e)) {
          ld8_ro(g + e, x[r]);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) x[r][i] = 0.0f;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) x[r][i] = (e + i < n) ? __ldg(g + e + i) : 0.0f;
      }
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) acc.add8(x[r]);  // out-of-range elements are 0 and add nothing
  }
  return acc;
}

__global__ void __launch_bounds__(kSqThreads) sqnorm_tiles_kernel(const float* __restrict__ g, int64_t n,
                                                                  int64_t ntiles, bool vec_ok,
                                                                  double* __restrict__ partials) {
  __shared__ float2 red[kSqThreads / 32];
  for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    const int64_t base = tile * kSqTile;
    const NormAcc ts = (vec_ok && base + kSqTile <= n) ? thread_tile_sum<true>(g, base, n)
                                                       : thread_tile_sum<false>(g, base, n);
    const double bs = block_sum_norm<kSqThreads>(ts, red);
    if (threadIdx.x == 0 && ZS_CHECK(tile < ntiles, 31, tile)) partials[tile] = bs;
  }
}

constexpr int kFinThreads = 1024;
constexpr int kFinCluster = 8;  // blocks of the finalize (a portable cluster size)

// The finalize over the tile partials runs as one thread-block cluster of 8
// blocks on 8 SMs: binary64 runs at a small fraction of the binary32 rate on
// GB300, and one SM's binary64 pipe alone took ~66 us for Llama-7B's 205,641
// partials.  Block r adds the contiguous chunk r of the partials (thread
// stride, then block_sum); after the cluster barrier block 0 reads the 8
// block totals from the other blocks' shared memory (distributed shared
// memory) in rank order and writes the result; a second barrier keeps every
// block's shared memory alive until then.  The order depends on ntiles only.
__global__ void __cluster_dims__(kFinCluster, 1, 1) __launch_bounds__(kFinThreads)
    sqnorm_finalize_kernel(const double* __restrict__ partials, int64_t ntiles, double extra_sqnorm,
                           double max_norm, zero_norm_result* __restrict__ out) {
  __shared__ double red[kFinThreads / 32];
  __shared__ double block_total;
  cg::cluster_group cluster = cg::this_cluster();
  const int64_t r = cluster.block_rank();
  const int64_t chunk = (ntiles + kFinCluster - 1) / kFinCluster;
  const int64_t lo = r * chunk, hi = (lo + chunk < ntiles) ? lo + chunk : ntiles;
  double acc = 0.0;
  for (int64_t j = lo + threadIdx.x; j < hi; j += kFinThreads) acc += partials[j];
  const double local = block_sum<kFinThreads>(acc, red);
  if (threadIdx.x == 0) block_total = local;
  cluster.sync();
  if (r == 0 && threadIdx.x == 0) {
    double total = 0.0;
    for (int i = 0; i < kFinCluster; ++i) total += *cluster.map_shared_rank(&block_total, i);
    const double sq = total + extra_sqnorm;
    const double norm = __dsqrt_rn(sq);
    const double q = __ddiv_rn(max_norm, __dadd_rn(norm, 1e-6));
    zero_norm_result res;
    res.sqnorm = sq;
    res.norm = norm;
    res.clip_coef = (q < 1.0) ? __double2float_rn(q) : 1.0f;
    res.finite = isfinite(norm) ? 1 : 0;
    *out = res;
  }
  cluster.sync();
}

// Global norm from the ranks' local sums of squares, added in rank order by
// one thread so that every rank derives the same binary64 total and the same
// binary32 coefficient from the same gathered vector.
__global__ void sqnorm_combine_kernel(const double* __restrict__ sq, int n_parts, double max_norm,
                                      zero_norm_result* __restrict__ out) {
  if (threadIdx.x != 0 || blockIdx.x != 0) return;
  double total = 0.0;
  for (int i = 0; i < n_parts; ++i) total = __dadd_rn(total, sq[i]);
  const double norm = __dsqrt_rn(total);
  const double q = __ddiv_rn(max_norm, __dadd_rn(norm, 1e-6));
  zero_norm_result r;
  r.sqnorm = total;
  r.norm = norm;
  r.clip_coef = (q < 1.0) ? __double2float_rn(q) : 1.0f;
  r.finite = isfinite(norm) ? 1 : 0;
  *out = r;
}

ZS_DEBUG_UNIT(sqnorm)

zero_status launch_sqnorm_combine(const double* sq, int n_parts, double max_norm, zero_norm_result* out,
                                  cudaStream_t st) {
  sqnorm_combine_kernel<<<1, 32, 0, st>>>(sq, n_parts, max_norm, out);
  return check_launch("sqnorm_combine_kernel");
}

zero_status launch_sqnorm_finalize(const double* partials, int64_t n, double extra_sqnorm, double max_norm,
                                   zero_norm_result* out, cudaStream_t st) {
  const int64_t ntiles = (n + kSqTile - 1) / kSqTile;
  sqnorm_finalize_kernel<<<kFinCluster, kFinThreads, 0, st>>>(partials, ntiles, extra_sqnorm, max_norm, out);
  return check_launch("sqnorm_finalize_kernel");
}

zero_status launch_sqnorm(const float* g, int64_t n, double extra_sqnorm, double max_norm, double* partials,
                          zero_norm_result* out, cudaStream_t st) {
  const int64_t ntiles = (n + kSqTile - 1) / kSqTile;
  if (ntiles > 0) {
    sqnorm_tiles_kernel<<<one_pass_blocks(ntiles, 1), kSqThreads, 0, st>>>(g, n, ntiles, aligned(g, 32), partials);
    zero_status s = check_launch("sqnorm_tiles_kernel");
    if (s != ZERO_OK) return s;
  }
  sqnorm_finalize_kernel<<<kFinCluster, kFinThreads, 0, st>>>(partials, ntiles, extra_sqnorm, max_norm, out);
  return check_launch("sqnorm_finalize_kernel");
}

// ---------------------------------------------------------------------------
// zero_grad_sqnorm_noalloc: the same grad-norm computation for callers that
// cannot allocate device memory.  The tile partials live in a fixed array in
// this library's own device memory instead of a caller-provided workspace.
// The array is a module global: every GPU that loads the library holds its
// 4 MiB until the process exits.  In host code `g_noalloc_partials` is only a
// host-side stand-in for the symbol, never a device address; the device
// address is looked up with cudaGetSymbolAddress once per device and
// context, with that device current.  The cache is keyed on the context's
// process-unique ID (cuCtxGetId, reached through the runtime's driver entry
// point, so the library does not link libcuda): after cudaDeviceReset the
// runtime creates a new primary context, which loads the module again and
// may place the array elsewhere, and the next call looks it up again.

constexpr int64_t kNoAllocMaxTiles = int64_t(1) << 19;  // 4 MiB of binary64 partials

static __device__ __align__(256) double g_noalloc_partials[kNoAllocMaxTiles];

namespace {
constexpr int kMaxDevices = 256;
std::mutex g_noalloc_mu;
struct NoAllocSlot {
  unsigned long long ctx_id;  // ID of the context the address belongs to (0: none yet)
  void* addr;
};
NoAllocSlot g_noalloc_slot[kMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// The current context's process-unique ID.  Before the runtime has made any
// context current (the process's first CUDA work) the handle is null and an
// error comes back; the caller then looks the address up without caching it,
// which also initialises the context for the next call.
cudaError_t current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  if (get_current == nullptr || get_id == nullptr) {
    cudaDriverEntryPointQueryResult q1 = cudaDriverEntryPointSymbolNotFound, q2 = cudaDriverEntryPointSymbolNotFound;
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaError_t e1 = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1);
    if (e1 != cudaSuccess) return e1;
    cudaError_t e2 = cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2);
    if (e2 != cudaSuccess) return e2;
    if (q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || !f1 || !f2)
      return cudaErrorSymbolNotFound;
    get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
    get_id = reinterpret_cast<CtxGetIdFn>(f2);
  }
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
  if (get_id(ctx, id) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  return cudaSuccess;
}
}  // namespace

}  // namespace zs

extern "C" zero_status zero_grad_sqnorm_noalloc(const float* d_grad, int64_t n, double extra_sqnorm,
                                                double max_norm, zero_norm_result* d_out, void* stream) {
  using zs::fail;
  if (n < 0) return fail(ZERO_EINVAL, "zero_grad_sqnorm_noalloc: n %lld < 0", (long long)n);
  if (n > zs::kNoAllocMaxTiles * zs::kSqTile)
    return fail(ZERO_EINVAL,
                "zero_grad_sqnorm_noalloc: n = %lld exceeds the built-in scratch limit of %lld elements "
                "(%lld tiles of %lld); use zero_grad_sqnorm with a caller workspace",
                (long long)n, (long long)(zs::kNoAllocMaxTiles * zs::kSqTile), (long long)zs::kNoAllocMaxTiles,
                (long long)zs::kSqTile);
  if (n > 0 && d_grad == nullptr) return fail(ZERO_EINVAL, "zero_grad_sqnorm_noalloc: NULL d_grad");
  if (d_out == nullptr) return fail(ZERO_EINVAL, "zero_grad_sqnorm_noalloc: NULL d_out");
  if (std::isnan(max_norm) || max_norm < 0.0) return fail(ZERO_EINVAL, "zero_grad_sqnorm_noalloc: bad max_norm");
  if (!std::isfinite(extra_sqnorm) || extra_sqnorm < 0.0)
    return fail(ZERO_EINVAL, "zero_grad_sqnorm_noalloc: bad extra_sqnorm");
  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return fail(ZERO_ECUDA, "zero_grad_sqnorm_noalloc: cudaGetDevice: %s", cudaGetErrorString(ce));
  if (dev < 0 || dev >= zs::kMaxDevices) return fail(ZERO_EINVAL, "zero_grad_sqnorm_noalloc: device %d", dev);
  void* scratch = nullptr;
  {
    // once per device and context, with that device current: find the array's device address
    std::lock_guard<std::mutex> lk(zs::g_noalloc_mu);
    unsigned long long ctx_id = 0;
    zs::NoAllocSlot& slot = zs::g_noalloc_slot[dev];
    ce = zs::current_context_id(&ctx_id);
    if (ce != cudaSuccess || ctx_id == 0) {
      // no usable context ID: look the address up on every call (always correct, a little slower)
      void* p = nullptr;
      ce = cudaGetSymbolAddress(&p, zs::g_noalloc_partials);
      if (ce != cudaSuccess || p == nullptr)
        return fail(ZERO_ECUDA, "zero_grad_sqnorm_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(ce));
      scratch = p;
    } else {
      if (slot.addr == nullptr || slot.ctx_id != ctx_id) {
        void* p = nullptr;
        ce = cudaGetSymbolAddress(&p, zs::g_noalloc_partials);
        if (ce != cudaSuccess || p == nullptr)
          return fail(ZERO_ECUDA, "zero_grad_sqnorm_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(ce));
        slot.addr = p;
        slot.ctx_id = ctx_id;
      }
      scratch = slot.addr;
    }
  }
  return zs::launch_sqnorm(d_grad, n, extra_sqnorm, max_norm, static_cast<double*>(scratch), d_out,
                           zs::as_stream(stream));
}
