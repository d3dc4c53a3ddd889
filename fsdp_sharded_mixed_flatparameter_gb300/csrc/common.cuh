// common.cuh -- internal helpers of libzeroshard (not part of the C ABI).
//
// Streaming memory operations, exact binary32 arithmetic helpers, launch
// sizing and the per-thread error message shared by the translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "zero_shard.h"

namespace zs {

// ----------------------------------------------------------------- errors
// Record a message for zero_last_error() and return the status.
zero_status fail(zero_status st, const char* fmt, ...);
// Map the launch's cudaGetLastError() to ZERO_OK / ZERO_ECUDA.
zero_status check_launch(const char* what);

// ----------------------------------------------------------- launch sizing
// Every streaming kernel is launched as ONE PASS: one block per tile of work,
// as many blocks as there are tiles, no grid-stride loop.  On GB300 this is
// ~10% faster than a persistent grid of SM count x resident blocks for the
// same kernel (AdamW: 7.19 vs 6.55 TB/s at 6.7B params): the in-order block
// dispatch keeps the set of addresses in flight compact, while persistent
// blocks drift apart and spread their accesses over more DRAM rows.
// Blocks needed to give `per_block` units to each block, at least 1 and
// at most the grid limit (kernels keep a stride loop for anything beyond).
inline unsigned one_pass_blocks(int64_t units, int64_t per_block) {
  int64_t b = (units + per_block - 1) / per_block;
  if (b < 1) b = 1;
  if (b > 0x7fffffffLL) b = 0x7fffffffLL;
  return static_cast<unsigned>(b);
}

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// ----------------------------------------------------------- debug builds
// Built with -DZERO_DEBUG (libzeroshard_debug.so), every global-memory access
// site first checks its index against the extent it must stay in and its
// address against the alignment its vector width needs: ZS_CHECK(cond,
// site, index) is true when the access is valid; otherwise it counts the
// violation, records the first one (site, index, block) and is false, and
// the caller skips the access -- so a bad index is reported instead of
// faulting.  This stands in for a memory checker on GPUs where none runs.
// Device globals are per translation unit (no relocatable device code), so
// each unit defines its record and a host reader with ZS_DEBUG_UNIT(name).
// Release builds compile every check to `true`.
#ifdef ZERO_DEBUG
static __device__ unsigned long long g_zs_debug[4];  // count, first site, first index, first block
static __device__ __noinline__ bool debug_fail(int site, long long index) {
  if (atomicAdd(&g_zs_debug[0], 1ull) == 0ull) {
    g_zs_debug[1] = static_cast<unsigned long long>(site);
    g_zs_debug[2] = static_cast<unsigned long long>(index);
    g_zs_debug[3] = blockIdx.x;
  }
  return false;
}
#define ZS_CHECK(cond, site, index) ((cond) || ::zs::debug_fail((site), static_cast<long long>(index)))
#define ZS_DEBUG_UNIT(name)                                                                        \
  zero_status debug_read_##name(unsigned long long* out, bool reset) {                             \
    if (cudaMemcpyFromSymbol(out, g_zs_debug, sizeof(g_zs_debug)) != cudaSuccess)                  \
      return check_launch("debug record of " #name);                                               \
    if (reset) {                                                                                    \
      const unsigned long long z[4] = {0ull, 0ull, 0ull, 0ull};                                     \
      if (cudaMemcpyToSymbol(g_zs_debug, z, sizeof(z)) != cudaSuccess)                              \
        return check_launch("debug record of " #name);                                             \
    }                                                                                               \
    return ZERO_OK;                                                                                 \
  }
#else
#define ZS_CHECK(cond, site, index) true
#define ZS_DEBUG_UNIT(name)
#endif

__host__ __device__ inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// ------------------------------------------------------ streaming loads
// 32-byte loads/stores (8 x binary32 in one instruction, sm_100+) with
// streaming hints: every byte of the step's buffers is touched once, so
// nothing is worth keeping in L1 or the 129 MB L2.  (Measured on GB300:
// the hints matter far less than the grid shape; see the launchers.)

// read-only input (never written by the kernel): non-coherent path
__device__ __forceinline__ void ld8_ro(const float* p, float (&r)[8]) {
  asm("ld.global.nc.L1::no_allocate.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]), "=f"(r[6]), "=f"(r[7])
      : "l"(p));
}
// state read once then overwritten by the same thread: coherent streaming load
__device__ __forceinline__ void ld8_rw(const float* p, float (&r)[8]) {
  asm volatile("ld.global.cs.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]), "=f"(r[6]), "=f"(r[7])
               : "l"(p));
}
__device__ __forceinline__ void st8(float* p, const float (&r)[8]) {
  asm volatile("st.global.cs.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(r[0]), "f"(r[1]), "f"(r[2]),
               "f"(r[3]), "f"(r[4]), "f"(r[5]), "f"(r[6]), "f"(r[7])
               : "memory");
}
// 16-byte read-only load as four 32-bit words (8 x 16-bit, or 4 x binary32)
__device__ __forceinline__ uint4 ld16_ro(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p));
  return r;
}
__device__ __forceinline__ void st16(void* p, uint4 r) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(r.x),
               "r"(r.y), "r"(r.z), "r"(r.w)
               : "memory");
}

// ----------------------------------------------------------- conversions
// 16-bit floating formats widen exactly to binary32.
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h16) { return __uint_as_float(h16 << 16); }
__device__ __forceinline__ float f16_bits_to_f32(uint32_t h16) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h16)));
}
template <int DT>
__device__ __forceinline__ float half_bits_to_f32(uint32_t h16) {
  return DT == ZERO_BF16 ? bf16_bits_to_f32(h16) : f16_bits_to_f32(h16);
}
// Round two binary32 values to nearest-even 16-bit values packed low|high.
template <int DT>
__device__ __forceinline__ uint32_t pack2_rn(float lo, float hi) {
  if (DT == ZERO_BF16) {
    __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&b);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}
template <int DT>
__device__ __forceinline__ unsigned short round1_rn(float x) {
  if (DT == ZERO_BF16) return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  return __half_as_ushort(__float2half_rn(x));
}

// Element load of a grad of dtype DT at index j (exact widening to binary32).
template <int DT>
__device__ __forceinline__ float load_elem(const void* base, int64_t j) {
  if (DT == ZERO_F32) return __ldg(static_cast<const float*>(base) + j);
  const unsigned short h = __ldg(static_cast<const unsigned short*>(base) + j);
  return half_bits_to_f32<DT>(h);
}

__device__ __forceinline__ bool finite_f(float x) { return (__float_as_uint(x) & 0x7f800000u) != 0x7f800000u; }

}  // namespace zs
