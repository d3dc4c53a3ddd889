// table.cuh -- reading grads through the FlatParameter tensor table:
// locating the tensor that holds a flat index, 8-element vector loads of a
// grad source (aligned, or realigned in registers), and staging a range of
// the flat buffer into shared memory with loads aligned to each SOURCE
// tensor.  Shared by the flatten kernel and the AdamW kernel that reads
// grads straight from the table.  Internal.
#pragma once

#include "common.cuh"

namespace zs {

constexpr int kFlThreads = 256;
constexpr int kFlTile = 8192;
constexpr int kFlStage = kFlTile + kFlTile / 8;

__device__ __forceinline__ int stage_idx(int q) { return q + (q >> 3); }

// last i with table[i].flat_offset <= k (the tensor that holds flat index k)
__device__ __forceinline__ int find_tensor(const zero_tensor* __restrict__ table, int n, int64_t k) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(&table[mid].flat_offset) <= k)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// find_tensor by a warp at once: the 32 lanes test 32 evenly spaced
// candidates per round and __ballot_sync picks the segment that holds k, so
// n tensors take ceil(log32 n) rounds of independent loads (2 for the 291 of
// Llama-7B, 3 for 20,000) instead of log2 n dependent ones.  Every lane of
// the warp must call it; all get the same index, the binary search's.
__device__ __forceinline__ int find_tensor_warp(const zero_tensor* __restrict__ table, int n, int64_t k) {
  const int lane = threadIdx.x & 31;
  int lo = 0, span = n;  // invariant: table[lo].flat_offset <= k, the answer is in [lo, lo + span)
  while (span > 1) {
    const int step = (span + 31) >> 5;
    const int off = lane * step;
    const bool le = off < span && __ldg(&table[lo + off].flat_offset) <= k;
    const unsigned mask = __ballot_sync(0xffffffffu, le);  // a prefix of the lanes (offsets ascend)
    const int j = 31 - __clz(mask);
    lo += j * step;
    span = (span - j * step < step) ? span - j * step : step;
  }
  return lo;
}

template <int DT>
struct SrcTraits {
  static constexpr int esize = (DT == ZERO_F32) ? 4 : 2;
};

// 8 consecutive source elements starting at a 32-byte (f32) or 16-byte
// (16-bit) aligned address, widened to binary32.
template <int DT>
__device__ __forceinline__ void load8_src(const void* p, float (&x)[8]) {
  if (DT == ZERO_F32) {
    ld8_ro(static_cast<const float*>(p), x);
  } else {
    const uint4 w = ld16_ro(p);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[2 * j] = half_bits_to_f32<DT>(ws[j] & 0xffffu);
      x[2 * j + 1] = half_bits_to_f32<DT>(ws[j] >> 16);
    }
  }
}

// Words m .. m+4 of the 8 words a:b (m block-uniform, 0..3), shifted right by
// sh = 0 or 16 bits across word boundaries: the 8 16-bit values that start
// 2*m + sh/16 values into a:b.
__device__ __forceinline__ uint4 realign16(uint4 a, uint4 b, int m, unsigned sh) {
  uint32_t q0, q1, q2, q3, q4;
  switch (m) {
    case 0: q0 = a.x; q1 = a.y; q2 = a.z; q3 = a.w; q4 = b.x; break;
    case 1: q0 = a.y; q1 = a.z; q2 = a.w; q3 = b.x; q4 = b.y; break;
    case 2: q0 = a.z; q1 = a.w; q2 = b.x; q3 = b.y; q4 = b.z; break;
    default: q0 = a.w; q1 = b.x; q2 = b.y; q3 = b.z; q4 = b.w; break;
  }
  return make_uint4(__funnelshift_r(q0, q1, sh), __funnelshift_r(q1, q2, sh), __funnelshift_r(q2, q3, sh),
                    __funnelshift_r(q3, q4, sh));
}

// R groups of 8 per thread (groups t + 256 r of a block of 256 threads) from
// a 16-bit source `src` that is element- but not 16-byte aligned: every
// thread loads the aligned 16-byte vector under its group, takes the next
// vector from the neighbouring lane (lane 31 loads it: it is the next
// warp's), and cuts its 8 values out of the pair in registers -- no
// shared-memory staging.  The vectors read reach up to 7 values before src
// and after the last group's end; the caller guarantees both lie inside the
// tensor.  Every lane of each warp must call it (warp shuffles).
template <int DT, int R>
__device__ __forceinline__ void load8_shifted(const char* src, float (&x)[R][8]) {
  const uintptr_t mis = reinterpret_cast<uintptr_t>(src) % 16;  // 2, 4, ..., 14
  const char* abase = src - mis;
  const int m = static_cast<int>(mis >> 2);
  const unsigned sh = static_cast<unsigned>(mis & 2u) * 8u;
  const int lane = threadIdx.x & 31;
  uint4 w[R], nx[R];
#pragma unroll
  for (int r = 0; r < R; ++r) w[r] = ld16_ro(abase + 16 * (threadIdx.x + r * kFlThreads));
#pragma unroll
  for (int r = 0; r < R; ++r) {
    nx[r] = make_uint4(0u, 0u, 0u, 0u);
    if (lane == 31) nx[r] = ld16_ro(abase + 16 * (threadIdx.x + r * kFlThreads + 1));
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const uint4 d = make_uint4(__shfl_down_sync(0xffffffffu, w[r].x, 1), __shfl_down_sync(0xffffffffu, w[r].y, 1),
                               __shfl_down_sync(0xffffffffu, w[r].z, 1), __shfl_down_sync(0xffffffffu, w[r].w, 1));
    if (lane != 31) nx[r] = d;
    const uint4 o = realign16(w[r], nx[r], m, sh);
    const uint32_t ws[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[r][2 * j] = half_bits_to_f32<DT>(ws[j] & 0xffffu);
      x[r][2 * j + 1] = half_bits_to_f32<DT>(ws[j] >> 16);
    }
  }
}

// Write fl(scale * x) of source elements [j0, j0 + len) into stage[q0 ...);
// qcap: the staged tile's length (q0 + len <= qcap).
template <int DT>
__device__ __forceinline__ void stage_segment(const void* __restrict__ src, int64_t j0, int len, int q0, int qcap,
                                              float scale, float* stage, bool& bad) {
  if (!ZS_CHECK(q0 >= 0 && len >= 0 && q0 + len <= qcap && j0 >= 0, 40, q0)) return;
  if (src == nullptr) {
    const float y = __fmul_rn(scale, 0.0f);
    for (int e = threadIdx.x; e < len; e += kFlThreads) stage[stage_idx(q0 + e)] = y;
    return;
  }
  constexpr int es = SrcTraits<DT>::esize;
  constexpr int vb = (DT == ZERO_F32) ? 32 : 16;  // bytes of one 8-element source vector
  const char* sp = static_cast<const char*>(src) + es * j0;
  int h = static_cast<int>(((vb - reinterpret_cast<uintptr_t>(sp) % vb) % vb) / es);
  if (h > len) h = len;
  const int nv = (len - h) / 8;
  const int body_end = h + 8 * nv;
  for (int e = threadIdx.x; e < h; e += kFlThreads) {
    const float y = __fmul_rn(scale, load_elem<DT>(src, j0 + e));
    bad |= !finite_f(y);
    stage[stage_idx(q0 + e)] = y;
  }
  // body: four source vectors in flight per thread (loads first), then one at a time
  int vi = threadIdx.x;
  for (; vi + 3 * kFlThreads < nv; vi += 4 * kFlThreads) {
    if (!ZS_CHECK(aligned(sp + es * (h + 8 * vi), vb) && h + 8 * (vi + 3 * kFlThreads) + 8 <= len, 41, vi)) continue;
    float x[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u) load8_src<DT>(sp + es * (h + 8 * (vi + u * kFlThreads)), x[u]);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int q = q0 + h + 8 * (vi + u * kFlThreads);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float y = __fmul_rn(scale, x[u][i]);
        bad |= !finite_f(y);
        stage[stage_idx(q + i)] = y;
      }
    }
  }
  for (; vi < nv; vi += kFlThreads) {
    if (!ZS_CHECK(aligned(sp + es * (h + 8 * vi), vb) && h + 8 * vi + 8 <= len, 42, vi)) continue;
    float x[8];
    load8_src<DT>(sp + es * (h + 8 * vi), x);
    const int q = q0 + h + 8 * vi;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float y = __fmul_rn(scale, x[i]);
      bad |= !finite_f(y);
      stage[stage_idx(q + i)] = y;
    }
  }
  for (int e = body_end + threadIdx.x; e < len; e += kFlThreads) {
    const float y = __fmul_rn(scale, load_elem<DT>(src, j0 + e));
    bad |= !finite_f(y);
    stage[stage_idx(q0 + e)] = y;
  }
}

// Stage fl(scale * x) of the flat range [klo, khi) into stage[0, khi - klo):
// walk the tensors from ti (the one holding klo) forward, each segment read
// with loads aligned to its source; whatever the table does not cover reads
// as zeros.  Every thread of the block must call it (the caller syncs).
template <int DT>
__device__ __forceinline__ void stage_range(const zero_tensor* __restrict__ table, int n_tensors, int ti, int64_t klo,
                                            int64_t khi, float scale, float* stage, bool& bad) {
  int64_t k = klo;
  int j = ti;
  while (k < khi && j < n_tensors) {
    const int64_t off = __ldg(&table[j].flat_offset), num = __ldg(&table[j].numel);
    const int64_t seg_end = (off + num < khi) ? off + num : khi;
    if (seg_end > k) {
      stage_segment<DT>(table[j].ptr, k - off, static_cast<int>(seg_end - k), static_cast<int>(k - klo),
                        static_cast<int>(khi - klo), scale, stage, bad);
      k = seg_end;
    }
    ++j;
  }
  const int tlen = static_cast<int>(khi - klo);
  for (int q = static_cast<int>(k - klo) + threadIdx.x; q < tlen; q += kFlThreads) stage[stage_idx(q)] = 0.0f;
}

}  // namespace zs
