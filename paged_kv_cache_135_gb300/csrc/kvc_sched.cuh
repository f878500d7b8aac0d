// Work partition shared by the persistent attention kernels: every
// (sequence, head group, 64-token tile) unit in one linear order, split into
// P equal contiguous shares (stream-K); helpers to walk a share and to find
// the owner of a unit.
#pragma once

#include <stdint.h>

#include "kvc_device.cuh"

namespace kvc {
namespace sched {

__device__ __forceinline__ int clamp_len(int L, int cap, uint32_t* err_flag) {
  if (L < 0 || L > cap) {
    set_flag(err_flag, KVC_FLAG_LEN_RANGE);
    return L < 0 ? 0 : cap;
  }
  return L;
}

// Owner of unit x when N units are split over P shares, share c taking
// [c*N/P, (c+1)*N/P): the largest c whose start is <= x.
__device__ __forceinline__ int share_of(long long x, long long N, int P) {
  return static_cast<int>(((x + 1) * P + N - 1) / N - 1);
}
__device__ __forceinline__ long long share_begin(int c, long long N, int P) {
  return static_cast<long long>(c) * N / P;
}

// Walks the linear unit list (b, g, j) in order; cum[b] = units of the
// sequences before b for one head group, hg head groups per sequence.
struct Cursor {
  int b, g, j, n;
  __device__ __forceinline__ void locate(long long t, const int* cum, int batch, int hg) {
    int lo = 0, hi = batch - 1;  // largest b with hg*cum[b] <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (static_cast<long long>(hg) * cum[mid] <= t) lo = mid; else hi = mid - 1;
    }
    b = lo;
    n = cum[b + 1] - cum[b];
    const long long r = t - static_cast<long long>(hg) * cum[b];
    g = static_cast<int>(r / n);
    j = static_cast<int>(r - static_cast<long long>(g) * n);
  }
  __device__ __forceinline__ void advance(const int* cum, int batch, int hg) {
    if (++j < n) return;
    j = 0;
    if (++g < hg) return;
    g = 0;
    do {
      ++b;
    } while (b < batch && cum[b + 1] == cum[b]);
    if (b < batch) n = cum[b + 1] - cum[b];
  }
};

// Clamped lengths and the exclusive prefix sum of ceil(len / tile) for B
// sequences, computed by the calling warp into shared memory (cum[B] = total).
// With extra > 0 every sequence with at least one tile counts extra more
// units (work-split weights that stand for a sequence's fixed costs).
__device__ __forceinline__ void plan_tiles(const int* lens, int* cum, int B, int tile,
                                           int lane, int extra = 0) {
  int carry = 0;
  for (int base = 0; base < B; base += 32) {
    const int i = base + lane;
    const int t = i < B ? (lens[i] + tile - 1) / tile : 0;
    const int n = t > 0 ? t + extra : 0;
    int x = n;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (i < B) cum[i] = carry + x - n;
    carry += __shfl_sync(0xffffffffu, x, 31);
  }
  if (lane == 0) cum[B] = carry;
}

}  // namespace sched
}  // namespace kvc
