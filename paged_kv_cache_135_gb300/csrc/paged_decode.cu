// Paged decode attention with split-KV (rows a3 and a4 of the hot path).
//
// What it computes: "external-cannbot-model-model-infer-kvcache" Mode 2 --
// one query token per sequence attends to the sequence's cached K/V, read
// through block_table from the ND cache [num_blocks, block_size, Hkv, D],
// with per-sequence actual KV lengths and GQA head groups (sparse_mode 0,
// Appendix C).  The kernel's inner loop walks the sequence's physical
// blocks, as the hotelren.com notes "Paged KV Cache + Packed Sequence" 4.2
// describe for paged attention kernels.
//
// GB300 design (not on the pages):
//  * Work unit = a 64-token tile of one (sequence b, kv head g) segment.
//    All tiles of all segments form one linear list ordered (b, g, tile);
//    each of the P persistent CTAs takes one contiguous 1/P share of it
//    ("stream-K" split-KV), so every SM streams the same number of bytes
//    whatever the length mix.  A segment cut by a share boundary leaves
//    per-CTA partial softmax states (m, l, unnormalised O) in the workspace;
//    a second kernel merges them in a fixed order (deterministic, and
//    independent of physical block IDs).
//  * One producer warp gathers tiles with TMA: per tile and per K/V half
//    (64 head-dim elements = 128 B rows) one 4-D box {64, 1, min(bs,64), 1}
//    per physical block at coordinate (d0, g, token-in-block, block id), into
//    a 3-stage mbarrier ring, 128-byte swizzled.  The block_table entry is the
//    box's block coordinate, so the gather costs no address arithmetic per
//    row.  Physical blocks never fetched past a sequence's length.
//  * Four consumer warps each take 16 tokens of a stage.  The GQA query
//    group (G = Hq/Hkv heads, zero-padded to 16 rows) is the M side of
//    mma.sync m16n8k16 (QK^T with K from ldmatrix, then P.V with V from
//    ldmatrix.trans), fp32 accumulation, online softmax in the log2 domain
//    with quad shuffles, P rounded to the input type and l summed from the
//    rounded P so that normalisation matches the weights actually applied.
//  * Rows of a partial tile past the sequence length are masked in S (-inf)
//    and zeroed in V, so stale or non-finite cache contents cannot leak.
#include <cuda_runtime.h>

#include <math.h>

#include <map>
#include <mutex>
#include <utility>

#include "kvc_device.cuh"
#include "kvc_host.h"

namespace kvc {

namespace {

constexpr int kTile = 64;            // tokens per pipeline stage
constexpr int kConsumerWarps = 4;    // 16 tokens each
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 3;
constexpr int kMaxBatch = 1024;
constexpr int kHalfBytes = kTile * 128;  // one 64-element half of a K or V tile

struct DecodeParams {
  const void* q;
  void* out;
  const int32_t* block_table;
  const int32_t* seq_lens;
  float* ws_o;   // [P][2][G][D] unnormalised partial outputs
  float* ws_ml;  // [P][2][G][2] partial (max, sum) in the log2 domain
  uint32_t* err_flag;
  int batch, num_q_heads, num_kv_heads, group, head_dim;
  int block_size, log2_bs, max_blocks, num_blocks, box_tokens;
  float scale_log2;
};

template <int D>
struct Layout {
  static constexpr int kHalves = D / 64;
  static constexpr int kKBytes = kHalves * kHalfBytes;
  static constexpr int kStageBytes = 2 * kKBytes;  // K tile then V tile
  static constexpr int kBarOff = kStages * kStageBytes;
  static constexpr int kAbortOff = kBarOff + 2 * kStages * 8;
  static constexpr int kLensOff = kBarOff + 128;
  // lens[batch], cum[batch + 1], then the cross-warp combine buffers.
  __host__ __device__ static int cum_off(int batch) { return kLensOff + ((batch + 3) & ~3) * 4; }
  __host__ __device__ static int cmb_off(int batch) {
    return cum_off(batch) + ((batch + 1 + 3) & ~3) * 4;
  }
  static size_t bytes(int batch, int group) {
    return 1024 /*alignment slack*/ + cmb_off(batch) +
           static_cast<size_t>(kConsumerWarps) * group * (D + 2) * 4;
  }
};

__device__ __forceinline__ int clamp_len(int L, int cap, uint32_t* err_flag) {
  if (L < 0 || L > cap) {
    set_flag(err_flag, KVC_FLAG_LEN_RANGE);
    return L < 0 ? 0 : cap;
  }
  return L;
}

// Owner of linear tile x when N tiles are split over P CTAs with CTA c taking
// [c*N/P, (c+1)*N/P): the largest c whose start is <= x.
__device__ __forceinline__ int cta_of(long long x, long long N, int P) {
  return static_cast<int>(((x + 1) * P + N - 1) / N - 1);
}
__device__ __forceinline__ long long tile_begin(int c, long long N, int P) {
  return static_cast<long long>(c) * N / P;
}

// Walks the linear tile list (b, g, j) in order.
struct Cursor {
  int b, g, j, n;
  __device__ __forceinline__ void locate(long long t, const int* cum, int batch, int hkv) {
    int lo = 0, hi = batch - 1;  // largest b with hkv*cum[b] <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (static_cast<long long>(hkv) * cum[mid] <= t) lo = mid; else hi = mid - 1;
    }
    b = lo;
    n = cum[b + 1] - cum[b];
    const long long r = t - static_cast<long long>(hkv) * cum[b];
    g = static_cast<int>(r / n);
    j = static_cast<int>(r - static_cast<long long>(g) * n);
  }
  __device__ __forceinline__ void advance(const int* cum, int batch, int hkv) {
    if (++j < n) return;
    j = 0;
    if (++g < hkv) return;
    g = 0;
    do {
      ++b;
    } while (b < batch && cum[b + 1] == cum[b]);
    if (b < batch) n = cum[b + 1] - cum[b];
  }
};

// Load the G query rows of (b, g) as mma A fragments (rows >= G are zero).
template <typename T, int D>
__device__ __forceinline__ void load_q(const T* __restrict__ q, const DecodeParams& p, int b,
                                       int g, int lane, uint32_t (&qa)[D / 16][4]) {
  const T* base = q + (static_cast<long long>(b) * p.num_q_heads + g * p.group) * D;
  const int r0 = lane >> 2, c = 2 * (lane & 3);
  const bool v0 = r0 < p.group, v1 = r0 + 8 < p.group;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const int col = kk * 16 + c;
    qa[kk][0] = v0 ? *reinterpret_cast<const uint32_t*>(base + r0 * D + col) : 0u;
    qa[kk][1] = v1 ? *reinterpret_cast<const uint32_t*>(base + (r0 + 8) * D + col) : 0u;
    qa[kk][2] = v0 ? *reinterpret_cast<const uint32_t*>(base + r0 * D + col + 8) : 0u;
    qa[kk][3] = v1 ? *reinterpret_cast<const uint32_t*>(base + (r0 + 8) * D + col + 8) : 0u;
  }
}

__device__ __forceinline__ uint32_t keep_rows(uint32_t x, int k, int valid) {
  const uint32_t lo = k < valid ? 0x0000FFFFu : 0u;
  const uint32_t hi = k + 1 < valid ? 0xFFFF0000u : 0u;
  return x & (lo | hi);
}

// One warp's 16 tokens of a stage: S = Q K^T, online softmax, O += P V.
template <typename T, int D>
__device__ __forceinline__ void attend_16(uint32_t kbase, uint32_t vbase, int warp, int lane,
                                          int valid, float scale_log2,
                                          const uint32_t (&qa)[D / 16][4], float (&o)[D / 8][4],
                                          float (&m)[2], float (&l)[2]) {
  const int mi = lane >> 3, rr = lane & 7;
  float s[2][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) s[i][e] = 0.f;
  {
    const int tok = warp * 16 + (mi >> 1) * 8 + rr;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int dcol = kk * 16 + (mi & 1) * 8;
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kbase + (dcol >> 6) * kHalfBytes + swz128(tok, (dcol & 63) >> 3), b0, b1, b2, b3);
      MmaOp<T>::run(s[0], qa[kk], b0, b1);
      MmaOp<T>::run(s[1], qa[kk], b2, b3);
    }
  }
  const int c0 = 2 * (lane & 3);
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int k = nt * 8 + c0 + (e & 1);
      s[nt][e] = k < valid ? s[nt][e] * scale_log2 : -INFINITY;
    }
  float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
  float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
  const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
  const float corr0 = fast_exp2(m[0] - mn0), corr1 = fast_exp2(m[1] - mn1);
  m[0] = mn0;
  m[1] = mn1;
  uint32_t pa[4];
  float rs0 = 0.f, rs1 = 0.f, ra, rb;
  pa[0] = Pack<T>::run(fast_exp2(s[0][0] - mn0), fast_exp2(s[0][1] - mn0), ra, rb);
  rs0 += ra + rb;
  pa[1] = Pack<T>::run(fast_exp2(s[0][2] - mn1), fast_exp2(s[0][3] - mn1), ra, rb);
  rs1 += ra + rb;
  pa[2] = Pack<T>::run(fast_exp2(s[1][0] - mn0), fast_exp2(s[1][1] - mn0), ra, rb);
  rs0 += ra + rb;
  pa[3] = Pack<T>::run(fast_exp2(s[1][2] - mn1), fast_exp2(s[1][3] - mn1), ra, rb);
  rs1 += ra + rb;
  l[0] = l[0] * corr0 + rs0;
  l[1] = l[1] * corr1 + rs1;
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
    o[n][0] *= corr0;
    o[n][1] *= corr0;
    o[n][2] *= corr1;
    o[n][3] *= corr1;
  }
  const int tok = warp * 16 + (mi & 1) * 8 + rr;
#pragma unroll
  for (int dp = 0; dp < D / 16; ++dp) {
    const int dcol = dp * 16 + (mi >> 1) * 8;
    uint32_t b0, b1, b2, b3;
    ldsm_x4_t(vbase + (dcol >> 6) * kHalfBytes + swz128(tok, (dcol & 63) >> 3), b0, b1, b2, b3);
    if (valid < 16) {
      b0 = keep_rows(b0, c0, valid);
      b1 = keep_rows(b1, 8 + c0, valid);
      b2 = keep_rows(b2, c0, valid);
      b3 = keep_rows(b3, 8 + c0, valid);
    }
    MmaOp<T>::run(o[2 * dp], pa, b0, b1);
    MmaOp<T>::run(o[2 * dp + 1], pa, b2, b3);
  }
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 2)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* empty = full + kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbortOff);
  int* lens = reinterpret_cast<int*>(smem + L::kLensOff);
  int* cum = reinterpret_cast<int*>(smem + L::cum_off(p.batch));
  float* cmb_m = reinterpret_cast<float*>(smem + L::cmb_off(p.batch));
  float* cmb_l = cmb_m + kConsumerWarps * p.group;
  float* cmb_o = cmb_l + kConsumerWarps * p.group;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int B = p.batch, hkv = p.num_kv_heads, G = p.group;
  const int cap = p.max_blocks * p.block_size;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kConsumerWarps && lane == 0) {
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  // Plan: clamped lengths and the prefix sum of 64-token tiles per sequence.
  for (int i = tid; i < B; i += kThreads) lens[i] = clamp_len(p.seq_lens[i], cap, p.err_flag);
  __syncthreads();
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < B; base += 32) {
      const int i = base + lane;
      const int n = i < B ? (lens[i] + kTile - 1) / kTile : 0;
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
  __syncthreads();

  const long long N = static_cast<long long>(hkv) * cum[B];
  const int P = gridDim.x, c = blockIdx.x;
  const long long t_begin = tile_begin(c, N, P), t_end = tile_begin(c + 1, N, P);
  if (t_begin >= t_end) return;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    Cursor cur;
    cur.locate(t_begin, cum, B, hkv);
    const int nsub = kTile / p.box_tokens;
    const uint32_t box_bytes = static_cast<uint32_t>(p.box_tokens) * 128u;
    int it = 0;
    for (long long t = t_begin; t < t_end; ++t, ++it) {
      const int stage = it % kStages;
      const uint32_t phase = (it / kStages) & 1;
      bool ok = !*abort_flag && mbar_wait_bounded(&empty[stage], phase ^ 1, p.err_flag);
      if (!ok) {
        *abort_flag = 1;
      } else {
        const int Lb = lens[cur.b];
        const int tok = cur.j * kTile + lane * p.box_tokens;
        bool valid = false;
        int pb = 0;
        if (lane < nsub && tok < Lb) {
          pb = p.block_table[static_cast<long long>(cur.b) * p.max_blocks + (tok >> p.log2_bs)];
          if (pb < 0 || pb >= p.num_blocks) set_flag(p.err_flag, KVC_FLAG_BLOCK_ID_RANGE);
          else valid = true;
        }
        const uint32_t nvalid = __popc(__ballot_sync(0xffffffffu, valid));
        if (lane == 0) mbar_arrive_expect_tx(&full[stage], nvalid * box_bytes * L::kHalves * 2);
        __syncwarp();
        if (valid) {
          uint8_t* kdst = smem + stage * L::kStageBytes + lane * box_bytes;
          const int in_blk = tok & (p.block_size - 1);
#pragma unroll
          for (int h = 0; h < L::kHalves; ++h) {
            tma_load_4d(kdst + h * kHalfBytes, &tm_k, &full[stage], h * 64, cur.g, in_blk, pb);
            tma_load_4d(kdst + L::kKBytes + h * kHalfBytes, &tm_v, &full[stage], h * 64, cur.g,
                        in_blk, pb);
          }
        }
      }
      cur.advance(cum, B, hkv);
    }
    // Drain: every issued copy must land before this CTA's shared memory
    // can be released (matters only after an abort).
    if (*abort_flag) {
      const int first = it > kStages ? it - kStages : 0;
      for (int k = first; k < it; ++k)
        mbar_wait_bounded(&full[k % kStages], (k / kStages) & 1, p.err_flag);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const T* q = static_cast<const T*>(p.q);
  T* out = static_cast<T*>(p.out);
  Cursor cur;
  cur.locate(t_begin, cum, B, hkv);
  uint32_t qa[D / 16][4];
  float o[D / 8][4], m[2], l[2];
  auto reset = [&]() {
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[n][e] = 0.f;
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
  };
  load_q<T, D>(q, p, cur.b, cur.g, lane, qa);
  reset();
  int seg_first_j = cur.j;
  int slot = 0;  // 0 for the first segment this CTA touches, 1 afterwards
  const uint32_t sbase = smem_u32(smem);
  int it = 0;
  for (long long t = t_begin; t < t_end; ++t, ++it) {
    const int stage = it % kStages;
    const uint32_t phase = (it / kStages) & 1;
    bool ok = !*abort_flag && mbar_wait_bounded(&full[stage], phase, p.err_flag);
    if (!ok) *abort_flag = 1;
    const int valid = min(16, lens[cur.b] - cur.j * kTile - warp * 16);
    if (ok && valid > 0) {
      const uint32_t kb = sbase + stage * L::kStageBytes;
      attend_16<T, D>(kb, kb + L::kKBytes, warp, lane, valid, p.scale_log2, qa, o, m, l);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);

    const bool last_of_seg = cur.j == cur.n - 1;
    if (last_of_seg || t == t_end - 1) {
      // ---- finalize this segment's share: merge the 4 warps' states.
      const bool complete = seg_first_j == 0 && last_of_seg;
      float l0 = l[0], l1 = l[1];
      l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
      l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
      const int r0 = lane >> 2, r1 = r0 + 8, c0 = 2 * (lane & 3);
      if ((lane & 3) == 0) {
        if (r0 < G) { cmb_m[warp * G + r0] = m[0]; cmb_l[warp * G + r0] = l0; }
        if (r1 < G) { cmb_m[warp * G + r1] = m[1]; cmb_l[warp * G + r1] = l1; }
      }
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        if (r0 < G)
          *reinterpret_cast<float2*>(&cmb_o[(warp * G + r0) * D + n * 8 + c0]) =
              make_float2(o[n][0], o[n][1]);
        if (r1 < G)
          *reinterpret_cast<float2*>(&cmb_o[(warp * G + r1) * D + n * 8 + c0]) =
              make_float2(o[n][2], o[n][3]);
      }
      named_bar_sync(1, kConsumerWarps * 32);
      const int ctid = warp * 32 + lane;
      const long long row0 = static_cast<long long>(cur.b) * p.num_q_heads + cur.g * G;
      for (int e = ctid; e < G * D; e += kConsumerWarps * 32) {
        const int r = e / D, d = e - r * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, cmb_m[w * G + r]);
        float Ls = 0.f, Os = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) {
          const float mw = cmb_m[w * G + r];
          const float f = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
          Ls += f * cmb_l[w * G + r];
          Os += f * cmb_o[(w * G + r) * D + d];
        }
        if (complete) {
          out[(row0 + r) * D + d] = Pack<T>::cvt(Ls > 0.f ? Os / Ls : 0.f);
        } else {
          const long long ws_row = (static_cast<long long>(c) * 2 + slot) * G + r;
          p.ws_o[ws_row * D + d] = Os;
          if (d == 0) {
            p.ws_ml[ws_row * 2] = M;
            p.ws_ml[ws_row * 2 + 1] = Ls;
          }
        }
      }
      named_bar_sync(1, kConsumerWarps * 32);
      slot = 1;
      cur.advance(cum, B, hkv);
      if (t + 1 < t_end) {
        load_q<T, D>(q, p, cur.b, cur.g, lane, qa);
        reset();
        seg_first_j = cur.j;
      }
    } else {
      cur.advance(cum, B, hkv);
    }
  }
}

// Merge the per-CTA partial states of segments that were split, write zeros
// for empty sequences.  One CTA per (b, g).
template <typename T>
__global__ void __launch_bounds__(128)
    paged_decode_merge_kernel(const DecodeParams p, int P) {
  const int b = blockIdx.x / p.num_kv_heads, g = blockIdx.x - b * p.num_kv_heads;
  const int G = p.group, D = p.head_dim;
  const int cap = p.max_blocks * p.block_size;
  __shared__ long long s_before, s_total;
  __shared__ long long red[2][4];
  long long before = 0, total = 0;
  for (int i = threadIdx.x; i < p.batch; i += blockDim.x) {
    int L = p.seq_lens[i];
    L = L < 0 ? 0 : (L > cap ? cap : L);
    const long long n = (L + kTile - 1) / kTile;
    total += n;
    if (i < b) before += n;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, off);
    total += __shfl_xor_sync(0xffffffffu, total, off);
  }
  if ((threadIdx.x & 31) == 0) {
    red[0][threadIdx.x >> 5] = before;
    red[1][threadIdx.x >> 5] = total;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    s_before = red[0][0] + red[0][1] + red[0][2] + red[0][3];
    s_total = red[1][0] + red[1][1] + red[1][2] + red[1][3];
  }
  __syncthreads();
  int Lb = p.seq_lens[b];
  Lb = Lb < 0 ? 0 : (Lb > cap ? cap : Lb);
  T* out = static_cast<T*>(p.out) + (static_cast<long long>(b) * p.num_q_heads + g * G) * D;
  if (Lb == 0) {
    for (int e = threadIdx.x; e < G * D; e += blockDim.x) out[e] = Pack<T>::cvt(0.f);
    return;
  }
  const long long nb = (Lb + kTile - 1) / kTile;
  const long long N = static_cast<long long>(p.num_kv_heads) * s_total;
  const long long seg0 = static_cast<long long>(p.num_kv_heads) * s_before + g * nb;
  const int c0 = cta_of(seg0, N, P), c1 = cta_of(seg0 + nb - 1, N, P);
  if (c0 == c1) return;  // written directly by the main kernel
  const int slot0 = tile_begin(c0, N, P) == seg0 ? 0 : 1;
  for (int e = threadIdx.x; e < G * D; e += blockDim.x) {
    const int r = e / D, d = e - r * D;
    float M = -INFINITY;
    for (int c = c0; c <= c1; ++c) {
      const long long row = (static_cast<long long>(c) * 2 + (c == c0 ? slot0 : 0)) * G + r;
      M = fmaxf(M, p.ws_ml[row * 2]);
    }
    float Ls = 0.f, Os = 0.f;
    for (int c = c0; c <= c1; ++c) {
      const long long row = (static_cast<long long>(c) * 2 + (c == c0 ? slot0 : 0)) * G + r;
      const float f = fast_exp2(p.ws_ml[row * 2] - M);
      Ls += f * p.ws_ml[row * 2 + 1];
      Os += f * p.ws_o[row * D + d];
    }
    out[e] = Pack<T>::cvt(Ls > 0.f ? Os / Ls : 0.f);
  }
}

template <typename T, int D>
struct DecodeKernel {
  // Resident CTAs per SM for a launch with `smem` bytes of dynamic shared
  // memory (cached per device and size; also sets the kernel's smem limit).
  static int occupancy(size_t smem) {
    static std::mutex mu;
    static std::map<std::pair<int, size_t>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find({dev, smem});
    if (it != cache.end()) return it->second;
    cudaFuncSetAttribute(paged_decode_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(Layout<D>::bytes(kMaxBatch, 16)));
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, paged_decode_kernel<T, D>, kThreads,
                                                      smem) != cudaSuccess || occ < 1)
      occ = 1;
    cache[{dev, smem}] = occ;
    return occ;
  }
};

template <typename T, int D>
kvc_status run_decode(const DecodeArgs& a) {
  const int G = a.num_q_heads / a.num_kv_heads;
  const size_t smem = Layout<D>::bytes(a.batch, G);
  const int occ = DecodeKernel<T, D>::occupancy(smem);  // also sets the smem limit
  const int P = a.num_ctas > 0 ? a.num_ctas : device_sm_count() * occ;
  if (a.workspace_bytes < paged_decode_workspace_bytes(G, D, P) || a.workspace == nullptr)
    return KVC_ERR_WORKSPACE;

  CUtensorMap tk, tv;
  const int box_tokens = a.block_size < kTile ? a.block_size : kTile;
  const uint64_t dims[4] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.num_kv_heads),
                            static_cast<uint64_t>(a.block_size),
                            static_cast<uint64_t>(a.num_blocks)};
  const uint64_t strides[3] = {static_cast<uint64_t>(D) * 2,
                               static_cast<uint64_t>(a.num_kv_heads) * D * 2,
                               static_cast<uint64_t>(a.block_size) * a.num_kv_heads * D * 2};
  const uint32_t box[4] = {64, 1, static_cast<uint32_t>(box_tokens), 1};
  if (!encode_tmap_16bit(&tk, a.dtype, 4, a.key_cache, dims, strides, box, true) ||
      !encode_tmap_16bit(&tv, a.dtype, 4, a.value_cache, dims, strides, box, true))
    return KVC_ERR_CUDA;

  DecodeParams p;
  p.q = a.q;
  p.out = a.out;
  p.block_table = a.block_table;
  p.seq_lens = a.seq_lens;
  p.ws_o = static_cast<float*>(a.workspace);
  p.ws_ml = p.ws_o + static_cast<size_t>(P) * 2 * G * D;
  p.err_flag = a.err_flag;
  p.batch = a.batch;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = G;
  p.head_dim = D;
  p.block_size = a.block_size;
  p.log2_bs = ilog2(a.block_size);
  p.max_blocks = a.max_blocks_per_seq;
  p.num_blocks = a.num_blocks;
  p.box_tokens = box_tokens;
  p.scale_log2 = a.scale * 1.4426950408889634f;

  paged_decode_kernel<T, D><<<P, kThreads, smem, a.stream>>>(tk, tv, p);
  if (cudaGetLastError() != cudaSuccess) return KVC_ERR_CUDA;
  paged_decode_merge_kernel<T><<<a.batch * a.num_kv_heads, 128, 0, a.stream>>>(p, P);
  if (cudaGetLastError() != cudaSuccess) return KVC_ERR_CUDA;
  return KVC_OK;
}

}  // namespace

size_t paged_decode_workspace_bytes(int group, int head_dim, int ctas) {
  return static_cast<size_t>(ctas) * 2 * group * (head_dim + 2) * sizeof(float);
}

int paged_decode_num_ctas(int group, int head_dim, kvc_dtype dtype, int num_ctas) {
  if (num_ctas > 0) return num_ctas;
  const int sms = device_sm_count();
  if (sms <= 0) return 0;
  // The smallest batch needs the least shared memory, hence the most CTAs.
  if (head_dim == 64) {
    const size_t smem = Layout<64>::bytes(1, group);
    return sms * (dtype == KVC_BF16 ? DecodeKernel<__nv_bfloat16, 64>::occupancy(smem)
                                    : DecodeKernel<__half, 64>::occupancy(smem));
  }
  if (head_dim == 128) {
    const size_t smem = Layout<128>::bytes(1, group);
    return sms * (dtype == KVC_BF16 ? DecodeKernel<__nv_bfloat16, 128>::occupancy(smem)
                                    : DecodeKernel<__half, 128>::occupancy(smem));
  }
  return 0;
}

kvc_status launch_paged_decode(const DecodeArgs& a) {
  if (a.head_dim == 64)
    return a.dtype == KVC_BF16 ? run_decode<__nv_bfloat16, 64>(a) : run_decode<__half, 64>(a);
  if (a.head_dim == 128)
    return a.dtype == KVC_BF16 ? run_decode<__nv_bfloat16, 128>(a) : run_decode<__half, 128>(a);
  return KVC_ERR_UNSUPPORTED;
}

}  // namespace kvc
