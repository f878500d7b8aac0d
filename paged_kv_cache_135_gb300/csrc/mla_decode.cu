// MLA paged decode on the tcgen05 tensor cores (row a6 of the hot path).
//
// What it computes: "external-cannbot-model-model-infer-kvcache" Mode 3 --
// the cache holds only the compressed latent cache_nope (kv_lora_rank = 512)
// and the positional cache_rope (64) per token; FA is called with key =
// value = cache_nope plus query_rope / key_rope, so for every head h
//   s_j = scale * (q_nope[h] . nope_j + q_rope[h] . rope_j),
//   out[h] = sum_j softmax_j(s) nope_j            (512 wide),
// all 128 query heads sharing the one latent head, read through block_table
// with per-sequence lengths (Mode 2).
//
// GB300 design.  The 128 heads are the M = 128 side of tcgen05.mma.  The
// output (128 x 512 fp32) does not fit one SM's tensor memory next to the
// scores, so a cluster of two CTAs shares each work unit:
//   * rank 0 owns key columns nope[0:256] and output columns 0..255, rank 1
//     owns nope[256:512] + rope[0:64] and output columns 256..511; each CTA
//     loads only its own columns of every cached token (the pair reads each
//     token once) and the query columns that go with them;
//   * each CTA computes a partial S = Q_own K_own^T (M 128, N 64 tokens) into
//     tensor memory; the two partials are exchanged through distributed
//     shared memory and summed, so both CTAs hold the full S;
//   * both run the same online softmax (one query row per thread, log2
//     domain, rescaling of O only when the running max grows by more than
//     2^8), write P (bf16, 128-byte swizzled) to shared memory and compute
//     O_own += P V_own with V = their nope columns, straight from the K tile
//     (MN-major operand), accumulating in tensor memory.
// Work: 64-token tiles of all sequences in one linear order, split evenly
// over the clusters (stream-K split-KV); the cluster that finishes a split
// sequence last merges the partial states (per rank), as in the GQA decode.
// Roles per CTA: warps 0-3 softmax / epilogue (one TMEM lane per thread),
// warp 4 TMA producer, warp 5 tcgen05 issuer (one thread) and TMEM owner.
#include <cuda_runtime.h>

#include <math.h>

#include <mutex>

#include "kvc_device.cuh"
#include "kvc_host.h"
#include "kvc_sched.cuh"
#include "kvc_tcgen05.cuh"

namespace kvc {

namespace {

constexpr int kH = 128;             // query heads = MMA M
constexpr int kTok = 64;            // tokens per tile = N of QK, K of PV
constexpr int kNope = 512, kRope = 64;
constexpr int kOutCols = 256;       // output columns per CTA
constexpr int kMaxChunks = 5;       // 64-wide key chunks per CTA (rank 1: 4 nope + rope)
constexpr int kQChunkBytes = kH * 128;     // [128 heads][64 elements]
constexpr int kKChunkBytes = kTok * 128;   // [64 tokens][64 elements]
constexpr int kStages = 2;
constexpr int kSoftmaxThreads = 128;
constexpr int kThreads = kSoftmaxThreads + 64;  // + producer warp + MMA warp
constexpr int kMaxBatch = 1024;
constexpr int kMaxPieces = 62;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows by > 2^8

// TMEM columns: O (256 fp32) then two S buffers (64 fp32 each).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0, kTmemS0 = 256, kTmemS1 = 320;

struct MlaParams {
  void* out;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int* ws_cnt;    // [clusters][2 slots][2 ranks]
  float* ws_o;    // [clusters][2][2][128][256]
  float* ws_ml;   // [clusters][2][2][128][2]
  uint32_t* err_flag;
  int batch, block_size, log2_bs, max_blocks, num_blocks, box_tokens;
  float scale_log2;
};

// Shared memory (1024-aligned base).  Regions sized for rank 1 (5 chunks).
struct MlaLayout {
  static constexpr int kQ = 0;                                       // 5 x 16 KB
  static constexpr int kK = kQ + kMaxChunks * kQChunkBytes;          // 2 x 5 x 8 KB
  static constexpr int kStageBytes = kMaxChunks * kKChunkBytes;
  static constexpr int kP = kK + kStages * kStageBytes;              // 16 KB
  static constexpr int kX = kP + kH * 128;                           // 32 KB
  static constexpr int kBar = kX + kH * kTok * 4;
  // barriers: q_full, q_free, k_full[2], k_empty[2], s_full[2], s_free[2],
  //           p_full, pv_done, x_full, x_empty
  static constexpr int kNumBars = 15;
  static constexpr int kMisc = kBar + kNumBars * 8;                  // tmem slot, flags
  static constexpr int kPieces = kMisc + 32;
  static constexpr int kLens = kPieces + kMaxPieces * 4 + 8;         // 16-aligned below
  __host__ __device__ static int lens_off() { return (kLens + 15) & ~15; }
  __host__ __device__ static int cum_off(int batch) { return lens_off() + ((batch + 3) & ~3) * 4; }
  static size_t bytes(int batch) { return 1024 + cum_off(batch) + (batch + 1) * 4 + 16; }
};

enum Bar { kQFull = 0, kQFree, kKFull0, kKFull1, kKEmpty0, kKEmpty1, kSFull0, kSFull1,
           kSFree0, kSFree1, kPFull, kPVDone, kXFull, kXEmpty, kDrain };

// Bounded wait that also gives up at once after another role aborted.
__device__ __forceinline__ bool wait_cta(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                         uint32_t* err) {
  if (*abort_flag) return false;
  if (mbar_wait_bounded(bar, parity, err)) return true;
  *abort_flag = 1;
  return false;
}
__device__ __forceinline__ bool wait_peer(uint64_t* bar, uint32_t parity,
                                          volatile int* abort_flag, uint32_t* err) {
  if (*abort_flag) return false;
  if (mbar_wait_cluster_bounded(bar, parity, err)) return true;
  *abort_flag = 1;
  return false;
}

// ------------------------------------------------------------- producer
// TMA loads: at each new sequence the CTA's query columns (after the tensor
// core has finished with the previous ones), then every tile's own key
// columns, one box per physical block per 64-wide chunk.
__device__ __forceinline__ void mla_producer(const MlaParams& p, const CUtensorMap* tm_qn,
                                             const CUtensorMap* tm_qr, const CUtensorMap* tm_cn,
                                             const CUtensorMap* tm_cr, uint8_t* smem,
                                             uint64_t* bars, volatile int* abort_flag,
                                             const int* lens, const int* cum, long long tb,
                                             long long te, int rank, int lane) {
  using L = MlaLayout;
  const int nq = rank ? 5 : 4;
  const int B = p.batch;
  sched::Cursor cur;
  cur.locate(tb, cum, B, 1);
  const int nsub = kTok / p.box_tokens;
  const uint32_t box_bytes = static_cast<uint32_t>(p.box_tokens) * 128u;
  int seg = 0;
  for (long long t = tb; t < te; ++t) {
    const int it = static_cast<int>(t - tb);
    if (it == 0 || cur.j == 0) {
      const bool q_ok = seg == 0 || wait_cta(&bars[kQFree], (seg - 1) & 1, abort_flag, p.err_flag);
      if (lane == 0 && q_ok) {
        mbar_arrive_expect_tx(&bars[kQFull], nq * kQChunkBytes);
        for (int c = 0; c < 4; ++c)
          tma_load_3d(smem + L::kQ + c * kQChunkBytes, tm_qn, &bars[kQFull], (rank * 4 + c) * 64,
                      0, cur.b);
        if (rank) tma_load_3d(smem + L::kQ + 4 * kQChunkBytes, tm_qr, &bars[kQFull], 0, 0, cur.b);
      }
      ++seg;
    }
    const int stage = it & 1;
    const int Lb = lens[cur.b];
    const int tok = cur.j * kTok + lane * p.box_tokens;
    int pb = -1;
    if (lane < nsub && tok < Lb)
      pb = __ldg(&p.block_table[static_cast<long long>(cur.b) * p.max_blocks + (tok >> p.log2_bs)]);
    const bool ok = wait_cta(&bars[kKEmpty0 + stage], ((it >> 1) & 1) ^ 1, abort_flag, p.err_flag);
    bool valid = false;
    if (lane < nsub && tok < Lb) {
      if (pb < 0 || pb >= p.num_blocks) set_flag(p.err_flag, KVC_FLAG_BLOCK_ID_RANGE);
      else valid = ok;
    }
    const uint32_t nvalid = __popc(__ballot_sync(0xffffffffu, valid));
    if (lane == 0) mbar_arrive_expect_tx(&bars[kKFull0 + stage], nvalid * box_bytes * nq);
    __syncwarp();
    if (valid) {
      uint8_t* dst = smem + L::kK + stage * L::kStageBytes + lane * box_bytes;
      const int in_blk = tok & (p.block_size - 1);
      for (int c = 0; c < 4; ++c)
        tma_load_3d(dst + c * kKChunkBytes, tm_cn, &bars[kKFull0 + stage], (rank * 4 + c) * 64,
                    in_blk, pb);
      if (rank) tma_load_3d(dst + 4 * kKChunkBytes, tm_cr, &bars[kKFull0 + stage], 0, in_blk, pb);
    }
    cur.advance(cum, B, 1);
  }
}

// --------------------------------------------------------------- tcgen05
// S = Q K^T over NQ 64-wide chunks, fully unrolled from two base descriptors.
template <int NQ>
__device__ __forceinline__ void mla_issue_s(uint32_t d, uint64_t q0, uint64_t k0, uint32_t idesc) {
#pragma unroll
  for (int c = 0; c < NQ; ++c)
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t a = desc_advance(q0, c * kQChunkBytes + kk * 32);
      const uint64_t b = desc_advance(k0, c * kKChunkBytes + kk * 32);
      if (c == 0 && kk == 0) umma_f16_fresh(d, a, b, idesc);
      else umma_f16_acc(d, a, b, idesc);
    }
}

// One thread.  S(t+1) = Q K(t+1)^T is issued before O += P(t) V(t), so the
// tensor core computes the next scores while the softmax works on P(t).
template <bool kBf16>
__device__ __forceinline__ void mla_mma(const MlaParams& p, uint8_t* smem, uint64_t* bars,
                                        volatile int* abort_flag, const int* cum, uint32_t tmem,
                                        long long tb, long long te, int rank) {
  using L = MlaLayout;
  const uint32_t idesc_s = umma_idesc_f16(kBf16, kH, kTok, 0, 0);
  const uint32_t idesc_o = umma_idesc_f16(kBf16, kH, kOutCols, 0, 1);
  const uint64_t q0 = umma_desc_sw128(smem_u32(smem + L::kQ), 16, 1024);
  const uint64_t k0 = umma_desc_sw128(smem_u32(smem + L::kK), 16, 1024);
  const uint64_t p0 = umma_desc_sw128(smem_u32(smem + L::kP), 16, 1024);
  // V = the first four chunks of a stage, MN-major: next 64 columns 8 KB on.
  const uint64_t v0 = umma_desc_sw128(smem_u32(smem + L::kK), kKChunkBytes, 1024);
  const int n_it = static_cast<int>(te - tb);
  sched::Cursor cs;  // tile whose S is issued next
  cs.locate(tb, cum, p.batch, 1);
  int seg_s = -1;
  bool first_flags[2] = {false, false};

  auto issue_s = [&](int it) -> bool {
    const bool first = it == 0 || cs.j == 0;
    const bool last = it == n_it - 1 || cs.j == cs.n - 1;
    if (first) ++seg_s;
    first_flags[it & 1] = first;
    const int stage = it & 1;
    if (!wait_cta(&bars[kKFull0 + stage], (it >> 1) & 1, abort_flag, p.err_flag)) return false;
    if (!wait_cta(&bars[kSFree0 + stage], ((it >> 1) & 1) ^ 1, abort_flag, p.err_flag)) return false;
    if (!wait_cta(&bars[kQFull], seg_s & 1, abort_flag, p.err_flag)) return false;
    tc_fence_after();
    const uint32_t d = tmem + (stage ? kTmemS1 : kTmemS0);
    const uint64_t k_st = desc_advance(k0, stage * L::kStageBytes);
    if (rank) mla_issue_s<5>(d, q0, k_st, idesc_s);
    else mla_issue_s<4>(d, q0, k_st, idesc_s);
    umma_commit(&bars[kSFull0 + stage]);
    if (last) umma_commit(&bars[kQFree]);
    cs.advance(cum, p.batch, 1);
    return true;
  };
  auto issue_pv = [&](int it) -> bool {
    if (!wait_cta(&bars[kPFull], it & 1, abort_flag, p.err_flag)) return false;
    tc_fence_after();
    const uint64_t v_st = desc_advance(v0, (it & 1) * L::kStageBytes);
    if (first_flags[it & 1]) umma_f16_fresh(tmem + kTmemO, p0, v_st, idesc_o);
    else umma_f16_acc(tmem + kTmemO, p0, v_st, idesc_o);
#pragma unroll
    for (int ks = 1; ks < kTok / 16; ++ks)
      umma_f16_acc(tmem + kTmemO, desc_advance(p0, ks * 32), desc_advance(v_st, ks * 16 * 128),
                   idesc_o);
    umma_commit(&bars[kPVDone]);
    umma_commit(&bars[kKEmpty0 + (it & 1)]);
    return true;
  };

  if (n_it > 0 && !issue_s(0)) return;
  for (int it = 0; it < n_it; ++it) {
    if (it + 1 < n_it && !issue_s(it + 1)) return;
    if (!issue_pv(it)) return;
  }
}

// ----------------------------------------------------------- epilogue
// End of one sequence's share for query row `row` (one thread): write the
// normalised output columns of this rank, or publish a partial state; the
// cluster arriving last at a split sequence merges every share (per rank).
template <typename T>
__device__ __noinline__ void mla_finish(const MlaParams& p, uint32_t o_taddr, int row, int b,
                                        bool complete, int cl, int slot, long long seg0,
                                        int seg_tiles, long long N, int P, int rank, float m_used,
                                        float l, volatile int* last_flag, volatile int* npieces,
                                        int* pieces) {
  T* out = static_cast<T*>(p.out) + (static_cast<long long>(b) * kH + row) * kNope + rank * kOutCols;
  if (complete) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    for (int c = 0; c < kOutCols / 16; ++c) {
      float v[16];
      tmem_ld16(o_taddr + c * 16, v);
      tmem_wait_ld();
      uint32_t w[8];
      float ra, rb;
#pragma unroll
      for (int k = 0; k < 8; ++k) w[k] = Pack<T>::run(v[2 * k] * inv, v[2 * k + 1] * inv, ra, rb);
      *reinterpret_cast<uint4*>(out + c * 16) = make_uint4(w[0], w[1], w[2], w[3]);
      *reinterpret_cast<uint4*>(out + c * 16 + 8) = make_uint4(w[4], w[5], w[6], w[7]);
    }
    return;
  }
  const long long wrow = ((static_cast<long long>(cl) * 2 + slot) * 2 + rank) * kH + row;
  for (int c = 0; c < kOutCols / 16; ++c) {
    float v[16];
    tmem_ld16(o_taddr + c * 16, v);
    tmem_wait_ld();
    float4* dst = reinterpret_cast<float4*>(p.ws_o + wrow * kOutCols + c * 16);
#pragma unroll
    for (int k = 0; k < 4; ++k) dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
  }
  *reinterpret_cast<float2*>(p.ws_ml + wrow * 2) = make_float2(m_used, l);
  named_bar_sync(1, kSoftmaxThreads);
  const int cfirst = sched::share_of(seg0, N, P), clast = sched::share_of(seg0 + seg_tiles - 1, N, P);
  const int slot0 = sched::share_begin(cfirst, N, P) == seg0 ? 0 : 1;
  if (row == 0) {
    int n = 0;
    long long tb = sched::share_begin(cfirst, N, P);
    for (int cc = cfirst; cc <= clast; ++cc) {
      const long long te = sched::share_begin(cc + 1, N, P);
      if (tb < te) {
        if (n < kMaxPieces) pieces[n] = cc * 2 + (cc == cfirst ? slot0 : 0);
        ++n;
      }
      tb = te;
    }
    *npieces = n;
    *last_flag =
        atomic_add_acq_rel(&p.ws_cnt[(cfirst * 2 + slot0) * 2 + rank], 1) == n - 1 ? 1 : 0;
  }
  named_bar_sync(1, kSoftmaxThreads);
  if (*last_flag) {
    __threadfence();
    const int n = *npieces;
    // Workspace row of every share in CTA order: from the shared-memory list,
    // or (very many shares) by walking the cluster range again.
    const bool listed = n <= kMaxPieces;
    int cc = cfirst;
    auto next_row = [&](int i) -> long long {
      if (listed) return (static_cast<long long>(pieces[i]) * 2 + rank) * kH + row;
      while (sched::share_begin(cc, N, P) == sched::share_begin(cc + 1, N, P)) ++cc;
      const long long r =
          ((static_cast<long long>(cc) * 2 + (cc == cfirst ? slot0 : 0)) * 2 + rank) * kH + row;
      ++cc;
      return r;
    };
    float M = -INFINITY;
    cc = cfirst;
    for (int i = 0; i < n; ++i) M = fmaxf(M, __ldcg(p.ws_ml + next_row(i) * 2));
    float Ls = 0.f;
    cc = cfirst;
    for (int i = 0; i < n; ++i) {
      const long long r = next_row(i);
      Ls += fast_exp2(__ldcg(p.ws_ml + r * 2) - M) * __ldcg(p.ws_ml + r * 2 + 1);
    }
    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
    for (int c = 0; c < kOutCols / 16; ++c) {
      float acc[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) acc[k] = 0.f;
      cc = cfirst;
      for (int i = 0; i < n; ++i) {
        const long long r = next_row(i);
        const float f = fast_exp2(__ldcg(p.ws_ml + r * 2) - M);
        const float4* src = reinterpret_cast<const float4*>(p.ws_o + r * kOutCols + c * 16);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float4 v = __ldcg(src + k);
          acc[4 * k] += f * v.x;
          acc[4 * k + 1] += f * v.y;
          acc[4 * k + 2] += f * v.z;
          acc[4 * k + 3] += f * v.w;
        }
      }
      uint32_t w[8];
      float ra, rb;
#pragma unroll
      for (int k = 0; k < 8; ++k) w[k] = Pack<T>::run(acc[2 * k] * inv, acc[2 * k + 1] * inv, ra, rb);
      *reinterpret_cast<uint4*>(out + c * 16) = make_uint4(w[0], w[1], w[2], w[3]);
      *reinterpret_cast<uint4*>(out + c * 16 + 8) = make_uint4(w[4], w[5], w[6], w[7]);
    }
    if (row == 0) p.ws_cnt[(cfirst * 2 + slot0) * 2 + rank] = 0;
  }
  named_bar_sync(1, kSoftmaxThreads);
}

// --------------------------------------------------------------- softmax
// Warps 0-3; thread `row` owns query head `row` (TMEM lane `row`).
template <typename T>
__device__ __forceinline__ void mla_softmax(const MlaParams& p, uint8_t* smem, uint64_t* bars,
                                            volatile int* abort_flag, volatile int* last_flag,
                                            volatile int* npieces, int* pieces, const int* lens,
                                            const int* cum, uint32_t tmem, long long tb,
                                            long long te, long long N, int P, int cl, int rank,
                                            int row) {
  using L = MlaLayout;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>((row >> 5) * 32) << 16);
  const uint32_t peer = static_cast<uint32_t>(rank ^ 1);
  const uint32_t x_peer = map_to_rank(smem_u32(smem + L::kX), peer);
  const uint32_t xfull_peer = map_to_rank(smem_u32(&bars[kXFull]), peer);
  const uint32_t xempty_peer = map_to_rank(smem_u32(&bars[kXEmpty]), peer);
  const float4* x_mine = reinterpret_cast<const float4*>(smem + L::kX);
  sched::Cursor cur;
  cur.locate(tb, cum, p.batch, 1);
  float m_used = -INFINITY, l = 0.f;
  int seg_first_j = cur.j, slot = 0;
  for (long long t = tb; t < te; ++t) {
    const int it = static_cast<int>(t - tb);
    const bool first = it == 0 || cur.j == 0;
    const bool last = t == te - 1 || cur.j == cur.n - 1;
    if (first) {
      m_used = -INFINITY;
      l = 0.f;
      seg_first_j = cur.j;
    }
    const int stage = it & 1;
    const int valid = min(kTok, lens[cur.b] - cur.j * kTok);

    // 1. This CTA's partial scores (the collective TMEM reads run even after
    //    an abort; only the waits give up).
    float s[kTok];
    wait_cta(&bars[kSFull0 + stage], (it >> 1) & 1, abort_flag, p.err_flag);
    tc_fence_after();
#pragma unroll
    for (int c = 0; c < kTok / 16; ++c)
      tmem_ld16(lane_base + (stage ? kTmemS1 : kTmemS0) + c * 16, s + c * 16);
    tmem_wait_ld();
    tc_fence_before();
    mbar_arrive(&bars[kSFree0 + stage]);

    // 2. Exchange partial scores with the other CTA of the pair and sum them.
    //    One elected thread signals after a CTA barrier: its cluster-scope
    //    release covers every thread's remote stores before it.
    wait_peer(&bars[kXEmpty], (it & 1) ^ 1, abort_flag, p.err_flag);
#pragma unroll
    for (int q = 0; q < kTok / 4; ++q)
      st_cluster_v4(x_peer + (q * kH + row) * 16,
                    make_float4(s[4 * q], s[4 * q + 1], s[4 * q + 2], s[4 * q + 3]));
    named_bar_sync(2, kSoftmaxThreads);
    if (row == 0) mbar_arrive_cluster(xfull_peer);
    wait_peer(&bars[kXFull], it & 1, abort_flag, p.err_flag);
#pragma unroll
    for (int q = 0; q < kTok / 4; ++q) {
      const float4 v = x_mine[q * kH + row];
      s[4 * q] += v.x;
      s[4 * q + 1] += v.y;
      s[4 * q + 2] += v.z;
      s[4 * q + 3] += v.w;
    }
    named_bar_sync(2, kSoftmaxThreads);
    if (row == 0) mbar_arrive_cluster(xempty_peer);

    // 3. Online softmax in the log2 domain; O is rescaled only when the
    //    running max grows by more than 2^kRescaleThreshold.
    float mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < kTok; ++k) {
      s[k] = k < valid ? s[k] * p.scale_log2 : -INFINITY;
      mx = fmaxf(mx, s[k]);
    }
    float corr = 1.f;
    bool rescale = false;
    if (m_used == -INFINITY) {
      m_used = mx;
      corr = 0.f;
    } else if (mx > m_used + kRescaleThreshold) {
      corr = fast_exp2(m_used - mx);
      m_used = mx;
      rescale = true;
    }
    uint32_t pk[kTok / 2];
    float ps = 0.f, ra, rb;
#pragma unroll
    for (int k = 0; k < kTok / 2; ++k) {
      pk[k] = Pack<T>::run(fast_exp2(s[2 * k] - m_used), fast_exp2(s[2 * k + 1] - m_used), ra, rb);
      ps += ra + rb;
    }
    l = l * corr + ps;

    // 4. The previous P V must be finished before P and O are touched.
    if (it > 0) {
      wait_cta(&bars[kPVDone], (it - 1) & 1, abort_flag, p.err_flag);
      tc_fence_after();
    }
    if (__any_sync(0xffffffffu, rescale)) {
      for (int c = 0; c < kOutCols / 16; ++c) {
        float v[16];
        tmem_ld16(lane_base + kTmemO + c * 16, v);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] *= corr;
        tmem_st16(lane_base + kTmemO + c * 16, v);
      }
      tmem_wait_st();
    }

    // 5. P row -> shared memory (K-major, 128-byte swizzle); zero the value
    //    rows past the sequence so stale cache contents cannot reach P V.
    uint8_t* sp = smem + L::kP;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch)
      *reinterpret_cast<uint4*>(sp + swz128(row, ch)) =
          make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
    if (valid < kTok) {
      uint8_t* kst = smem + L::kK + stage * L::kStageBytes;
      const int n16 = (kTok - valid) * 4 * 8;
      for (int e = row; e < n16; e += kSoftmaxThreads) {
        const int r = valid + e / 32, c = (e % 32) / 8, q = e % 8;
        *reinterpret_cast<uint4*>(kst + c * kKChunkBytes + r * 128 + q * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    mbar_arrive(&bars[kPFull]);

    // 6. End of this sequence's share.
    if (last) {
      wait_cta(&bars[kPVDone], it & 1, abort_flag, p.err_flag);
      tc_fence_after();
      mla_finish<T>(p, lane_base + kTmemO, row, cur.b, seg_first_j == 0 && cur.j == cur.n - 1, cl,
                    slot, static_cast<long long>(cum[cur.b]), cur.n, N, P, rank, m_used, l,
                    last_flag, npieces, pieces);
      tc_fence_before();
      slot = 1;
    }
    cur.advance(cum, p.batch, 1);
  }
}

template <typename T, bool kBf16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tm_qn,
                      const __grid_constant__ CUtensorMap tm_qr,
                      const __grid_constant__ CUtensorMap tm_cn,
                      const __grid_constant__ CUtensorMap tm_cr,
                      const __grid_constant__ MlaParams p) {
  using L = MlaLayout;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  volatile int* last_flag = abort_flag + 1;
  volatile int* npieces = abort_flag + 2;
  int* pieces = reinterpret_cast<int*>(smem + L::kPieces);
  int* lens = reinterpret_cast<int*>(smem + L::lens_off());
  int* cum = reinterpret_cast<int*>(smem + L::cum_off(p.batch));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const int cl = static_cast<int>(blockIdx.x >> 1), P = static_cast<int>(gridDim.x >> 1);
  const int B = p.batch, cap = p.max_blocks * p.block_size;

  if (tid == 0) {
    const uint32_t counts[L::kNumBars] = {1, 1, 1, 1, 1, 1, 1, 1, kSoftmaxThreads,
                                          kSoftmaxThreads, kSoftmaxThreads, 1, 1, 1, 1};
    for (int i = 0; i < L::kNumBars; ++i) mbar_init(&bars[i], counts[i]);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 5) tmem_alloc(tslot, kTmemCols);
  if (warp == 4 && lane == 0) {
    prefetch_tmap(&tm_qn);
    prefetch_tmap(&tm_qr);
    prefetch_tmap(&tm_cn);
    prefetch_tmap(&tm_cr);
  }
  for (int i = tid; i < B; i += kThreads) lens[i] = sched::clamp_len(p.seq_lens[i], cap, p.err_flag);
  __syncthreads();
  if (warp == 0) sched::plan_tiles(lens, cum, B, kTok, lane);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // both CTAs' barriers exist before any remote arrive

  const uint32_t tmem = *tslot;
  const long long N = cum[B];
  const long long tb = sched::share_begin(cl, N, P), te = sched::share_begin(cl + 1, N, P);
  {  // sequences with no cached token: rows of zeros (this rank's columns)
    T* out = static_cast<T*>(p.out);
    for (int b = cl; b < B; b += P)
      if (lens[b] == 0)
        for (int e = tid; e < kH * kOutCols; e += kThreads)
          out[(static_cast<long long>(b) * kH + e / kOutCols) * kNope + rank * kOutCols +
              e % kOutCols] = Pack<T>::cvt(0.f);
  }
  if (tb < te) {
    if (warp < 4) {
      mla_softmax<T>(p, smem, bars, abort_flag, last_flag, npieces, pieces, lens, cum, tmem, tb, te,
                     N, P, cl, rank, tid);
    } else if (warp == 4) {
      mla_producer(p, &tm_qn, &tm_qr, &tm_cn, &tm_cr, smem, bars, abort_flag, lens, cum, tb, te,
                   rank, lane);
      // Every copy issued must land before shared memory can be released.
      const int n_it = static_cast<int>(te - tb);
      for (int it = max(0, n_it - kStages); it < n_it; ++it)
        mbar_wait_bounded(&bars[kKFull0 + (it & 1)], (it >> 1) & 1, p.err_flag);
    } else if (lane == 0) {
      mla_mma<kBf16>(p, smem, bars, abort_flag, cum, tmem, tb, te, rank);
    }
  }
  // Teardown: all tensor-core work done, TMEM freed, and neither CTA leaves
  // while its partner may still write into its shared memory.
  if (warp == 5 && lane == 0) {
    umma_commit(&bars[kDrain]);
    mbar_wait_bounded(&bars[kDrain], 0, p.err_flag);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_sync();
}

}  // namespace

namespace {

size_t mla_counter_bytes(int clusters) {
  return (static_cast<size_t>(clusters) * 4 * sizeof(int) + 255) & ~static_cast<size_t>(255);
}

template <typename T, bool kBf16>
kvc_status run_mla(const MlaArgs& a, int clusters) {
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(mla_decode_kernel<T, kBf16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(MlaLayout::bytes(kMaxBatch)));
  });
  const int box_tokens = a.block_size < kTok ? a.block_size : kTok;
  CUtensorMap qn, qr, cn, cr;
  const uint64_t qn_dims[3] = {kNope, kH, static_cast<uint64_t>(a.batch)};
  const uint64_t qn_str[2] = {kNope * 2, static_cast<uint64_t>(kH) * kNope * 2};
  const uint64_t qr_dims[3] = {kRope, kH, static_cast<uint64_t>(a.batch)};
  const uint64_t qr_str[2] = {kRope * 2, static_cast<uint64_t>(kH) * kRope * 2};
  const uint32_t qbox[3] = {64, kH, 1};
  const uint64_t cn_dims[3] = {kNope, static_cast<uint64_t>(a.block_size),
                               static_cast<uint64_t>(a.num_blocks)};
  const uint64_t cn_str[2] = {kNope * 2, static_cast<uint64_t>(a.block_size) * kNope * 2};
  const uint64_t cr_dims[3] = {kRope, static_cast<uint64_t>(a.block_size),
                               static_cast<uint64_t>(a.num_blocks)};
  const uint64_t cr_str[2] = {kRope * 2, static_cast<uint64_t>(a.block_size) * kRope * 2};
  const uint32_t cbox[3] = {64, static_cast<uint32_t>(box_tokens), 1};
  if (!encode_tmap_16bit(&qn, a.dtype, 3, a.q_nope, qn_dims, qn_str, qbox, true) ||
      !encode_tmap_16bit(&qr, a.dtype, 3, a.q_rope, qr_dims, qr_str, qbox, true) ||
      !encode_tmap_16bit(&cn, a.dtype, 3, a.cache_nope, cn_dims, cn_str, cbox, true) ||
      !encode_tmap_16bit(&cr, a.dtype, 3, a.cache_rope, cr_dims, cr_str, cbox, true))
    return KVC_ERR_CUDA;
  MlaParams p;
  p.out = a.out;
  p.block_table = a.block_table;
  p.seq_lens = a.seq_lens;
  p.ws_cnt = static_cast<int*>(a.workspace);
  p.ws_o = reinterpret_cast<float*>(static_cast<char*>(a.workspace) + mla_counter_bytes(clusters));
  p.ws_ml = p.ws_o + static_cast<size_t>(clusters) * 4 * kH * kOutCols;
  p.err_flag = a.err_flag;
  p.batch = a.batch;
  p.block_size = a.block_size;
  p.log2_bs = ilog2(a.block_size);
  p.max_blocks = a.max_blocks_per_seq;
  p.num_blocks = a.num_blocks;
  p.box_tokens = box_tokens;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  mla_decode_kernel<T, kBf16><<<2 * clusters, kThreads, MlaLayout::bytes(a.batch), a.stream>>>(
      qn, qr, cn, cr, p);
  return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

}  // namespace

int mla_decode_num_ctas(int num_ctas) {
  if (num_ctas > 0) return num_ctas & ~1;
  const int sms = device_sm_count();
  return sms > 1 ? sms & ~1 : 0;  // one CTA per SM, pairs
}

size_t mla_decode_workspace_bytes(int ctas) {
  const int clusters = ctas / 2;
  return mla_counter_bytes(clusters) +
         static_cast<size_t>(clusters) * 4 * kH * (kOutCols + 2) * sizeof(float);
}

kvc_status launch_mla_decode(const MlaArgs& a) {
  const int ctas = mla_decode_num_ctas(a.num_ctas);
  if (ctas < 2) return KVC_ERR_INVALID_ARG;
  if (a.workspace == nullptr || a.workspace_bytes < mla_decode_workspace_bytes(ctas))
    return KVC_ERR_WORKSPACE;
  return a.dtype == KVC_BF16 ? run_mla<__nv_bfloat16, true>(a, ctas / 2)
                             : run_mla<__half, false>(a, ctas / 2);
}

}  // namespace kvc
