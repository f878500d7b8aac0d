// MLA paged decode on the tcgen05 tensor cores.
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
//     token once);
//   * the CTA's 256 nope query columns live in tensor memory (the A operand
//     of S = Q K^T), which leaves shared memory for a 4-stage key ring;
//     rank 1's rope query columns stay in shared memory;
//   * each CTA computes a partial S (M 128, N 64 tokens) into tensor memory;
//     the partials are exchanged through distributed shared memory and
//     summed, so both CTAs hold the full S;
//   * both run the same online softmax (two threads per query row, log2
//     domain, O rescaled only when the running max grows by more than 2^8),
//     write P (bf16/fp16, 128-byte swizzled) to shared memory and compute
//     O_own += P V_own with V = their nope columns straight from the key
//     tile (MN-major operand), accumulating in tensor memory.
// The softmax runs one tile behind the exchange: while tile t's partial
// scores travel to the other CTA, the softmax of tile t-1 runs, and the
// tensor core computes S two tiles ahead of P V.
// Work: 64-token tiles of all sequences in one linear order, split evenly
// over the clusters (stream-K split-KV); pieces of split sequences leave
// partial states that a small second kernel (mla_merge_kernel) combines.
// Roles per CTA: warps 0-3 exchange the partial scores (one thread per
// query row), warps 4-11 run the softmax and the epilogue (two threads per
// row), warp 12 is the TMA producer, warp 13 the tcgen05 issuer (warp-
// convergent, one elected lane) and TMEM owner.  Warp w reads TMEM lanes 32*(w%4)...
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
constexpr int kOutCols = 256;       // output (and nope key) columns per CTA
constexpr int kQChunkBytes = kH * 128;     // [128 heads][64 elements]
constexpr int kKChunkBytes = kTok * 128;   // [64 tokens][64 elements]
constexpr int kStageChunks = 5;            // rank 1: 4 nope + rope
constexpr int kStageBytes = kStageChunks * kKChunkBytes;
constexpr int kStages = 4;
constexpr int kExchangeThreads = 128;   // warps 0-3
constexpr int kMathThreads = 256;       // warps 4-11, two threads per query row
constexpr int kProducerWarp = 12, kMmaWarp = 13;
constexpr int kThreads = kExchangeThreads + kMathThreads + 64;
constexpr int kMaxBatch = 1024;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows by > 2^8
// Work split: each sequence counts kSeqUnits units of work beyond its tiles,
// for its fixed costs (the query load and the epilogue of a piece), so that
// clusters whose shares touch more sequences get fewer tiles.  The units are
// virtual: no role visits them.  4 measured best of 0 to 10.
constexpr int kSeqUnits = 4;
// Bytes of one exchanged partial score: the scaled partial travels in fp32,
// so the full score each CTA forms is the fp32 sum of the two halves.
constexpr int kXElt = 4;
constexpr int kXBytes = kH * kTok * kXElt;

// TMEM columns: O (256 fp32), two S buffers (64 fp32 each), then the CTA's
// 256 nope query columns as packed 16-bit pairs (128 columns).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0, kTmemS0 = 256, kTmemS1 = 320, kTmemQ = 384;

struct MlaParams {
  void* out;
  const void* q_nope;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int* ws_plan;   // [batch + 1] tiles before each sequence (written by CTA 0)
  float* ws_o;    // [clusters][2][2][128][256]
  float* ws_ml;   // [clusters][2][2][128][2]
  uint32_t* err_flag;
  // Appending decode (all null for plain decode): the latent row of each
  // sequence's new token, new_nope [B, 512] and new_rope [B, 64], is written
  // at position seq_lens[b] - 1 into cache_nope / cache_rope by the CTAs that
  // then read that position, each rank the columns it loads; slot_out[b]
  // (nullable) gets its slot.
  const void* new_nope;
  const void* new_rope;
  void* cache_nope;
  void* cache_rope;
  int32_t* slot_out;
  int batch, block_size, log2_bs, max_blocks, num_blocks, box_tokens;
  float scale_log2;
};

constexpr int align_up_c(int x, int a) { return (x + a - 1) / a * a; }

// Shared memory (1024-aligned base), regions sized for rank 1.  The per-
// sequence plan (clamped lengths, prefix sums of tiles) is built in the P
// region at start and read only until every thread has found its first
// tile.
struct MlaLayout {
  static constexpr int kQr = 0;                                    // 16 KB
  static constexpr int kK = kQr + kQChunkBytes;                    // 4 x 40 KB
  static constexpr int kP = kK + kStages * kStageBytes;            // 16 KB
  static constexpr int kX = kP + kH * 128;                         // 32 KB
  static constexpr int kRed = kX + kXBytes;                        // [2][128] fp32
  static constexpr int kBar = kRed + 2 * kH * 4;
  static constexpr int kMisc = align_up_c(kBar + 19 * 8, 16);      // tmem slot, flags
  static constexpr int kEnd = kMisc + 32;
  static constexpr size_t kBytes = 1024 + static_cast<size_t>(kEnd);
  static constexpr int kPlanLens = kP;                             // lens[batch]
  static constexpr int kPlanCum = kP + kMaxBatch * 4;              // cum[batch + 1] (units)
  static constexpr int kPlanTiles = kPlanCum + (kMaxBatch + 1) * 4;  // tiles[batch + 1]
  static_assert(3 * kMaxBatch * 4 + 8 <= kH * 128, "plan fits the P region");
  static_assert(kBytes <= 232448, "fits the opt-in shared memory of one SM");
};

// q_full, q_free, k_full[4], k_empty[4], s_full[2], s_free[2], p_full,
// pv_done, x_full, x_empty, drain
enum Bar {
  kQFull = 0, kQFree = 1, kKFull0 = 2, kKEmpty0 = kKFull0 + kStages,
  kSFull0 = kKEmpty0 + kStages, kSFree0 = kSFull0 + 2, kPFull = kSFree0 + 2, kPVDone,
  kXFull, kXEmpty, kDrain, kNumBars
};
static_assert(kNumBars == 19, "barrier count used by the layout");

// Walks the linear tile order (b, j); len = clamped length of b, base = its
// first tile.  Past the first tile only the global lengths are read.
struct MlaCursor {
  int b, j, n, len;
  long long base;
  // The first tile at or after unit t of the work split (units: cum, with
  // kSeqUnits virtual units before each sequence's tiles; tiles: the plain
  // prefix sum of tiles).
  __device__ __forceinline__ void locate(long long t, const int* cum, const int* tiles,
                                         const int* lens, int B) {
    int lo = 0, hi = B - 1;  // largest b with cum[b] <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cum[mid] <= t) lo = mid; else hi = mid - 1;
    }
    b = lo;
    base = cum[b];
    n = tiles[b + 1] - tiles[b];
    len = lens[b];
    const long long off = t - base - kSeqUnits;
    j = off > 0 ? static_cast<int>(off) : 0;
  }
  __device__ __forceinline__ void advance(const int32_t* seq_lens, int cap, int B) {
    if (++j < n) return;
    j = 0;
    base += n;
    int L = 0;
    do {
      ++b;
      if (b < B) {
        L = __ldg(&seq_lens[b]);
        L = L < 0 ? 0 : (L > cap ? cap : L);
      }
    } while (b < B && L == 0);
    len = L;
    n = (L + kTok - 1) / kTok;
  }
  __device__ __forceinline__ bool last() const { return j == n - 1; }
};

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
// TMA loads: at each new sequence rank 1's rope query columns (after the
// tensor core has finished with the previous ones), then every tile's own
// key columns, one box per physical block per 64-wide chunk.
__device__ __forceinline__ void mla_producer(const MlaParams& p, const CUtensorMap* tm_qr,
                                             const CUtensorMap* tm_cn, const CUtensorMap* tm_cr,
                                             uint8_t* smem, uint64_t* bars,
                                             volatile int* abort_flag, MlaCursor cur, int n_it,
                                             int rank, int lane) {
  using L = MlaLayout;
  const int nq = rank ? 5 : 4;
  const int cap = p.max_blocks * p.block_size;
  const int nsub = kTok / p.box_tokens;
  const uint32_t box_bytes = static_cast<uint32_t>(p.box_tokens) * 128u;
  int seg = 0;
  for (int it = 0; it < n_it; ++it) {
    if (it == 0 || cur.j == 0) {
      const bool q_ok = seg == 0 || wait_cta(&bars[kQFree], (seg - 1) & 1, abort_flag, p.err_flag);
      if (lane == 0) {
        if (rank && q_ok) {
          mbar_arrive_expect_tx(&bars[kQFull], kQChunkBytes);
          tma_load_3d(smem + L::kQr, tm_qr, &bars[kQFull], 0, 0, cur.b);
        } else {
          mbar_arrive(&bars[kQFull]);
        }
      }
      ++seg;
    }
    const int stage = it % kStages;
    const uint32_t phase = static_cast<uint32_t>(it / kStages) & 1u;
    const int tok = cur.j * kTok + lane * p.box_tokens;
    if (p.new_nope != nullptr && cur.last()) {
      // The sequence's last tile holds its new token: write the columns this
      // rank loads (rank 0: nope 0..255; rank 1: nope 256..511 and rope), 16
      // bytes per lane, make them visible to the TMA unit, then load the tile
      // as usual.  No other CTA reads them.
      const int pos = cur.len - 1;
      const int pbn = __ldg(&p.block_table[static_cast<long long>(cur.b) * p.max_blocks +
                                           (pos >> p.log2_bs)]);
      if (pbn >= 0 && pbn < p.num_blocks) {
        const long long row = static_cast<long long>(pbn) * p.block_size + (pos & (p.block_size - 1));
        const uint4* src = reinterpret_cast<const uint4*>(p.new_nope) +
                           static_cast<long long>(cur.b) * (kNope / 8) + rank * (kOutCols / 8);
        uint4* dst = reinterpret_cast<uint4*>(p.cache_nope) + row * (kNope / 8) + rank * (kOutCols / 8);
        dst[lane] = __ldg(src + lane);  // 32 lanes x 8 elements = the rank's 256 columns
        if (rank == 1 && lane < kRope / 8)
          reinterpret_cast<uint4*>(p.cache_rope)[row * (kRope / 8) + lane] =
              __ldg(reinterpret_cast<const uint4*>(p.new_rope) +
                    static_cast<long long>(cur.b) * (kRope / 8) + lane);
        asm volatile("fence.proxy.async.global;" ::: "memory");
        if (rank == 0 && lane == 0 && p.slot_out) p.slot_out[cur.b] = static_cast<int32_t>(row);
      } else if (lane == 0) {
        set_flag(p.err_flag, KVC_FLAG_BLOCK_ID_RANGE);
        if (rank == 0 && p.slot_out) p.slot_out[cur.b] = -1;
      }
      __syncwarp();
      if (lane == 0) asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    int pb = -1;
    if (lane < nsub && tok < cur.len)
      pb = __ldg(&p.block_table[static_cast<long long>(cur.b) * p.max_blocks + (tok >> p.log2_bs)]);
    const bool ok = wait_cta(&bars[kKEmpty0 + stage], phase ^ 1u, abort_flag, p.err_flag);
    bool valid = false;
    if (lane < nsub && tok < cur.len) {
      if (pb < 0 || pb >= p.num_blocks) set_flag(p.err_flag, KVC_FLAG_BLOCK_ID_RANGE);
      else valid = ok;
    }
    const uint32_t nvalid = __popc(__ballot_sync(0xffffffffu, valid));
    if (lane == 0) mbar_arrive_expect_tx(&bars[kKFull0 + stage], nvalid * box_bytes * nq);
    __syncwarp();
    if (valid) {
      uint8_t* dst = smem + L::kK + stage * kStageBytes + lane * box_bytes;
      const int in_blk = tok & (p.block_size - 1);
      for (int c = 0; c < 4; ++c)
        tma_load_3d(dst + c * kKChunkBytes, tm_cn, &bars[kKFull0 + stage], (rank * 4 + c) * 64,
                    in_blk, pb);
      if (rank) tma_load_3d(dst + 4 * kKChunkBytes, tm_cr, &bars[kKFull0 + stage], 0, in_blk, pb);
    }
    cur.advance(p.seq_lens, cap, p.batch);
  }
}

// --------------------------------------------------------------- tcgen05
// S = Q K^T for one tile: 16 K-steps over the nope columns with A (the
// query) in tensor memory, then on rank 1 four K-steps over the rope
// columns with A in shared memory.  Fully unrolled from base descriptors.
template <bool kWithRope>
__device__ __forceinline__ void mla_issue_s(uint32_t d, uint32_t q_tmem, uint64_t qr0, uint64_t k0,
                                            uint32_t idesc, uint32_t leader) {
#pragma unroll
  for (int k = 0; k < 16; ++k)
    umma_ts_e(d, q_tmem + k * 8, desc_advance(k0, (k >> 2) * kKChunkBytes + (k & 3) * 32), idesc,
              k != 0, leader);
  if (kWithRope) {
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      umma_ss_e(d, desc_advance(qr0, kk * 32), desc_advance(k0, 4 * kKChunkBytes + kk * 32), idesc,
                1u, leader);
  }
}

// The MMA warp, all lanes converged (one elected lane issues; see
// elect_one_sync).  S(t) and P V(t) are issued as soon as their inputs are ready,
// whichever comes first (P V first when both are): S(t) needs its key stage,
// a free S buffer and the sequence's query; P V(t) needs P(t).  So a key tile
// still in flight never holds back the P V of an earlier tile.  A stall of
// kWaitLimitNs without progress sets KVC_FLAG_WAIT_TIMEOUT and aborts.
template <bool kBf16>
__device__ __forceinline__ void mla_mma(const MlaParams& p, uint8_t* smem, uint64_t* bars,
                                        volatile int* abort_flag, uint32_t tmem, MlaCursor cs,
                                        int n_it, int rank, uint32_t leader) {
  using L = MlaLayout;
  const int cap = p.max_blocks * p.block_size;
  const uint32_t idesc_s = umma_idesc_f16(kBf16, kH, kTok, 0, 0);
  const uint32_t idesc_o = umma_idesc_f16(kBf16, kH, kOutCols, 0, 1);
  const uint64_t qr0 = umma_desc_sw128(smem_u32(smem + L::kQr), 16, 1024);
  const uint64_t k0 = umma_desc_sw128(smem_u32(smem + L::kK), 16, 1024);
  const uint64_t p0 = umma_desc_sw128(smem_u32(smem + L::kP), 16, 1024);
  // V = the first four chunks of a stage, MN-major: next 64 columns 8 KB on.
  const uint64_t v0 = umma_desc_sw128(smem_u32(smem + L::kK), kKChunkBytes, 1024);
  int seg_s = -1, ns = 0, npv = 0;
  uint32_t first_bits = 0;  // bit (t & 3): tile t starts a sequence's share
  unsigned long long t_prog = global_timer_ns();
  int idle = 0;
  while (npv < n_it) {
    if (*abort_flag) return;
    bool progress = false;
    if (npv < ns && mbar_test_wait(&bars[kPFull], npv & 1)) {
      tc_fence_after();
      const int stage = npv % kStages;
      const uint64_t v_st = desc_advance(v0, stage * kStageBytes);
      umma_ss_e(tmem + kTmemO, p0, v_st, idesc_o, ((first_bits >> (npv & 3)) & 1u) ^ 1u, leader);
#pragma unroll
      for (int ks = 1; ks < kTok / 16; ++ks)
        umma_ss_e(tmem + kTmemO, desc_advance(p0, ks * 32), desc_advance(v_st, ks * 16 * 128),
                  idesc_o, 1u, leader);
      umma_commit_e(&bars[kPVDone], leader);
      umma_commit_e(&bars[kKEmpty0 + stage], leader);
      ++npv;
      progress = true;
    }
    if (ns < n_it && ns < npv + 4) {
      const bool first = ns == 0 || cs.j == 0;
      const int seg = first ? seg_s + 1 : seg_s;
      const int stage = ns % kStages, sb = ns & 1;
      if (mbar_test_wait(&bars[kKFull0 + stage], static_cast<uint32_t>(ns / kStages) & 1u) &&
          mbar_test_wait(&bars[kSFree0 + sb], ((ns >> 1) & 1) ^ 1) &&
          mbar_test_wait(&bars[kQFull], seg & 1)) {
        tc_fence_after();
        const bool last = ns == n_it - 1 || cs.last();
        seg_s = seg;
        first_bits = (first_bits & ~(1u << (ns & 3))) | (first ? 1u << (ns & 3) : 0u);
        const uint32_t d = tmem + (sb ? kTmemS1 : kTmemS0);
        const uint64_t k_st = desc_advance(k0, stage * kStageBytes);
        if (rank) mla_issue_s<true>(d, tmem + kTmemQ, qr0, k_st, idesc_s, leader);
        else mla_issue_s<false>(d, tmem + kTmemQ, qr0, k_st, idesc_s, leader);
        umma_commit_e(&bars[kSFull0 + sb], leader);
        if (last) umma_commit_e(&bars[kQFree], leader);
        cs.advance(p.seq_lens, cap, p.batch);
        ++ns;
        progress = true;
      }
    }
    if (progress) {
      idle = 0;
      t_prog = 0;
    } else if (++idle >= 64) {
      idle = 0;
      const unsigned long long now = global_timer_ns();
      if (t_prog == 0) {
        t_prog = now;
      } else if (now - t_prog > kWaitLimitNs) {
        set_flag(p.err_flag, KVC_FLAG_WAIT_TIMEOUT);
        *abort_flag = 1;
        return;
      }
    }
  }
}

// ----------------------------------------------------------- epilogue
// End of one sequence's share for query row `row`, column half `h` (128 of
// this rank's 256 output columns).  The two halves' partial sums l are added
// first.  A sequence the share holds whole is normalised and written out; a
// piece of a split sequence publishes its partial state (m, l, unnormalised
// O) in workspace slot (cluster, slot, rank) for mla_merge_kernel.  Each
// warp passes its 32 rows through `stg` (2 KB of shared memory: 32 rows of
// 64 bytes, 16-byte chunk q of row r at r*64 + (q ^ ((r >> 1) & 3))*16, so
// neither the row-wise writes nor the chunk-wise reads conflict), so that a
// store instruction writes 8 rows x 64 contiguous bytes rather than 32 rows
// x 16 bytes.
template <typename T>
__device__ __noinline__ void mla_finish(const MlaParams& p, uint32_t o_taddr, int row, int h,
                                        int b, bool complete, int cl, int slot, int rank,
                                        float m_used, float l_half, float* red, uint8_t* stg) {
  named_bar_sync(1, kMathThreads);
  red[h * kH + row] = l_half;
  named_bar_sync(1, kMathThreads);
  const float l = red[row] + red[kH + row];
  const int lane = row & 31, wrow0 = row & ~31;
  // This thread's 64 bytes -> its staging row; then chunk i of the read-back
  // pattern (row i*8 + lane/4, 16-byte piece lane%4).
  auto put = [&](const uint32_t* w) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<uint4*>(stg + lane * 64 + ((q ^ ((lane >> 1) & 3)) * 16)) =
          make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    __syncwarp();
  };
  auto get = [&](int i) -> uint4 {
    const int r = i * 8 + (lane >> 2), q = lane & 3;
    return *reinterpret_cast<const uint4*>(stg + r * 64 + ((q ^ ((r >> 1) & 3)) * 16));
  };
  if (complete) {
    T* out = static_cast<T*>(p.out) + (static_cast<long long>(b) * kH + wrow0) * kNope +
             rank * kOutCols + h * 128;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    for (int c = 0; c < 8; c += 2) {  // two loads in flight per wait
      float v[32];
      tmem_ld16(o_taddr + c * 16, v);
      tmem_ld16(o_taddr + c * 16 + 16, v + 16);
      tmem_wait_ld();
      uint32_t w[16];
      float ra, rb;
#pragma unroll
      for (int k = 0; k < 16; ++k) w[k] = Pack<T>::run(v[2 * k] * inv, v[2 * k + 1] * inv, ra, rb);
      put(w);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = i * 8 + (lane >> 2), q = lane & 3;
        *reinterpret_cast<uint4*>(out + r * kNope + c * 16 + q * 8) = get(i);
      }
      __syncwarp();
    }
    return;
  }
  float* wbase = p.ws_o +
                 (((static_cast<long long>(cl) * 2 + slot) * 2 + rank) * kH + wrow0) * kOutCols +
                 h * 128;
  for (int c = 0; c < 8; c += 2) {  // two loads in flight per wait
    float v[32];
    tmem_ld16(o_taddr + c * 16, v);
    tmem_ld16(o_taddr + c * 16 + 16, v + 16);
    tmem_wait_ld();
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {  // 16 fp32 columns = 64 bytes per row
      put(reinterpret_cast<const uint32_t*>(v + hf * 16));
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = i * 8 + (lane >> 2), q = lane & 3;
        *reinterpret_cast<uint4*>(wbase + r * kOutCols + c * 16 + hf * 16 + q * 4) = get(i);
      }
      __syncwarp();
    }
  }
  if (h == 0) {
    const long long wrow = ((static_cast<long long>(cl) * 2 + slot) * 2 + rank) * kH + row;
    *reinterpret_cast<float2*>(p.ws_ml + wrow * 2) = make_float2(m_used, l);
  }
}

// ------------------------------------------------------------- exchange
// This CTA's 256 nope query columns of sequence b, row `row` (128 packed
// TMEM columns), loaded in two halves.
template <typename T>
__device__ __forceinline__ void mla_load_q(const MlaParams& p, uint32_t lane_base, int b, int row,
                                           int rank) {
  const uint4* src = reinterpret_cast<const uint4*>(
      static_cast<const T*>(p.q_nope) + (static_cast<long long>(b) * kH + row) * kNope +
      rank * kOutCols);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint4 v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __ldg(src + half * 16 + i);
#pragma unroll
    for (int c = 0; c < 4; ++c)
      tmem_st16_u32(lane_base + kTmemQ + half * 64 + c * 16,
                    reinterpret_cast<const uint32_t*>(v + 4 * c));
  }
  tmem_wait_st();
}

// Warps 0-3, thread `row` = query head.  Per tile: this CTA's partial scores
// (TMEM), scaled to the log2 domain (fp32), go to the other CTA as st.async
// stores that complete its x_full transaction count, once the other CTA has
// freed its X buffer (x_empty, a relaxed arrive from its math warps): 256
// bytes per query head and tile, chunk q holding tokens 4q .. 4q+3.
// These warps also load each sequence's query into TMEM.
template <typename T>
__device__ __forceinline__ void mla_exchange(const MlaParams& p, uint8_t* smem, uint64_t* bars,
                                             volatile int* abort_flag, uint32_t tmem, MlaCursor cx,
                                             int n_it, int rank, int row) {
  using L = MlaLayout;
  const int cap = p.max_blocks * p.block_size;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(row & ~31) << 16);
  const uint32_t peer = static_cast<uint32_t>(rank ^ 1);
  const uint32_t x_peer = map_to_rank(smem_u32(smem + L::kX), peer);
  const uint32_t xfull_peer = map_to_rank(smem_u32(&bars[kXFull]), peer);
  int seg_x = 0;

  mla_load_q<T>(p, lane_base, cx.b, row, rank);  // tensor memory is fresh
  tc_fence_before();
  mbar_arrive(&bars[kQFull]);

  for (int it = 0; it < n_it; ++it) {
    const int sb = it & 1;
    const uint32_t s_col = lane_base + (sb ? kTmemS1 : kTmemS0);
    float so[kTok];
    wait_cta(&bars[kSFull0 + sb], (it >> 1) & 1, abort_flag, p.err_flag);
    tc_fence_after();
#pragma unroll
    for (int c = 0; c < kTok / 16; ++c) tmem_ld16(s_col + c * 16, so + c * 16);
    tmem_wait_ld();
    tc_fence_before();
    mbar_arrive(&bars[kSFree0 + sb]);
#pragma unroll
    for (int k = 0; k < kTok; ++k) so[k] *= p.scale_log2;
    wait_peer(&bars[kXEmpty], (it & 1) ^ 1, abort_flag, p.err_flag);
#pragma unroll
    for (int q = 0; q < kTok / 4; ++q)  // chunk q: tokens 4q .. 4q+3
      st_async_cluster_v4(x_peer + (q * kH + row) * 16,
                          make_float4(so[4 * q], so[4 * q + 1], so[4 * q + 2], so[4 * q + 3]),
                          xfull_peer);
    // Tile it+1 starts the next sequence: its query replaces this one (S(it)
    // complete => every S of this sequence is done).  Its rows are first
    // fetched into L2, so the load after q_free does not wait on HBM.
    if (it + 1 < n_it && cx.last()) {
      {
        MlaCursor nx = cx;
        nx.advance(p.seq_lens, cap, p.batch);
        const char* q = reinterpret_cast<const char*>(
            static_cast<const T*>(p.q_nope) + (static_cast<long long>(nx.b) * kH + row) * kNope +
            rank * kOutCols);
#pragma unroll
        for (int i = 0; i < kOutCols * static_cast<int>(sizeof(T)) / 128; ++i)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(q + i * 128));
      }
      wait_cta(&bars[kQFree], seg_x & 1, abort_flag, p.err_flag);
      tc_fence_after();
      MlaCursor nx = cx;
      nx.advance(p.seq_lens, cap, p.batch);
      mla_load_q<T>(p, lane_base, nx.b, row, rank);
      tc_fence_before();
      mbar_arrive(&bars[kQFull]);
      ++seg_x;
    }
    cx.advance(p.seq_lens, cap, p.batch);
  }
}

// ----------------------------------------------------------------- math
// Warps 4-11, thread (row, h) = query head `row`, tokens and output columns
// of half h: online softmax in the log2 domain (O rescaled only when the
// running max grows by more than 2^kRescaleThreshold; the two halves of a
// row share their maxima through shared memory), P (bf16/fp16, K-major,
// 128-byte swizzle) to shared memory, then the end-of-share epilogue.
template <typename T>
__device__ __forceinline__ void mla_math(const MlaParams& p, uint8_t* smem, uint64_t* bars,
                                         volatile int* abort_flag, uint32_t tmem, MlaCursor cm,
                                         int n_it, int cl, int rank, int row, int h) {
  using L = MlaLayout;
  const int cap = p.max_blocks * p.block_size;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(row & ~31) << 16);
  float* red = reinterpret_cast<float*>(smem + L::kRed);
  const uint4* x_mine = reinterpret_cast<const uint4*>(smem + L::kX);
  const uint32_t xempty_peer = map_to_rank(smem_u32(&bars[kXEmpty]), static_cast<uint32_t>(rank ^ 1));
  const bool elected = row == 0 && h == 0;
  float m_used = -INFINITY, l = 0.f;
  int seg_first_j = cm.j, slot = 0;
  for (int it = 0; it < n_it; ++it) {
    const int sb = it & 1;
    const bool first = it == 0 || cm.j == 0;
    const bool last = it == n_it - 1 || cm.last();
    if (first) {
      m_used = -INFINITY;
      l = 0.f;
      seg_first_j = cm.j;
    }
    // Scores of this thread's 32 tokens in the log2 domain: own partial
    // (TMEM, fp32) times scale_log2 plus the other CTA's (X, already scaled,
    // fp32); then both buffers are released.
    float s[32];
    wait_cta(&bars[kSFull0 + sb], (it >> 1) & 1, abort_flag, p.err_flag);
    tc_fence_after();
    tmem_ld16(lane_base + (sb ? kTmemS1 : kTmemS0) + h * 32, s);
    tmem_ld16(lane_base + (sb ? kTmemS1 : kTmemS0) + h * 32 + 16, s + 16);
    tmem_wait_ld();
    tc_fence_before();
    mbar_arrive(&bars[kSFree0 + sb]);
    wait_peer(&bars[kXFull], it & 1, abort_flag, p.err_flag);
    const float2 sl2 = make_float2(p.scale_log2, p.scale_log2);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const uint4 v = x_mine[(h * 8 + q) * kH + row];
      const float2 o01 = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
      const float2 o23 = make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
      const int k = 4 * q;
      const float2 t0 = fma2(make_float2(s[k], s[k + 1]), sl2, o01);
      const float2 t1 = fma2(make_float2(s[k + 2], s[k + 3]), sl2, o23);
      s[k] = t0.x;
      s[k + 1] = t0.y;
      s[k + 2] = t1.x;
      s[k + 3] = t1.y;
    }
    const int tile_valid = min(kTok, cm.len - cm.j * kTok);
    const int valid = tile_valid - h * 32;  // of this thread's 32 tokens
    // Row max of the scaled scores; tokens past the sequence only in a tail
    // tile.
    float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    if (valid >= 32) {
#pragma unroll
      for (int k = 0; k < 32; ++k) mx4[k & 3] = fmaxf(mx4[k & 3], s[k]);
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        s[k] = k < valid ? s[k] : -INFINITY;
        mx4[k & 3] = fmaxf(mx4[k & 3], s[k]);
      }
    }
    red[h * kH + row] = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
    named_bar_sync(3, kMathThreads);  // also: every thread has read X
    if (elected) {
      // The next tile's scores arrive as 32 KB of transactions on x_full.
      if (it + 1 < n_it) mbar_arrive_expect_tx(&bars[kXFull], kXBytes);
      mbar_arrive_cluster_relaxed(xempty_peer);
    }
    const float mx = fmaxf(red[row], red[kH + row]);  // same order in both halves
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
    // p = 2^(s - m_used) (s already scaled); l adds the exponentials before
    // rounding (P itself is rounded to T for the tensor core).
    const float neg_m = m_used == -INFINITY ? 0.f : -m_used;
    const float2 nm2 = make_float2(neg_m, neg_m);
    uint32_t pk[16];
    float2 ps2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const float2 x = add2(make_float2(s[2 * k], s[2 * k + 1]), nm2);
      const float2 e = make_float2(fast_exp2(x.x), fast_exp2(x.y));
      pk[k] = pack_pair<T>(e.x, e.y);
      ps2[k & 1] = add2(ps2[k & 1], e);
    }
    const float2 pst = add2(ps2[0], ps2[1]);
    l = l * corr + (pst.x + pst.y);
    if (it > 0) {  // P V of the previous tile must be done before P and O are touched
      wait_cta(&bars[kPVDone], (it - 1) & 1, abort_flag, p.err_flag);
      tc_fence_after();
    }
    if (__any_sync(0xffffffffu, rescale)) {
      for (int c = 0; c < 8; ++c) {
        float v[16];
        tmem_ld16(lane_base + kTmemO + h * 128 + c * 16, v);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] *= corr;
        tmem_st16(lane_base + kTmemO + h * 128 + c * 16, v);
      }
      tmem_wait_st();
    }
    // P row half -> shared memory; the value rows past the sequence are
    // zeroed so stale contents cannot reach P V.
    uint8_t* pptr = smem + L::kP;
#pragma unroll
    for (int ch = 0; ch < 4; ++ch)
      *reinterpret_cast<uint4*>(pptr + swz128(row, h * 4 + ch)) =
          make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
    if (tile_valid < kTok) {
      uint8_t* kst = smem + L::kK + (it % kStages) * kStageBytes;
      const int n16 = (kTok - tile_valid) * 4 * 8;
      for (int e = h * kH + row; e < n16; e += kMathThreads) {
        const int r = tile_valid + e / 32, c = (e % 32) / 8, q = e % 8;
        *reinterpret_cast<uint4*>(kst + c * kKChunkBytes + r * 128 + q * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    mbar_arrive(&bars[kPFull]);
    if (last) {  // end of this sequence's share
      wait_cta(&bars[kPVDone], it & 1, abort_flag, p.err_flag);
      tc_fence_after();
      // P V is done, so the P buffer is free: 2 KB of it stage each warp's rows.
      mla_finish<T>(p, lane_base + kTmemO + h * 128, row, h, cm.b, seg_first_j == 0 && cm.last(),
                    cl, slot, rank, m_used, l, red, smem + L::kP + (h * 4 + (row >> 5)) * 2048);
      tc_fence_before();
      slot = 1;
    }
    cm.advance(p.seq_lens, cap, p.batch);
  }
}

template <typename T, bool kBf16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tm_qr,
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
  int* lens = reinterpret_cast<int*>(smem + L::kPlanLens);
  int* cum = reinterpret_cast<int*>(smem + L::kPlanCum);
  int* tiles = reinterpret_cast<int*>(smem + L::kPlanTiles);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int rank = static_cast<int>(cluster_ctarank());
  const int cl = static_cast<int>(blockIdx.x >> 1), P = static_cast<int>(gridDim.x >> 1);
  const int B = p.batch, cap = p.max_blocks * p.block_size;

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t c = 1;
      if (i == kQFull) c = 1 + kExchangeThreads;
      if (i == kSFree0 || i == kSFree0 + 1) c = kExchangeThreads + kMathThreads;
      if (i == kPFull) c = kMathThreads;
      mbar_init(&bars[i], c);
    }
    *abort_flag = 0;
    fence_barrier_init();
    // The first tile's scores from the other CTA arrive as 16 KB of
    // transactions on x_full (harmless if this cluster has no tile).
    mbar_arrive_expect_tx(&bars[kXFull], kXBytes);
  }
  uint32_t leader = 0;  // the MMA warp's issuing lane
  if (warp == kMmaWarp) {
    tmem_alloc(tslot, kTmemCols);
    leader = elect_one_sync();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tmap(&tm_qr);
    prefetch_tmap(&tm_cn);
    prefetch_tmap(&tm_cr);
  }
  for (int i = tid; i < B; i += kThreads) lens[i] = sched::clamp_len(p.seq_lens[i], cap, p.err_flag);
  __syncthreads();
  if (warp == 0) sched::plan_tiles(lens, cum, B, kTok, lane, kSeqUnits);
  if (warp == 1) sched::plan_tiles(lens, tiles, B, kTok, lane);
  tc_fence_before();
  __syncthreads();
  if (blockIdx.x == 0)  // the plan, for the merge of split sequences
    for (int i = tid; i <= B; i += kThreads) p.ws_plan[i] = cum[i];
  tc_fence_after();
  cluster_sync();  // both CTAs' barriers exist before any remote arrive

  const uint32_t tmem = *tslot;
  const long long N = cum[B];
  const long long tb = sched::share_begin(cl, N, P), te = sched::share_begin(cl + 1, N, P);
  {  // sequences with no cached token: rows of zeros (this rank's columns)
     // and, when appending, no slot (-1): there is no new token to write
    T* out = static_cast<T*>(p.out);
    for (int b = cl; b < B; b += P)
      if (lens[b] == 0) {
        for (int e = tid; e < kH * kOutCols; e += kThreads)
          out[(static_cast<long long>(b) * kH + e / kOutCols) * kNope + rank * kOutCols +
              e % kOutCols] = Pack<T>::cvt(0.f);
        if (tid == 0 && rank == 0 && p.slot_out) p.slot_out[b] = -1;
      }
  }
  // Tiles of units [0, x): the tiles of the sequences before the one holding
  // unit x, plus those of its tiles that lie before x.
  auto tiles_before = [&](long long x) -> long long {
    if (x >= N) return tiles[B];
    int lo = 0, hi = B - 1;  // largest b with cum[b] <= x
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cum[mid] <= x) lo = mid; else hi = mid - 1;
    }
    const long long in = x - cum[lo] - kSeqUnits, nb = tiles[lo + 1] - tiles[lo];
    return tiles[lo] + (in < 0 ? 0 : (in > nb ? nb : in));
  };
  const int n_it = static_cast<int>(tiles_before(te) - tiles_before(tb));
  MlaCursor cur;
  if (n_it > 0) cur.locate(tb, cum, tiles, lens, B);
  __syncthreads();  // the plan (in the P region) is not read past this point
  if (n_it > 0) {
    if (warp < 4) {
      mla_exchange<T>(p, smem, bars, abort_flag, tmem, cur, n_it, rank, tid);
    } else if (warp < 12) {
      mla_math<T>(p, smem, bars, abort_flag, tmem, cur, n_it, cl, rank, (warp & 3) * 32 + lane,
                  (warp - 4) >> 2);
    } else if (warp == kProducerWarp) {
      mla_producer(p, &tm_qr, &tm_cn, &tm_cr, smem, bars, abort_flag, cur, n_it, rank, lane);
      // Every copy issued must land before shared memory can be released.
      for (int it = max(0, n_it - kStages); it < n_it; ++it)
        mbar_wait_bounded(&bars[kKFull0 + it % kStages], static_cast<uint32_t>(it / kStages) & 1u,
                          p.err_flag);
    } else {
      mla_mma<kBf16>(p, smem, bars, abort_flag, tmem, cur, n_it, rank, leader);
    }
  }
  // Teardown: all tensor-core work done, TMEM freed, and neither CTA leaves
  // while its partner may still write into its shared memory.
  if (warp == kMmaWarp) {
    __syncwarp();
    umma_commit_e(&bars[kDrain], leader);
    mbar_wait_bounded(&bars[kDrain], 0, p.err_flag);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_sync();
}

// ------------------------------------------------------- split merge
// One CTA per (sequence, rank, 16 query heads); 16 threads per head, each
// owning 16 adjacent output columns, so a warp reads and writes whole rows.
// Sequences split over several clusters combine their partial states,
//   out = sum_i 2^(m_i - M) O_i / sum_i 2^(m_i - M) l_i,   M = max_i m_i,
// over the pieces in cluster order (deterministic).  Up to four pieces are
// loaded at once (one memory round trip); more go through a loop.  Sequences
// held whole by one cluster were written by the decode kernel and are skipped.
struct MlaMergeParams {
  void* out;
  const int* plan;
  const float* ws_o;
  const float* ws_ml;
  int batch, clusters;
};

constexpr int kMergeRows = 16;                       // query heads per CTA
constexpr int kMergeThreads = kMergeRows * 16;       // 16 threads per head
constexpr int kMergeFast = 4;

template <typename T>
__global__ void __launch_bounds__(kMergeThreads) mla_merge_kernel(
    const __grid_constant__ MlaMergeParams m) {
  const int b = blockIdx.x;
  const int rank = blockIdx.y / (kH / kMergeRows);
  const int row = (blockIdx.y % (kH / kMergeRows)) * kMergeRows + threadIdx.x / 16;
  const int col0 = (threadIdx.x % 16) * 16;
  // The plan counts kSeqUnits virtual units before each sequence's tiles.
  if (m.plan[b + 1] == m.plan[b]) return;
  const long long seg0 = m.plan[b] + kSeqUnits, n = m.plan[b + 1] - seg0;
  const long long N = m.plan[m.batch];
  const int P = m.clusters;
  const int cfirst = sched::share_of(seg0, N, P), clast = sched::share_of(seg0 + n - 1, N, P);
  if (cfirst == clast) return;
  // The sequence is the first piece of cluster cfirst iff its share starts
  // within the sequence's units (virtual or not).
  const int slot0 = sched::share_begin(cfirst, N, P) >= m.plan[b] ? 0 : 1;
  auto piece_row = [&](int cc) -> long long {
    return ((static_cast<long long>(cc) * 2 + (cc == cfirst ? slot0 : 0)) * 2 + rank) * kH + row;
  };
  long long rows[kMergeFast];
  int np = 0;
  for (int cc = cfirst; cc <= clast; ++cc)
    if (sched::share_begin(cc, N, P) < sched::share_begin(cc + 1, N, P)) {
      if (np < kMergeFast) rows[np] = piece_row(cc);
      ++np;
    }
  float acc[16];
#pragma unroll
  for (int k = 0; k < 16; ++k) acc[k] = 0.f;
  float Ls = 0.f;
  if (np <= kMergeFast) {
    float2 ml[kMergeFast];
    float4 v[kMergeFast][4];
#pragma unroll
    for (int i = 0; i < kMergeFast; ++i) {
      if (i < np) {
        ml[i] = __ldcg(reinterpret_cast<const float2*>(m.ws_ml + rows[i] * 2));
        const float4* src = reinterpret_cast<const float4*>(m.ws_o + rows[i] * kOutCols + col0);
#pragma unroll
        for (int k = 0; k < 4; ++k) v[i][k] = __ldcg(src + k);
      } else {
        ml[i] = make_float2(-INFINITY, 0.f);
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int i = 0; i < kMergeFast; ++i) M = fmaxf(M, ml[i].x);
#pragma unroll
    for (int i = 0; i < kMergeFast; ++i) {
      if (i < np) {
        const float f = fast_exp2(ml[i].x - M);
        Ls += f * ml[i].y;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          acc[4 * k] += f * v[i][k].x;
          acc[4 * k + 1] += f * v[i][k].y;
          acc[4 * k + 2] += f * v[i][k].z;
          acc[4 * k + 3] += f * v[i][k].w;
        }
      }
    }
  } else {  // many pieces: one at a time
    float M = -INFINITY;
    for (int cc = cfirst; cc <= clast; ++cc)
      if (sched::share_begin(cc, N, P) < sched::share_begin(cc + 1, N, P))
        M = fmaxf(M, __ldcg(m.ws_ml + piece_row(cc) * 2));
    for (int cc = cfirst; cc <= clast; ++cc) {
      if (sched::share_begin(cc, N, P) >= sched::share_begin(cc + 1, N, P)) continue;
      const long long r = piece_row(cc);
      const float2 ml = __ldcg(reinterpret_cast<const float2*>(m.ws_ml + r * 2));
      const float f = fast_exp2(ml.x - M);
      Ls += f * ml.y;
      const float4* src = reinterpret_cast<const float4*>(m.ws_o + r * kOutCols + col0);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 x = __ldcg(src + k);
        acc[4 * k] += f * x.x;
        acc[4 * k + 1] += f * x.y;
        acc[4 * k + 2] += f * x.z;
        acc[4 * k + 3] += f * x.w;
      }
    }
  }
  const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
  T* out = static_cast<T*>(m.out) + (static_cast<long long>(b) * kH + row) * kNope +
           rank * kOutCols + col0;
  uint32_t w[8];
  float ra, rb;
#pragma unroll
  for (int k = 0; k < 8; ++k) w[k] = Pack<T>::run(acc[2 * k] * inv, acc[2 * k + 1] * inv, ra, rb);
  *reinterpret_cast<uint4*>(out) = make_uint4(w[0], w[1], w[2], w[3]);
  *reinterpret_cast<uint4*>(out + 8) = make_uint4(w[4], w[5], w[6], w[7]);
}

}  // namespace

namespace {

// Workspace: the plan ([kMaxBatch + 1] int, padded to 256 B), then the
// partial states of [clusters][2 slots][2 ranks] pieces.
constexpr size_t kPlanBytes = ((kMaxBatch + 1) * sizeof(int) + 255) & ~static_cast<size_t>(255);

template <typename T, bool kBf16>
void mla_set_smem_attr() {
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(mla_decode_kernel<T, kBf16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         static_cast<int>(MlaLayout::kBytes));
  });
}

// Clusters of two CTAs that can be resident at once on the current device.
// A GPC with an odd number of free SMs leaves one idle, so this can be below
// SMs / 2; launching more would run the extra clusters as a second wave.
int mla_resident_clusters() {
  static std::mutex mu;
  static int cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (cache[dev] > 0) return cache[dev];
  const int sms = device_sm_count();
  mla_set_smem_attr<__nv_bfloat16, true>();
  mla_set_smem_attr<__half, false>();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = MlaLayout::kBytes;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, mla_decode_kernel<__nv_bfloat16, true>, &cfg) !=
          cudaSuccess ||
      n <= 0) {
    cudaGetLastError();
    n = sms / 2;
  }
  cache[dev] = n < sms / 2 ? n : sms / 2;
  return cache[dev];
}

template <typename T, bool kBf16>
kvc_status run_mla(const MlaArgs& a, int clusters) {
  mla_set_smem_attr<T, kBf16>();
  const int box_tokens = a.block_size < kTok ? a.block_size : kTok;
  CUtensorMap qr, cn, cr;
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
  if (!encode_tmap_16bit(&qr, a.dtype, 3, a.q_rope, qr_dims, qr_str, qbox, true) ||
      !encode_tmap_16bit(&cn, a.dtype, 3, a.cache_nope, cn_dims, cn_str, cbox, true) ||
      !encode_tmap_16bit(&cr, a.dtype, 3, a.cache_rope, cr_dims, cr_str, cbox, true))
    return KVC_ERR_CUDA;
  MlaParams p;
  p.out = a.out;
  p.q_nope = a.q_nope;
  p.block_table = a.block_table;
  p.seq_lens = a.seq_lens;
  p.ws_plan = static_cast<int*>(a.workspace);
  p.ws_o = reinterpret_cast<float*>(static_cast<char*>(a.workspace) + kPlanBytes);
  p.ws_ml = p.ws_o + static_cast<size_t>(clusters) * 4 * kH * kOutCols;
  p.err_flag = a.err_flag;
  p.batch = a.batch;
  p.block_size = a.block_size;
  p.log2_bs = ilog2(a.block_size);
  p.max_blocks = a.max_blocks_per_seq;
  p.num_blocks = a.num_blocks;
  p.box_tokens = box_tokens;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.new_nope = a.new_nope;
  p.new_rope = a.new_rope;
  p.cache_nope = const_cast<void*>(a.cache_nope);
  p.cache_rope = const_cast<void*>(a.cache_rope);
  p.slot_out = a.slot_out;
  mla_decode_kernel<T, kBf16><<<2 * clusters, kThreads, MlaLayout::kBytes, a.stream>>>(qr, cn, cr,
                                                                                       p);
  if (cudaGetLastError() != cudaSuccess) return KVC_ERR_CUDA;
  MlaMergeParams mp;
  mp.out = a.out;
  mp.plan = p.ws_plan;
  mp.ws_o = p.ws_o;
  mp.ws_ml = p.ws_ml;
  mp.batch = a.batch;
  mp.clusters = clusters;
  mla_merge_kernel<T><<<dim3(a.batch, 2 * (kH / kMergeRows)), kMergeThreads, 0, a.stream>>>(mp);
  return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

}  // namespace

int mla_decode_num_ctas(int num_ctas) {
  if (num_ctas > 0) return num_ctas & ~1;
  return 2 * mla_resident_clusters();  // one CTA per SM, pairs, all resident
}

size_t mla_decode_workspace_bytes(int ctas) {
  const int clusters = ctas / 2;
  return kPlanBytes + static_cast<size_t>(clusters) * 4 * kH * (kOutCols + 2) * sizeof(float);
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
