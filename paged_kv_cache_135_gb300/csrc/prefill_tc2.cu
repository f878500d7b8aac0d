// Packed-varlen causal prefill over the paged cache on the tcgen05 tensor
// cores, two query heads of one GQA group per CTA (the attention part of
// kvc_varlen_prefill_paged, used when the group size is even).
//
// What it computes: the hotelren.com notes "Paged KV Cache + Packed
// Sequence" 3.1-3.3 -- packed sequences delimited by cu_seqlens, each token
// attending causally (diagonal included) to its own sequence's tokens only,
// read back from the paged cache through the sequence's block_table;
// "external-cannbot-model-model-infer-kvcache" Appendix C sparse_mode 3.
//
// GB300 design.  A work item is (sequence, 128-query tile, pair of query
// heads sharing a KV head).  The CTAs are persistent, one per SM; each takes
// its items from a schedule sorted by weight (tiles attended) and dealt in a
// serpentine, and loads the next item's queries, K/V and first S while the
// previous item's epilogue runs.  Both heads' 128-row query tiles stay in
// shared memory and share one stream of 128-token K and V tiles (TMA
// through block_table, 2-stage rings), so every K/V byte feeds two heads.
// Tensor memory holds O and S for each head (4 x 128 columns).
// Each head has its own softmax warpgroup, one thread per query row and all
// 128 columns of the tile (no cross-thread reduction).  P (bf16/fp16) is
// written back into the head's S columns of tensor memory and read from
// there as the A operand of P V, so each head runs S -> softmax -> P V ->
// next S while the tensor core works on the other head.  The signal that S
// of a tile is complete also means every earlier MMA of the issuing thread
// is complete (tcgen05.commit tracks all of them), so P and O may be written
// without a further wait; the next S of a head is issued after its P V, and
// the tensor core performs one thread's MMAs in issue order.  The MMA warp
// issues warp-convergent from one elected lane, in a fixed order (S of both
// heads, then per tile and head P V followed by the next S), releasing P in
// two halves so P V starts during the exponentials.  Online softmax in the
// log2 domain; O is rescaled only when a row's max grows by more than 2^8.
// The epilogue passes each warp's output rows through shared memory so that
// every store instruction writes whole 64-byte row segments.
//
// Fused write (chunks without cached context): the K/V tiles are read from
// the packed key/value input itself -- the write copies those rows unchanged
// into the cache, so they are the rows the cache would hold -- and an extra
// writer warp in every CTA copies its share of the chunk's rows to the cache
// at slot_mapping, beside the attention and independent of it.  The write
// then runs under the compute-bound attention instead of as a launch before
// it.
#include <cuda_runtime.h>

#include <math.h>

#include <mutex>

#include "kvc_device.cuh"
#include "kvc_host.h"
#include "kvc_tcgen05.cuh"

namespace kvc {

namespace {

constexpr int kBM = 128;                    // query rows per head = MMA M
constexpr int kBN = 128;                    // kv tokens per tile
constexpr int kHeadThreads = 128;           // softmax threads per head
constexpr int kSmxThreads = 2 * kHeadThreads;
constexpr int kProducerWarp = 8, kMmaWarp = 9, kWriterWarp = 10;
constexpr int kThreads = kSmxThreads + 64;
// Threads of a kernel instance: the fused-write instance adds the writer warp.
template <bool kFused>
constexpr int threads_of() { return kFused ? kThreads + 32 : kThreads; }
constexpr int kStages = 2;
constexpr int kChunk = 128 * 128;           // one [128 rows][64 elements] swizzled region
constexpr float kRescaleThreshold = 8.0f;
constexpr int kMaxN = 2048;      // distinct per-item tile counts the sorted schedule handles
constexpr int kMaxSched = 512;   // items per CTA in the sorted schedule
constexpr uint32_t kTmemCols = 512;
// Epilogue staging of one softmax warp: 32 rows of 32 output elements
// (64 bytes), rows 80 bytes apart so that 16-byte accesses of 8 consecutive
// rows fall in distinct banks.
constexpr int kStgRow = 80;
constexpr int kStgWarpBytes = 32 * kStgRow;
// TMEM columns of head x: O at 128x, S at 256 + 128x.
__host__ __device__ constexpr uint32_t tmem_o(int x) { return 128u * x; }
__host__ __device__ constexpr uint32_t tmem_s(int x) { return 256u + 128u * x; }

struct Tc2Params {
  void* out;
  const int32_t* cu_seqlens;
  const int32_t* context_lens;
  const int32_t* block_table;
  uint32_t* err_flag;
  int num_seqs, num_q_heads, group;
  int block_size, log2_bs, max_blocks, num_blocks, box_tokens;
  int window;  // band: a query at position p sees p - window + 1 .. p (0: all of 0 .. p)
  float scale_log2;
  // Fused write only: the rows to store and where.
  const uint8_t* key;
  const uint8_t* value;
  uint8_t* key_cache;
  uint8_t* value_cache;
  const int32_t* slot_mapping;
  int num_tokens, num_kv_heads;
  long long num_slots;
};

// First key position of the band of a query at position `pos` (0 without a band).
__device__ __forceinline__ int band_start(int pos, int window) {
  return window > 0 && pos >= window ? pos - window + 1 : 0;
}
// The band of a kernel instance: the kernel is compiled separately for band
// and causal attention, so the causal instance carries none of the band's
// arithmetic (its window is the constant 0).
template <bool kBand>
__device__ __forceinline__ int window_of(const Tc2Params& p) {
  return kBand ? p.window : 0;
}

template <int D>
struct Tc2Layout {
  static constexpr int kHalves = D / 64;
  static constexpr int kStageBytes = kHalves * kChunk;         // one K or one V tile
  static constexpr int kQ = 0;                                 // head A then head B
  static constexpr int kK = kQ + 2 * kStageBytes;
  static constexpr int kV = kK + kStages * kStageBytes;
  static constexpr int kBar = kV + kStages * kStageBytes;
  static constexpr int kNumBars = 19;
  static constexpr int kMisc = kBar + kNumBars * 8;  // tmem slot, abort, schedule ints, progress
  static constexpr int kHist = kMisc + 64;                     // int[kMaxN]
  static constexpr int kList = kHist + kMaxN * 4;              // int2[kMaxSched]
  static constexpr int kStg = (kList + kMaxSched * 8 + 15) & ~15;  // epilogue staging, per warp
  static constexpr int kTotal = 1024 + kStg + (kSmxThreads / 32) * kStgWarpBytes;
  static_assert(kTotal <= 232448, "fits the opt-in shared memory of one SM");
};

// k_empty / v_empty complete when both heads' S / P V of the tile are done:
// one commit after head 1's, which the tensor core performs after head 0's;
// s_full[h], p_full[h], o_done[h] are per head.
enum Bar {
  kQFull = 0, kKFull0, kKFull1, kKEmpty0, kKEmpty1, kVFull0, kVFull1, kVEmpty0, kVEmpty1,
  kSFull0, kSFull1, kPFull0, kPFull1, kODone0, kODone1, kDrain, kPHalf0, kPHalf1, kQEmpty
};

__device__ __forceinline__ bool wait_t2(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                        uint32_t* err) {
  if (*abort_flag) return false;
  if (mbar_wait_bounded(bar, parity, err)) return true;
  *abort_flag = 1;
  return false;
}

// Work item -> (sequence, query tile), the tiles of each sequence from its
// last (heaviest under the causal mask) to its first; one warp scans
// cu_seqlens 32 sequences at a time.
__device__ __forceinline__ bool tc2_locate(const Tc2Params& p, int item, int lane, int& s,
                                           int& tile, int& ctx, int& len) {
  int before = 0;
  for (int base = 0; base < p.num_seqs; base += 32) {
    const int i = base + lane;
    int n = 0, L = 0;
    if (i < p.num_seqs) {
      L = p.cu_seqlens[i + 1] - p.cu_seqlens[i];
      n = L > 0 ? (L + kBM - 1) / kBM : 0;
    }
    int x = n;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    const int lo = before + x - n;
    const unsigned hit = __ballot_sync(0xffffffffu, i < p.num_seqs && item >= lo && item < lo + n);
    if (hit) {
      const int src = __ffs(hit) - 1;
      s = base + src;
      tile = __shfl_sync(0xffffffffu, n, src) - 1 - (item - __shfl_sync(0xffffffffu, lo, src));
      len = __shfl_sync(0xffffffffu, L, src);
      ctx = p.context_lens ? p.context_lens[s] : 0;
      return true;
    }
    before += __shfl_sync(0xffffffffu, x, 31);
  }
  return false;
}

// TMA producer (one warp): both heads' query tiles once, then each 128-token
// K and V tile, one box per physical block per 64-wide chunk (fused write:
// one box of the packed input per 64-wide chunk; tokens past the sequence
// are masked, and zeroed in V, like cache rows past it).
template <int D, bool kFused>
__device__ __forceinline__ void tc2_producer(const Tc2Params& p, const CUtensorMap* tm_q,
                                             const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                             uint8_t* smem, uint64_t* bars,
                                             volatile int* abort_flag, int s, int h0, int g,
                                             int tok0, int seq_tok0, int kv_len, int j0,
                                             int n_tiles, int band0, int gj0, int kit, int lane) {
  using L = Tc2Layout<D>;
  // This item's query tiles replace the previous item's once its last S is
  // done (q_empty).
  if (kit > 0 && !wait_t2(&bars[kQEmpty], (kit - 1) & 1, abort_flag, p.err_flag)) return;
  if (lane == 0) {
    mbar_arrive_expect_tx(&bars[kQFull], 2 * L::kStageBytes);
#pragma unroll
    for (int x = 0; x < 2; ++x)
#pragma unroll
      for (int c = 0; c < L::kHalves; ++c)
        tma_load_3d(smem + L::kQ + x * L::kStageBytes + c * kChunk, tm_q, &bars[kQFull], c * 64,
                    h0 + x, tok0);
  }
  const int nsub = kBN / p.box_tokens;
  const uint32_t box_bytes = static_cast<uint32_t>(p.box_tokens) * 128u;
  for (int j = 0; j < n_tiles; ++j) {
    const int gj = gj0 + j;  // the CTA's running tile count sets stage and phase
    const int stage = gj & 1;
    const int tok = (j0 + j) * kBN + lane * p.box_tokens;
    // A box wholly before the band of the tile's first query row is not
    // fetched (its rows are masked for every row and zeroed in V).
    const bool wanted = lane < nsub && tok < kv_len && tok + p.box_tokens > band0;
    int pb = -1;
    if (wanted)
      pb = __ldg(&p.block_table[static_cast<long long>(s) * p.max_blocks + (tok >> p.log2_bs)]);
    bool valid = false;
    if (wanted) {
      if (pb < 0 || pb >= p.num_blocks) set_flag(p.err_flag, KVC_FLAG_BLOCK_ID_RANGE);
      else valid = true;
    }
    const int in_blk = tok & (p.block_size - 1);
    // K(j) once both heads' S(j-2) have consumed its stage, V(j) once both
    // heads' P V(j-2) have (fused write: and the writer is done with it).
    if constexpr (kFused) {
      for (int part = 0; part < 2; ++part) {
        const int empty = part ? kVEmpty0 : kKEmpty0, full = part ? kVFull0 : kKFull0;
        const bool ok = wait_t2(&bars[empty + stage], ((gj >> 1) & 1) ^ 1, abort_flag, p.err_flag);
        if (__any_sync(0xffffffffu, !ok)) return;
        if (lane == 0) {
          mbar_arrive_expect_tx(&bars[full + stage], L::kStageBytes);
          uint8_t* dst = smem + (part ? L::kV : L::kK) + stage * L::kStageBytes;
#pragma unroll
          for (int c = 0; c < L::kHalves; ++c)
            tma_load_3d(dst + c * kChunk, part ? tm_v : tm_k, &bars[full + stage], c * 64, g,
                        seq_tok0 + (j0 + j) * kBN);
        }
        __syncwarp();
      }
    } else {
      for (int part = 0; part < 2; ++part) {
        const int empty = part ? kVEmpty0 : kKEmpty0, full = part ? kVFull0 : kKFull0;
        const bool ok = wait_t2(&bars[empty + stage], ((gj >> 1) & 1) ^ 1, abort_flag, p.err_flag);
        const bool go = valid && ok;
        const uint32_t nvalid = __popc(__ballot_sync(0xffffffffu, go));
        if (lane == 0) mbar_arrive_expect_tx(&bars[full + stage], nvalid * box_bytes * L::kHalves);
        __syncwarp();
        if (go) {
          uint8_t* dst = smem + (part ? L::kV : L::kK) + stage * L::kStageBytes + lane * box_bytes;
#pragma unroll
          for (int c = 0; c < L::kHalves; ++c)
            tma_load_4d(dst + c * kChunk, part ? tm_v : tm_k, &bars[full + stage], c * 64, g,
                        in_blk, pb);
        }
      }
    }
  }
}

// The MMA warp, all lanes converged (one elected lane issues; see
// elect_one_sync), in a fixed order: S_0(0), S_1(0), then for each tile j
// and head x one block of P V_x(j) followed by S_x(j+1) (the head's P in its
// S columns is read before S_x(j+1) overwrites them: one thread's MMAs run
// in issue order).  The tensor core keeps only a short queue, so any latency
// between two MMAs is idle tensor time.  Hence a block issues its 16 MMAs
// with nothing between them but commits; the barriers the next block needs
// are tested inside the instruction sequence of the block's last two MMAs
// (their latency hides behind those issues), and the warp blocks in a wait
// only when an input is really not ready yet.  A wait that runs past
// kWaitLimitNs sets KVC_FLAG_WAIT_TIMEOUT and aborts.
template <int D, bool kBf16>
__device__ __forceinline__ void tc2_mma(const Tc2Params& p, uint8_t* smem, uint64_t* bars,
                                        volatile int* abort_flag, uint32_t tmem, int n_tiles,
                                        int gj0, int kit, uint32_t leader) {
  using L = Tc2Layout<D>;
  constexpr int kSSteps = D / 16;   // K steps of S = Q K^T
  constexpr int kPSteps = kBN / 16; // K steps of O += P V
  constexpr uint32_t idesc_s = umma_idesc_f16(kBf16, kBM, kBN, 0, 0);
  constexpr uint32_t idesc_o = umma_idesc_f16(kBf16, kBM, D, 0, 1);
  const uint64_t q0 = umma_desc_sw128(smem_u32(smem + L::kQ), 16, 1024);
  const uint64_t k0 = umma_desc_sw128(smem_u32(smem + L::kK), 16, 1024);
  const uint64_t v0 = umma_desc_sw128(smem_u32(smem + L::kV), kChunk, 1024);

  // Tiles j, t, kt below are this item's; gj0 + j is the CTA's running tile
  // count, which sets the ring stage and every barrier phase.
  // S_x(j).  The next block is P V_y(t) + S_y(t+1): it starts on the first
  // half of P_y(t) and needs V(t) and K(kt) (kt = t+1, or any tile whose K
  // has surely landed when no S follows); returns whether all three were
  // there before the last MMA.  The item's last S releases its query tiles.
  auto s_group = [&](int x, int j, int y, int t, int kt) -> bool {
    const int G = gj0 + j, T = gj0 + t, KT = gj0 + kt;
    const uint32_t d = tmem + tmem_s(x);
    const uint64_t qx = desc_advance(q0, x * L::kStageBytes);
    const uint64_t k_st = desc_advance(k0, (G & 1) * L::kStageBytes);
    auto a_at = [&](int st) { return desc_advance(qx, (st / 4) * kChunk + (st % 4) * 32); };
    auto b_at = [&](int st) { return desc_advance(k_st, (st / 4) * kChunk + (st % 4) * 32); };
#pragma unroll
    for (int st = 0; st < kSSteps - 2; ++st) umma_ss_e(d, a_at(st), b_at(st), idesc_s, st != 0, leader);
    const bool ready = umma_ss_acc2_test3_e(
        d, a_at(kSSteps - 2), b_at(kSSteps - 2), a_at(kSSteps - 1), b_at(kSSteps - 1), idesc_s,
        &bars[kPHalf0 + y], T & 1, &bars[kVFull0 + (T & 1)], (T >> 1) & 1,
        &bars[kKFull0 + (KT & 1)], (KT >> 1) & 1, leader);
    umma_commit_e(&bars[kSFull0 + x], leader);
    if (x == 1) umma_commit_e(&bars[kKEmpty0 + (G & 1)], leader);
    if (x == 1 && j == n_tiles - 1) umma_commit_e(&bars[kQEmpty], leader);
    return ready;
  };
  // P V_x(j), A = P in the head's S columns of tensor memory: tokens 0-63
  // (released by p_half), then, once the whole of P_x(j) is there, 64-127.
  auto pv_group = [&](int x, int j) -> bool {
    const int G = gj0 + j;
    const uint64_t v_st = desc_advance(v0, (G & 1) * L::kStageBytes);
    const uint32_t d = tmem + tmem_o(x), a0 = tmem + tmem_s(x);
#pragma unroll
    for (int ks = 0; ks < kPSteps / 2; ++ks)
      umma_ts_e(d, a0 + ks * 8, desc_advance(v_st, ks * 16 * 128), idesc_o, ks > 0 || j > 0, leader);
    if (!wait_t2(&bars[kPFull0 + x], G & 1, abort_flag, p.err_flag)) return false;
    tc_fence_after();
#pragma unroll
    for (int ks = kPSteps / 2; ks < kPSteps; ++ks)
      umma_ts_e(d, a0 + ks * 8, desc_advance(v_st, ks * 16 * 128), idesc_o, 1u, leader);
    if (x == 1) umma_commit_e(&bars[kVEmpty0 + (G & 1)], leader);
    if (j == n_tiles - 1) umma_commit_e(&bars[kODone0 + x], leader);
    return true;
  };
  auto wait_inputs = [&](int x, int j, bool with_k) -> bool {
    const int G = gj0 + j;
    return wait_t2(&bars[kPHalf0 + x], G & 1, abort_flag, p.err_flag) &&
           wait_t2(&bars[kVFull0 + (G & 1)], (G >> 1) & 1, abort_flag, p.err_flag) &&
           (!with_k ||
            wait_t2(&bars[kKFull0 + ((G + 1) & 1)], ((G + 1) >> 1) & 1, abort_flag, p.err_flag));
  };

  if (!wait_t2(&bars[kQFull], kit & 1, abort_flag, p.err_flag)) return;
  if (!wait_t2(&bars[kKFull0 + (gj0 & 1)], (gj0 >> 1) & 1, abort_flag, p.err_flag)) return;
  tc_fence_after();
  s_group(0, 0, 0, 0, 0);
  bool ready = s_group(1, 0, 0, 0, n_tiles > 1 ? 1 : 0);
  for (int j = 0; j + 1 < n_tiles; ++j) {
    // Block (0, j); the next block is (1, j), whose K(j+1) was waited for here.
    if (!ready && !wait_inputs(0, j, true)) return;
    tc_fence_after();
    if (!pv_group(0, j)) return;
    ready = s_group(0, j + 1, 1, j, j + 1);
    // Block (1, j); the next block is (0, j+1), which needs K(j+2) unless it is
    // the last tile's P V.
    if (!ready && !wait_inputs(1, j, true)) return;
    tc_fence_after();
    if (!pv_group(1, j)) return;
    ready = s_group(1, j + 1, 0, j + 1, j + 2 < n_tiles ? j + 2 : j + 1);
  }
  // The last tile: P V only.
  const int j = n_tiles - 1;
#pragma unroll
  for (int x = 0; x < 2; ++x) {
    if (!ready && !wait_inputs(x, j, false)) return;
    tc_fence_after();
    if (!pv_group(x, j)) return;
    ready = false;
  }
}

// Softmax warpgroup of head x (threads x*128 .. +127): thread owns query row
// `row`, all 128 columns of each tile.
template <typename T, int D, bool kBand>
__device__ __forceinline__ void tc2_softmax(const Tc2Params& p, uint8_t* smem, uint64_t* bars,
                                            volatile int* abort_flag, uint32_t tmem, int x,
                                            int row, int j0, int n_tiles, int q0, int ctx,
                                            int kv_len, int q_rows, int tok0, int h, int gj0,
                                            int kit) {
  using L = Tc2Layout<D>;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(row & ~31) << 16);
  const int pos = ctx + q0 + row;
  float m_used = -INFINITY, l = 0.f;
  for (int j = 0; j < n_tiles; ++j) {
    const int gj = gj0 + j;  // the CTA's running tile count sets every phase
    wait_t2(&bars[kSFull0 + x], gj & 1, abort_flag, p.err_flag);
    tc_fence_after();
    // Row max of the raw scores (the scale is positive, so it commutes with
    // the max and is folded into the exponent below).  The scores stay in
    // tensor memory and are read in halves of 64 columns to keep register
    // pressure down: half 1 first (for its max only), then half 0, which is
    // kept in registers for its exponentials, so the first half of P is
    // released after two rounds of loads, not three.  Band + causal + length
    // mask: token k of the tile is visible iff lo <= k < lim; only tiles that
    // reach past this row, or start before its band, take the masked path.
    const int kv0 = (j0 + j) * kBN;
    const int lim = min(pos + 1, kv_len) - kv0;
    const int lo = kBand ? band_start(pos, p.window) - kv0 : 0;
    const bool masked = lim < kBN || lo > 0;
    float mx8[8];
#pragma unroll
    for (int a = 0; a < 8; ++a) mx8[a] = -INFINITY;
    float s[kBN / 2];
#pragma unroll
    for (int hf = 1; hf >= 0; --hf) {
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c)
        tmem_ld16(lane_base + tmem_s(x) + hf * (kBN / 2) + c * 16, s + c * 16);
      tmem_wait_ld();
      if (masked) {
#pragma unroll
        for (int k = 0; k < kBN / 2; ++k) {
          const int kk = hf * (kBN / 2) + k;
          s[k] = kk >= lo && kk < lim ? s[k] : -INFINITY;
        }
      }
#pragma unroll
      for (int k = 0; k < kBN / 2; k += 2) mx8[(k / 2) & 7] = fmax3(mx8[(k / 2) & 7], s[k], s[k + 1]);
    }
    const float mx = fmaxf(fmax3(mx8[0], mx8[1], mx8[2]),
                           fmax3(fmax3(mx8[3], mx8[4], mx8[5]), mx8[6], mx8[7])) *
                     p.scale_log2;
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
    // S(j) complete means this head's P V(j-1) is complete too, so O may be
    // rescaled and P written over the S columns now.
    if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
      for (int c = 0; c < D / 16; ++c) {
        float v[16];
        const uint32_t a = lane_base + tmem_o(x) + c * 16;
        tmem_ld16(a, v);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] *= corr;
        tmem_st16(a, v);
      }
      // Half 0 of the scores is read again (S is untouched until P is
      // written), so it need not stay in registers across this rare path.
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) tmem_ld16(lane_base + tmem_s(x) + c * 16, s + c * 16);
      tmem_wait_ld();
      if (masked) {
#pragma unroll
        for (int k = 0; k < kBN / 2; ++k) s[k] = k >= lo && k < lim ? s[k] : -INFINITY;
      }
    }
    // Value rows past the cached tokens, and rows before the band of the
    // item's first query row (seen by no row of the item), are zeroed (by
    // both heads, before either head's P V of the tile) so stale contents
    // cannot reach P V.
    const int valid = kv_len - kv0;
    const int zlo = kBand ? band_start(ctx + q0, p.window) - kv0 : 0;
    if (valid < kBN || zlo > 0) {
      wait_t2(&bars[kVFull0 + (gj & 1)], (gj >> 1) & 1, abort_flag, p.err_flag);
      uint8_t* vst = smem + L::kV + (gj & 1) * L::kStageBytes;
      const int top = valid < kBN ? kBN - valid : 0, bottom = zlo > 0 ? min(zlo, kBN) : 0;
      const int n16 = (top + bottom) * L::kHalves * 8;
      for (int e = row; e < n16; e += kHeadThreads) {
        const int i = e / (L::kHalves * 8), c = (e / 8) % L::kHalves, q = e % 8;
        const int r = i < bottom ? i : valid + (i - bottom);
        *reinterpret_cast<uint4*>(vst + c * kChunk + r * 128 + q * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
      fence_proxy_async_smem();
    }
    // p = 2^(s * scale_log2 - m_used); a row with nothing visible yet keeps
    // m_used = -inf and all its scores at -inf, so its p are 0.  P is rounded
    // to T for the tensor core, and the row sum l adds the rounded values, so
    // the output is a convex combination of V rows with exactly the weights
    // P V used (a peaked row then keeps its dominant row almost exactly,
    // whatever that row's magnitude).  P goes to the first 64 columns of the head's S (two
    // 16-bit tokens per column, token 2c in the low half of column c) in two
    // halves: tokens 0-63 (already in registers) are released (p_half) before
    // tokens 64-127 are read again and computed, so the first half of P V
    // overlaps the second half of the exponentials.  Half h of P overwrites
    // only scores of half 0, which are read before.
    const float neg_m = m_used == -INFINITY ? 0.f : -m_used;
    const float2 sc2 = make_float2(p.scale_log2, p.scale_log2), nm2 = make_float2(neg_m, neg_m);
    float2 ps2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      if (hf == 1) {
#pragma unroll
        for (int c = 0; c < kBN / 32; ++c)
          tmem_ld16(lane_base + tmem_s(x) + (kBN / 2) + c * 16, s + c * 16);
        tmem_wait_ld();
        if (masked) {
#pragma unroll
          for (int k = 0; k < kBN / 2; ++k) {
            const int kk = (kBN / 2) + k;
            s[k] = kk >= lo && kk < lim ? s[k] : -INFINITY;
          }
        }
      }
      uint32_t pk[kBN / 4];
#pragma unroll
      for (int k = 0; k < kBN / 4; ++k) {
        const float2 y = fma2(make_float2(s[2 * k], s[2 * k + 1]), sc2, nm2);
        const float2 e = make_float2(fast_exp2(y.x), fast_exp2(y.y));
        pk[k] = pack_pair<T>(e.x, e.y);
        acc_pair<T>(ps2[k & 1], pk[k]);
      }
#pragma unroll
      for (int c = 0; c < kBN / 64; ++c)
        tmem_st16_u32(lane_base + tmem_s(x) + hf * (kBN / 4) + c * 16, pk + c * 16);
      tmem_wait_st();
      if (hf == 0) {
        tc_fence_before();
        mbar_arrive(&bars[kPHalf0 + x]);
      }
    }
    const float2 pst = add2(ps2[0], ps2[1]);
    l = l * corr + (pst.x + pst.y);
    tc_fence_before();
    mbar_arrive(&bars[kPFull0 + x]);
  }

  // Epilogue: normalise and write this head's rows, 32 columns at a time.
  // Each warp passes its 32 rows through shared memory so that a store
  // instruction writes 8 rows x 64 contiguous bytes (8 lines) rather than
  // 32 rows x 16 bytes (32 lines).
  wait_t2(&bars[kODone0 + x], kit & 1, abort_flag, p.err_flag);
  tc_fence_after();
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const int lane = row & 31, wrow0 = row & ~31;
  uint8_t* stg = smem + L::kStg + (x * 4 + (row >> 5)) * kStgWarpBytes;
  const long long ostride = static_cast<long long>(p.num_q_heads) * D;
  T* obase = static_cast<T*>(p.out) + (static_cast<long long>(tok0) + wrow0) * ostride + h * D;
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {  // two TMEM loads in flight per wait
    float v[32];
    tmem_ld16(lane_base + tmem_o(x) + c * 32, v);
    tmem_ld16(lane_base + tmem_o(x) + c * 32 + 16, v + 16);
    tmem_wait_ld();
    uint32_t w[16];
    float a, b;
#pragma unroll
    for (int k = 0; k < 16; ++k) w[k] = Pack<T>::run(v[2 * k] * inv, v[2 * k + 1] * inv, a, b);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<uint4*>(stg + lane * kStgRow + q * 16) =
          make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = i * 8 + (lane >> 2), q = lane & 3;
      const uint4 val = *reinterpret_cast<const uint4*>(stg + r * kStgRow + q * 16);
      if (wrow0 + r < q_rows) *reinterpret_cast<uint4*>(obase + r * ostride + c * 32 + q * 8) = val;
    }
    __syncwarp();
  }
  tc_fence_before();
}

// Fused write.  The writer warp of each CTA walks the CTA's own items and,
// for each item of the first head pair of a KV head g, copies the item's
// query-tile rows -- packed tokens tok .. tok + rows - 1, head g, the rows of
// its diagonal K/V tile -- from key/value to the cache row of slot
// slot_mapping[t]: a negative slot is skipped, one outside the pool is
// skipped and flagged, as in kvc_reshape_and_cache.  Every packed token of a
// sequence lies in exactly one query tile, so each (token, head) row is
// copied once.  The copies run beside the attention, which reads the same
// rows from the input at about the same time (they meet in L2), and touch no
// ring stage or barrier: a writer that held a stage until it had read the
// rows out of shared memory stalled the K/V ring.  One warp is
// latency-bound, so each lane keeps kBatch K and V loads in flight; the
// item's slots are staged in shared memory (the schedule histogram's space,
// unused after the prologue).
// The writer paces itself by the producer's progress: kWriteBatchAhead loads
// in flight while it is two or more items ahead of the producer on an item of
// at least 4 key tiles, kWriteBatch otherwise -- fewer loads in flight take
// less from the attention (measured: 2 in flight 406 us, 8 in flight 418 us
// on 16 prompts of 50-3000 tokens, whose long items leave the writer ahead),
// while short items need the higher rate to keep up (96 prompts of 64-512
// tokens: 2 in flight 312 us, 8 in flight 194 us, paced 197 us).
constexpr int kWriteBatch = 8, kWriteBatchAhead = 2;
template <int D, int kBatch>
__device__ __forceinline__ void tc2_write_rows(const Tc2Params& p, int* slots, int tok, int rows,
                                               int g, int lane) {
  rows = min(rows, p.num_tokens - tok);
#pragma unroll
  for (int i = 0; i < kBM / 32; ++i) {
    const int r = lane + 32 * i;
    slots[r] = r < rows ? __ldg(&p.slot_mapping[tok + r]) : -1;
  }
  __syncwarp();
  constexpr int kCR = D / 8, kRPI = 32 / kCR;  // lanes per row, rows per warp access
  const int k = lane % kCR, rsub = lane / kCR;
  const long long rb = static_cast<long long>(p.num_kv_heads) * D * 2;
  const long long off = static_cast<long long>(g) * D * 2 + k * 16;
  bool outside = false;  // a slot outside the pool (flagged once, after the loop)
#pragma unroll 1
  for (int r0 = 0; r0 < rows; r0 += kBatch * kRPI) {
    uint4 kv[kBatch], vv[kBatch];
    int sl[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int r = r0 + u * kRPI + rsub;
      sl[u] = r < rows ? slots[r] : -1;
      if (r < rows) {
        kv[u] = __ldg(reinterpret_cast<const uint4*>(p.key + (tok + r) * rb + off));
        vv[u] = __ldg(reinterpret_cast<const uint4*>(p.value + (tok + r) * rb + off));
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      if (sl[u] < 0) continue;
      if (sl[u] >= p.num_slots) {
        outside = true;
        continue;
      }
      __stcs(reinterpret_cast<uint4*>(p.key_cache + sl[u] * rb + off), kv[u]);
      __stcs(reinterpret_cast<uint4*>(p.value_cache + sl[u] * rb + off), vv[u]);
    }
  }
  // The flag is set outside the copy loop: an atomic in the loop measured
  // 5 % slower for the whole kernel.
  if (outside) set_flag(p.err_flag, KVC_FLAG_SLOT_RANGE);
  __syncwarp();
}

// One work item: (sequence, 128-query tile, pair of query heads); every
// lane of the calling warp gets the same result.
struct Tc2Item {
  int s, h0, q0, q_rows, ctx, kv_len, j0, n_tiles, tok0;
  bool ok;  // kv_len fits the block table
};

// Key tiles j0 .. j0 + n_tiles - 1 of a query tile: from the tile holding
// the band start of its first row to the tile holding its last row.
template <bool kBand>
__device__ __forceinline__ void tc2_tiles(const Tc2Params& p, Tc2Item& it) {
  it.j0 = band_start(it.ctx + it.q0, window_of<kBand>(p)) / kBN;
  it.n_tiles = (it.ctx + it.q0 + it.q_rows - 1) / kBN + 1 - it.j0;
}
template <bool kBand>
__device__ __forceinline__ bool tc2_item(const Tc2Params& p, int w, int lane, Tc2Item& it) {
  const int pairs = p.num_q_heads / 2;
  int s = 0, tile = 0, ctx = 0, len = 0;
  if (!tc2_locate(p, w / pairs, lane, s, tile, ctx, len)) return false;
  it.s = s;
  it.h0 = 2 * (w % pairs);
  it.q0 = tile * kBM;
  it.q_rows = min(kBM, len - it.q0);
  it.ctx = ctx;
  it.kv_len = ctx + len;
  it.ok = it.kv_len <= p.max_blocks * p.block_size;
  tc2_tiles<kBand>(p, it);
  it.tok0 = p.cu_seqlens[s] + it.q0;
  return true;
}

// The work item of query tile t of sequence s, head pair `pair`.
template <bool kBand>
__device__ __forceinline__ void tc2_item_at(const Tc2Params& p, int s, int t, int pair,
                                            Tc2Item& it) {
  const int len = p.cu_seqlens[s + 1] - p.cu_seqlens[s];
  it.s = s;
  it.h0 = 2 * pair;
  it.q0 = t * kBM;
  it.q_rows = min(kBM, len - it.q0);
  it.ctx = p.context_lens ? p.context_lens[s] : 0;
  it.kv_len = it.ctx + len;
  it.ok = it.kv_len <= p.max_blocks * p.block_size;
  tc2_tiles<kBand>(p, it);
  it.tok0 = p.cu_seqlens[s] + it.q0;
}

// Tiles attended by query tile t of a sequence with `ctx` cached tokens and
// `len` new ones (its weight in the schedule).
__device__ __forceinline__ int tc2_weight(int ctx, int len, int t) {
  const int rows = min(kBM, len - kBM * t);
  return (ctx + kBM * t + rows - 1) / kBN + 1;
}

// Sorted schedule, built by every CTA in its prologue (all threads): the work
// items ordered by weight (tiles attended) from heaviest, then sequence,
// tile and head pair, dealt to the CTAs in a serpentine (CTA c takes
// positions c, 2G-1-c, 2G+c, ...), so every CTA gets a similar total.  A
// query tile's weight is c0 + t + 1 (c0 = ceil(ctx / 128)) except that the
// last tile of a sequence may share its predecessor's, so the tile of a
// given weight in a sequence is found in closed form.  Returns the number
// of items of this CTA, written as (s, t << 8 | pair) to `list`, or -1 when
// the bounds are exceeded (then the CTA walks items c, c + G, ... unsorted).
__device__ __forceinline__ int tc2_tiles_of_weight(const Tc2Params& p, int s, int n, int* t_out) {
  const int len = p.cu_seqlens[s + 1] - p.cu_seqlens[s];
  const int ctx = p.context_lens ? p.context_lens[s] : 0;
  const int nq = len > 0 ? (len + kBM - 1) / kBM : 0;
  int cnt = 0;
  const int t1 = n - 1 - (ctx + kBN - 1) / kBN;
  if (t1 >= 0 && t1 < nq - 1) t_out[cnt++] = t1;
  if (nq > 0 && tc2_weight(ctx, len, nq - 1) == n) t_out[cnt++] = nq - 1;
  return cnt;
}
template <int D, bool kBand>
__device__ int tc2_build_schedule(const Tc2Params& p, uint8_t* smem, int tid, int warp, int lane,
                                  int c, int G) {
  using L = Tc2Layout<D>;
  int* hist = reinterpret_cast<int*>(smem + L::kHist);
  int2* list = reinterpret_cast<int2*>(smem + L::kList);
  volatile int* misc = reinterpret_cast<volatile int*>(smem + L::kMisc + 16);  // qtot, bad, nsched
  const int pairs = p.num_q_heads / 2;
  const int nthr = blockDim.x;
  for (int i = tid; i < kMaxN; i += nthr) hist[i] = 0;
  if (tid == 0) {
    misc[0] = 0;
    // The closed forms below assume causal weights; a band walks unsorted.
    misc[1] = pairs > 255 || kBand ? 1 : 0;
  }
  __syncthreads();
  for (int s = tid; s < p.num_seqs; s += nthr) {
    const int len = p.cu_seqlens[s + 1] - p.cu_seqlens[s];
    const int ctx = p.context_lens ? p.context_lens[s] : 0;
    const int nq = len > 0 ? (len + kBM - 1) / kBM : 0;
    for (int t = 0; t < nq; ++t) {
      const int n = tc2_weight(ctx, len, t);
      if (n < kMaxN) atomicAdd(&hist[n], 1);
      else misc[1] = 1;
    }
    if (nq) atomicAdd(const_cast<int*>(&misc[0]), nq);
  }
  __syncthreads();
  if (warp == 0) {
    int nsched = -1;
    if (misc[1] == 0) {
      // hist[n] -> tiles with weight > n (suffix sums, 32 entries at a time).
      int carry = 0;
      for (int base = kMaxN - 32; base >= 0; base -= 32) {
        const int v = hist[base + lane];
        int x = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int y = __shfl_down_sync(0xffffffffu, x, off);
          if (lane + off < 32) x += y;
        }
        hist[base + lane] = carry + x - v;
        carry += __shfl_sync(0xffffffffu, x, 0);
      }
      __syncwarp();
      const long long items = static_cast<long long>(misc[0]) * pairs;
      nsched = 0;
      for (int k = 0;; ++k) {
        const long long i = static_cast<long long>(k) * G + ((k & 1) ? G - 1 - c : c);
        if (i >= items) break;
        if (k >= kMaxSched) {
          nsched = -1;
          break;
        }
        const int qi = static_cast<int>(i / pairs), pair = static_cast<int>(i % pairs);
        int lo = 1, hi = kMaxN - 1;  // smallest n with (tiles heavier than n) <= qi
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (hist[mid] <= qi) hi = mid; else lo = mid + 1;
        }
        const int n = lo;
        int r = qi - hist[n];  // rank among the tiles of weight n, in (s, t) order
        int found_s = -1, found_t = 0;
        for (int base = 0; base < p.num_seqs && found_s < 0; base += 32) {
          const int sq = base + lane;
          int ts[2] = {0, 0};
          const int cnt = sq < p.num_seqs ? tc2_tiles_of_weight(p, sq, n, ts) : 0;
          int x = cnt;
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
          }
          const unsigned hit = __ballot_sync(0xffffffffu, x > r && x - cnt <= r);
          if (hit) {
            const int src = __ffs(hit) - 1;
            const int before = __shfl_sync(0xffffffffu, x - cnt, src);
            const int t0 = __shfl_sync(0xffffffffu, ts[0], src);
            const int t1 = __shfl_sync(0xffffffffu, ts[1], src);
            found_s = base + src;
            found_t = (r - before) == 0 ? t0 : t1;
          } else {
            r -= __shfl_sync(0xffffffffu, x, 31);
          }
        }
        if (found_s < 0) {  // inconsistent counts: walk the items unsorted instead
          nsched = -1;
          break;
        }
        if (lane == 0) list[k] = make_int2(found_s, (found_t << 8) | pair);
        nsched = k + 1;
      }
    }
    if (lane == 0) misc[2] = nsched;
  }
  __syncthreads();
  return misc[2];
}

// Persistent: CTA c takes its items from the sorted schedule (or c, c + G,
// ... when that does not fit).  Every role walks the same items; the ring
// stages and barrier phases follow
// the CTA's running tile count (gj0) and item count (ni), so the next item's
// queries, K/V tiles and first S are loaded and computed while the softmax
// warps finish the previous item's epilogue.  An item whose sequence does not
// fit the block table is skipped (KVC_FLAG_LEN_RANGE, no output; the fused
// write still copies its rows, as the separate write does).
template <typename T, int D, bool kBf16, bool kBand, bool kFused>
__global__ void __launch_bounds__(threads_of<kFused>(), 1)
    prefill_tc2_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ Tc2Params p) {
  using L = Tc2Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  // The item the producer works on (fused write: paces the writer).
  volatile int* progress = reinterpret_cast<volatile int*>(smem + L::kMisc + 32);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, G = gridDim.x;

  if (tid == 0) {
    for (int i = 0; i < L::kNumBars; ++i) {
      uint32_t cnt = 1;
      if (i == kPFull0 || i == kPFull1 || i == kPHalf0 || i == kPHalf1) cnt = kHeadThreads;
      mbar_init(&bars[i], cnt);
    }
    *abort_flag = 0;
    *progress = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) tmem_alloc(tslot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const int nsched = tc2_build_schedule<D, kBand>(p, smem, tid, warp, lane, c, G);
  const int2* list = reinterpret_cast<const int2*>(smem + L::kList);
  // The k-th item of this CTA: from the sorted schedule, or items c + k*G.
  auto next_item = [&](int k, Tc2Item& it) -> bool {
    if (nsched >= 0) {
      if (k >= nsched) return false;
      const int2 e = list[k];
      tc2_item_at<kBand>(p, e.x, e.y >> 8, e.y & 255, it);
      return true;
    }
    return tc2_item<kBand>(p, c + k * G, lane, it);
  };

  int gj0 = 0, ni = 0;
  if (warp < kProducerWarp) {
    const int x = tid / kHeadThreads;
    for (int k = 0;; ++k) {
      Tc2Item it;
      if (!next_item(k, it)) break;
      if (!it.ok) continue;
      tc2_softmax<T, D, kBand>(p, smem, bars, abort_flag, tmem, x, tid % kHeadThreads, it.j0,
                        it.n_tiles, it.q0, it.ctx, it.kv_len, it.q_rows, it.tok0, it.h0 + x,
                        gj0, ni);
      gj0 += it.n_tiles;
      ++ni;
      if (*abort_flag) break;
    }
  } else if (warp == kProducerWarp) {
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
    }
    for (int k = 0;; ++k) {
      Tc2Item it;
      if (!next_item(k, it)) break;
      if (kFused && lane == 0) *progress = k;
      if (!it.ok) {
        if (lane == 0) set_flag(p.err_flag, KVC_FLAG_LEN_RANGE);
        continue;
      }
      tc2_producer<D, kFused>(p, &tm_q, &tm_k, &tm_v, smem, bars, abort_flag, it.s, it.h0,
                              it.h0 / p.group, it.tok0, it.tok0 - it.q0, it.kv_len, it.j0,
                              it.n_tiles, band_start(it.ctx + it.q0, window_of<kBand>(p)), gj0,
                              ni, lane);
      gj0 += it.n_tiles;
      ++ni;
      if (*abort_flag) break;
    }
    // Every copy issued must land before shared memory can be released.
    for (int gj = gj0 > kStages ? gj0 - kStages : 0; gj < gj0; ++gj) {
      mbar_wait_bounded(&bars[kKFull0 + (gj & 1)], (gj >> 1) & 1, p.err_flag);
      mbar_wait_bounded(&bars[kVFull0 + (gj & 1)], (gj >> 1) & 1, p.err_flag);
    }
  } else if (kFused && warp == kWriterWarp) {
    int* slots = reinterpret_cast<int*>(smem + L::kHist);
    for (int k = 0;; ++k) {
      Tc2Item it;
      if (!next_item(k, it)) break;
      if (it.h0 % p.group != 0) continue;
      if (k > *progress + 1 && it.n_tiles >= 4)
        tc2_write_rows<D, kWriteBatchAhead>(p, slots, it.tok0, it.q_rows, it.h0 / p.group, lane);
      else
        tc2_write_rows<D, kWriteBatch>(p, slots, it.tok0, it.q_rows, it.h0 / p.group, lane);
    }
    // Tokens after the last sequence belong to no item: every head of them,
    // 128 tokens per CTA in turn.
    for (int t = p.cu_seqlens[p.num_seqs] + c * kBM; t < p.num_tokens; t += G * kBM)
      for (int g = 0; g < p.num_kv_heads; ++g)
        tc2_write_rows<D, kWriteBatch>(p, slots, t, kBM, g, lane);
  } else if (warp == kMmaWarp) {
    const uint32_t leader = elect_one_sync();
    for (int k = 0;; ++k) {
      Tc2Item it;
      if (!next_item(k, it)) break;
      if (!it.ok) continue;
      tc2_mma<D, kBf16>(p, smem, bars, abort_flag, tmem, it.n_tiles, gj0, ni, leader);
      gj0 += it.n_tiles;
      ++ni;
      if (*abort_flag) break;
    }
    // Teardown: all tensor-core work done before TMEM is freed.
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
}

template <typename T, int D, bool kBf16, bool kBand, bool kFused>
kvc_status run_prefill_tc2(const PrefillArgs& a) {
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(prefill_tc2_kernel<T, D, kBf16, kBand, kFused>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, Tc2Layout<D>::kTotal);
  });
  CUtensorMap tq, tk, tv;
  const uint64_t qdims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.num_q_heads),
                             static_cast<uint64_t>(a.num_tokens)};
  const uint64_t qstrides[2] = {static_cast<uint64_t>(D) * 2,
                                static_cast<uint64_t>(a.num_q_heads) * D * 2};
  const uint32_t qbox[3] = {64, 1, kBM};
  const int box_tokens = a.block_size < kBN ? a.block_size : kBN;
  const uint64_t dims[4] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.num_kv_heads),
                            static_cast<uint64_t>(a.block_size),
                            static_cast<uint64_t>(a.num_blocks)};
  const uint64_t strides[3] = {static_cast<uint64_t>(D) * 2,
                               static_cast<uint64_t>(a.num_kv_heads) * D * 2,
                               static_cast<uint64_t>(a.block_size) * a.num_kv_heads * D * 2};
  const uint32_t box[4] = {64, 1, static_cast<uint32_t>(box_tokens), 1};
  // Fused write: K/V tiles of 128 packed tokens straight from the input.
  const uint64_t kvdims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.num_kv_heads),
                              static_cast<uint64_t>(a.num_tokens)};
  const uint64_t kvstrides[2] = {static_cast<uint64_t>(D) * 2,
                                 static_cast<uint64_t>(a.num_kv_heads) * D * 2};
  const uint32_t kvbox[3] = {64, 1, kBN};
  if (!encode_tmap_16bit(&tq, a.dtype, 3, a.q, qdims, qstrides, qbox, true))
    return KVC_ERR_CUDA;
  if (kFused ? !encode_tmap_16bit(&tk, a.dtype, 3, a.key, kvdims, kvstrides, kvbox, true) ||
                   !encode_tmap_16bit(&tv, a.dtype, 3, a.value, kvdims, kvstrides, kvbox, true)
             : !encode_tmap_16bit(&tk, a.dtype, 4, a.key_cache, dims, strides, box, true) ||
                   !encode_tmap_16bit(&tv, a.dtype, 4, a.value_cache, dims, strides, box, true))
    return KVC_ERR_CUDA;
  Tc2Params p;
  p.out = a.out;
  p.cu_seqlens = a.cu_seqlens;
  p.context_lens = a.context_lens;
  p.block_table = a.block_table;
  p.err_flag = a.err_flag;
  p.num_seqs = a.num_seqs;
  p.num_q_heads = a.num_q_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.block_size = a.block_size;
  p.log2_bs = ilog2(a.block_size);
  p.max_blocks = a.max_blocks_per_seq;
  p.num_blocks = a.num_blocks;
  p.box_tokens = box_tokens;
  p.window = a.window;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.key = static_cast<const uint8_t*>(a.key);
  p.value = static_cast<const uint8_t*>(a.value);
  p.key_cache = static_cast<uint8_t*>(a.key_cache);
  p.value_cache = static_cast<uint8_t*>(a.value_cache);
  p.slot_mapping = a.slot_mapping;
  p.num_tokens = a.num_tokens;
  p.num_kv_heads = a.num_kv_heads;
  p.num_slots = static_cast<long long>(a.num_blocks) * a.block_size;
  // Work items: (query tile, head pair); query tiles <= T / BM + S.  One
  // persistent CTA per SM, or fewer when there are fewer items.
  const long long items =
      (static_cast<long long>(a.num_tokens) / kBM + a.num_seqs) * (a.num_q_heads / 2);
  if (items > 0x7fffffffLL) return KVC_ERR_UNSUPPORTED;
  const int sms = device_sm_count();
  if (sms <= 0) return KVC_ERR_CUDA;
  const long long grid = items < sms ? items : sms;
  if (grid <= 0) return KVC_OK;
  prefill_tc2_kernel<T, D, kBf16, kBand, kFused>
      <<<static_cast<unsigned>(grid), threads_of<kFused>(), Tc2Layout<D>::kTotal, a.stream>>>(
          tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

// Two heads per CTA; the caller checks that the GQA group size is even.
template <bool kBand, bool kFused>
kvc_status launch_tc2(const PrefillArgs& a) {
  if (a.head_dim == 64)
    return a.dtype == KVC_BF16 ? run_prefill_tc2<__nv_bfloat16, 64, true, kBand, kFused>(a)
                               : run_prefill_tc2<__half, 64, false, kBand, kFused>(a);
  if (a.head_dim == 128)
    return a.dtype == KVC_BF16 ? run_prefill_tc2<__nv_bfloat16, 128, true, kBand, kFused>(a)
                               : run_prefill_tc2<__half, 128, false, kBand, kFused>(a);
  return KVC_ERR_UNSUPPORTED;
}
}  // namespace

kvc_status launch_prefill_attention_tc2(const PrefillArgs& a) {
  return a.window > 0 ? launch_tc2<true, false>(a) : launch_tc2<false, false>(a);
}

kvc_status launch_prefill_fused_tc2(const PrefillArgs& a) {
  return a.window > 0 ? launch_tc2<true, true>(a) : launch_tc2<false, true>(a);
}

}  // namespace kvc
