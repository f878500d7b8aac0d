// Packed-varlen causal prefill over the paged cache on the tcgen05 tensor
// cores (the attention part of kvc_varlen_prefill_paged; the call's cache
// write is in cache_write.cu).
//
// What it computes: the hotelren.com notes "Paged KV Cache + Packed
// Sequence" 3.1-3.3 -- packed sequences delimited by cu_seqlens, each token
// attending causally (diagonal included) to its own sequence's tokens only,
// read back from the paged cache through the sequence's block_table;
// "external-cannbot-model-model-infer-kvcache" Appendix C sparse_mode 3.
//
// GB300 design.  One CTA per (sequence, 128-query tile, q head), the
// heaviest tiles of each sequence first.  The 128 query rows are the M side
// of tcgen05.mma; K/V tiles are 128 tokens (N of S = Q K^T, K of O += P V),
// so every MMA is M128 x N128 (or N = head_dim) and runs near the tensor
// core's peak.  Roles: a TMA producer warp (query tile once, then K and V
// tiles through block_table into 2-stage K and V rings, K released as soon
// as its S is computed), one thread issuing the
// MMAs (S of the next tile is issued before P V of the current one, S
// double-buffered in tensor memory, O accumulated in tensor memory), and
// eight softmax warps, two threads per query row (64 columns each) that
// exchange only the row max through shared memory.  The softmax runs in the
// log2 domain with a position-based causal mask and rescales O only when a
// row's max grows by more than 2^8; P goes to shared memory (bf16/fp16,
// 128-byte swizzled) and V is consumed MN-major straight from its TMA tile.
#include <cuda_runtime.h>

#include <math.h>

#include <mutex>

#include "kvc_device.cuh"
#include "kvc_host.h"
#include "kvc_tcgen05.cuh"

namespace kvc {

namespace {

constexpr int kBM = 128;                 // query rows = MMA M
constexpr int kBN = 128;                 // kv tokens per tile
constexpr int kSmxThreads = 256;         // 8 softmax warps
constexpr int kThreads = kSmxThreads + 64;  // + producer warp + MMA warp
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr int kStages = 2;
constexpr int kChunk = 128 * 128;        // one [128 rows][64 elements] swizzled region (16 KB)
constexpr float kRescaleThreshold = 8.0f;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0, kTmemS0 = 128, kTmemS1 = 256;

struct TcPrefillParams {
  void* out;
  const int32_t* cu_seqlens;
  const int32_t* context_lens;
  const int32_t* block_table;
  uint32_t* err_flag;
  int num_seqs, num_q_heads, group;
  int block_size, log2_bs, max_blocks, num_blocks, box_tokens;
  int window;  // band: a query at position p sees p - window + 1 .. p (0: all of 0 .. p)
  float scale_log2;
};

// First key position of the band of a query at position `pos` (0 without a band).
__device__ __forceinline__ int band_start(int pos, int window) {
  return window > 0 && pos >= window ? pos - window + 1 : 0;
}

template <int D>
struct TcLayout {
  static constexpr int kHalves = D / 64;
  static constexpr int kQ = 0;                                 // kHalves chunks
  static constexpr int kStageBytes = kHalves * kChunk;         // one K or one V tile
  static constexpr int kK = kQ + kHalves * kChunk;             // K ring
  static constexpr int kV = kK + kStages * kStageBytes;        // V ring
  static constexpr int kP = kV + kStages * kStageBytes;        // 2 chunks (128 tokens)
  static constexpr int kRed = kP + 2 * kChunk;                 // float[2 tiles][2 halves][128]
  static constexpr int kBar = kRed + 2 * 2 * kBM * 4;
  static constexpr int kNumBars = 16;
  static constexpr int kMisc = kBar + kNumBars * 8;            // tmem slot, abort, info[4]
  static constexpr int kTotal = 1024 + kMisc + 64;
};

enum Bar { kQFull = 0, kKFull0, kKFull1, kKEmpty0, kKEmpty1, kSFull0, kSFull1, kSFree0, kSFree1,
           kPFull, kPVDone, kDrain, kVFull0, kVFull1, kVEmpty0, kVEmpty1 };

__device__ __forceinline__ bool wait_tc(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                        uint32_t* err) {
  if (*abort_flag) return false;
  if (mbar_wait_bounded(bar, parity, err)) return true;
  *abort_flag = 1;
  return false;
}

// Work item -> (sequence, query tile), the tiles of each sequence from its
// last (heaviest under the causal mask) to its first; one warp scans
// cu_seqlens 32 sequences at a time.
__device__ __forceinline__ bool tc_locate(const TcPrefillParams& p, int item, int lane, int& s,
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

}  // namespace

namespace {

// TMA producer (one warp): the query tile once, then each 128-token K and V
// tile, one box per physical block per 64-wide chunk.
template <int D>
__device__ __forceinline__ void tc_producer(const TcPrefillParams& p, const CUtensorMap* tm_q,
                                            const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                            uint8_t* smem, uint64_t* bars,
                                            volatile int* abort_flag, int s, int h, int g,
                                            int tok0, int kv_len, int j0, int n_tiles, int band0,
                                            int lane) {
  using L = TcLayout<D>;
  if (lane == 0) {
    mbar_arrive_expect_tx(&bars[kQFull], L::kHalves * kChunk);
#pragma unroll
    for (int c = 0; c < L::kHalves; ++c)
      tma_load_3d(smem + L::kQ + c * kChunk, tm_q, &bars[kQFull], c * 64, h, tok0);
  }
  const int nsub = kBN / p.box_tokens;
  const uint32_t box_bytes = static_cast<uint32_t>(p.box_tokens) * 128u;
  for (int j = 0; j < n_tiles; ++j) {
    const int stage = j & 1;
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
    // K(j) as soon as S(j-2) has consumed its stage, V(j) once P V(j-2) has.
    for (int part = 0; part < 2; ++part) {
      const int empty = part ? kVEmpty0 : kKEmpty0, full = part ? kVFull0 : kKFull0;
      const bool ok = wait_tc(&bars[empty + stage], ((j >> 1) & 1) ^ 1, abort_flag, p.err_flag);
      const bool go = valid && ok;
      const uint32_t nvalid = __popc(__ballot_sync(0xffffffffu, go));
      if (lane == 0) mbar_arrive_expect_tx(&bars[full + stage], nvalid * box_bytes * L::kHalves);
      __syncwarp();
      if (go) {
        uint8_t* dst = smem + (part ? L::kV : L::kK) + stage * L::kStageBytes + lane * box_bytes;
#pragma unroll
        for (int c = 0; c < L::kHalves; ++c)
          tma_load_4d(dst + c * kChunk, part ? tm_v : tm_k, &bars[full + stage], c * 64, g, in_blk,
                      pb);
      }
    }
  }
  // Every copy issued must land before shared memory can be released.
  for (int j = n_tiles > kStages ? n_tiles - kStages : 0; j < n_tiles; ++j) {
    mbar_wait_bounded(&bars[kKFull0 + (j & 1)], (j >> 1) & 1, p.err_flag);
    mbar_wait_bounded(&bars[kVFull0 + (j & 1)], (j >> 1) & 1, p.err_flag);
  }
}

// The MMA warp, all lanes converged (one elected lane issues; see
// elect_one_sync), issues every MMA: S(j+1) before P(j) V(j).
template <int D, bool kBf16>
__device__ __forceinline__ void tc_mma(const TcPrefillParams& p, uint8_t* smem, uint64_t* bars,
                                       volatile int* abort_flag, uint32_t tmem, int n_tiles,
                                       uint32_t leader) {
  using L = TcLayout<D>;
  constexpr uint32_t idesc_s = umma_idesc_f16(kBf16, kBM, kBN, 0, 0);
  constexpr uint32_t idesc_o = umma_idesc_f16(kBf16, kBM, D, 0, 1);
  const uint64_t q0 = umma_desc_sw128(smem_u32(smem + L::kQ), 16, 1024);
  const uint64_t k0 = umma_desc_sw128(smem_u32(smem + L::kK), 16, 1024);
  const uint64_t v0 = umma_desc_sw128(smem_u32(smem + L::kV), kChunk, 1024);
  const uint64_t p0 = umma_desc_sw128(smem_u32(smem + L::kP), 16, 1024);
  if (!wait_tc(&bars[kQFull], 0, abort_flag, p.err_flag)) return;

  auto issue_s = [&](int j) -> bool {
    const int stage = j & 1;
    if (!wait_tc(&bars[kKFull0 + stage], (j >> 1) & 1, abort_flag, p.err_flag)) return false;
    if (!wait_tc(&bars[kSFree0 + stage], ((j >> 1) & 1) ^ 1, abort_flag, p.err_flag)) return false;
    tc_fence_after();
    const uint32_t d = tmem + (stage ? kTmemS1 : kTmemS0);
    const uint64_t k_st = desc_advance(k0, stage * L::kStageBytes);
#pragma unroll
    for (int c = 0; c < L::kHalves; ++c)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t a = desc_advance(q0, c * kChunk + kk * 32);
        const uint64_t b = desc_advance(k_st, c * kChunk + kk * 32);
        umma_ss_e(d, a, b, idesc_s, c != 0 || kk != 0, leader);
      }
    umma_commit_e(&bars[kSFull0 + stage], leader);
    umma_commit_e(&bars[kKEmpty0 + stage], leader);
    return true;
  };
  auto issue_pv = [&](int j) -> bool {
    if (!wait_tc(&bars[kVFull0 + (j & 1)], (j >> 1) & 1, abort_flag, p.err_flag)) return false;
    if (!wait_tc(&bars[kPFull], j & 1, abort_flag, p.err_flag)) return false;
    tc_fence_after();
    const uint64_t v_st = desc_advance(v0, (j & 1) * L::kStageBytes);
#pragma unroll
    for (int ks = 0; ks < kBN / 16; ++ks) {
      const uint64_t a = desc_advance(p0, (ks >> 2) * kChunk + (ks & 3) * 32);
      const uint64_t b = desc_advance(v_st, ks * 16 * 128);
      umma_ss_e(tmem + kTmemO, a, b, idesc_o, j != 0 || ks != 0, leader);
    }
    umma_commit_e(&bars[kPVDone], leader);
    umma_commit_e(&bars[kVEmpty0 + (j & 1)], leader);
    return true;
  };
  if (!issue_s(0)) return;
  for (int j = 0; j < n_tiles; ++j) {
    if (j + 1 < n_tiles && !issue_s(j + 1)) return;
    if (!issue_pv(j)) return;
  }
}

}  // namespace

namespace {

// Softmax warps: thread pair (t, t + 128) owns query row t % 128, columns
// 0..63 and 64..127 of each tile; only the row max is exchanged per tile.
template <typename T, int D>
__device__ __forceinline__ void tc_softmax(const TcPrefillParams& p, uint8_t* smem, uint64_t* bars,
                                           volatile int* abort_flag, uint32_t tmem, int t,
                                           int j0, int n_tiles, int q0, int ctx, int kv_len,
                                           int q_rows, int tok0, int h) {
  using L = TcLayout<D>;
  const int warp = t >> 5, lane = t & 31;
  const int quad = warp & 3, half = warp >> 2;
  const int row = quad * 32 + lane;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
  const int pos = ctx + q0 + row;
  float* red = reinterpret_cast<float*>(smem + L::kRed);  // [2 tiles][2 halves][128]
  float m_used = -INFINITY, l = 0.f;
  for (int j = 0; j < n_tiles; ++j) {
    const int stage = j & 1;
    wait_tc(&bars[kSFull0 + stage], (j >> 1) & 1, abort_flag, p.err_flag);
    tc_fence_after();
    float s[64];
#pragma unroll
    for (int c = 0; c < 4; ++c)
      tmem_ld16(lane_base + (stage ? kTmemS1 : kTmemS0) + half * 64 + c * 16, s + c * 16);
    tmem_wait_ld();
    tc_fence_before();
    mbar_arrive(&bars[kSFree0 + stage]);

    // band + causal + length mask (only tiles reaching past this row, or
    // starting before its band, need it)
    const int kv0 = (j0 + j) * kBN + half * 64;
    const int lo = band_start(pos, p.window);
    const bool need_mask = kv0 + 63 > pos || kv0 + 64 > kv_len || kv0 < lo;
    float mx8[8];
#pragma unroll
    for (int a = 0; a < 8; ++a) mx8[a] = -INFINITY;
#pragma unroll
    for (int k = 0; k < 64; ++k) {
      float v = s[k] * p.scale_log2;
      if (need_mask && (kv0 + k > pos || kv0 + k >= kv_len || kv0 + k < lo)) v = -INFINITY;
      s[k] = v;
      mx8[k & 7] = fmaxf(mx8[k & 7], v);
    }
    float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                     fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
    red[(stage * 2 + half) * kBM + row] = mx;
    named_bar_sync(1, kSmxThreads);
    mx = fmaxf(mx, red[(stage * 2 + (half ^ 1)) * kBM + row]);

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
    // A row that has seen no visible key yet (possible inside a band) keeps
    // m_used = -inf and all its scores at -inf: its p are 0, not NaN.
    const float mu = m_used == -INFINITY ? 0.f : m_used;
    uint32_t pk[32];
    float ps[4] = {0.f, 0.f, 0.f, 0.f}, ra, rb;
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      pk[k] = Pack<T>::run(fast_exp2(s[2 * k] - mu), fast_exp2(s[2 * k + 1] - mu), ra, rb);
      ps[k & 3] += ra + rb;
    }
    l = l * corr + ((ps[0] + ps[1]) + (ps[2] + ps[3]));

    if (j > 0) {
      wait_tc(&bars[kPVDone], (j - 1) & 1, abort_flag, p.err_flag);
      tc_fence_after();
    }
    if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float v[16];
        const uint32_t a = lane_base + kTmemO + half * (D / 2) + c * 16;
        tmem_ld16(a, v);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] *= corr;
        tmem_st16(a, v);
      }
      tmem_wait_st();
    }
    // P -> shared memory: chunk `half` holds tokens half*64 .. +63 of the tile.
    uint8_t* pc = smem + L::kP + half * kChunk;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch)
      *reinterpret_cast<uint4*>(pc + swz128(row, ch)) =
          make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
    // Value rows past the cached tokens, and rows before the band of the
    // tile's first query row (seen by no row), are zeroed so stale cache
    // contents cannot reach P V.
    const int valid = kv_len - (j0 + j) * kBN;
    const int zlo = band_start(ctx + q0, p.window) - (j0 + j) * kBN;
    if (valid < kBN || zlo > 0) {
      wait_tc(&bars[kVFull0 + stage], (j >> 1) & 1, abort_flag, p.err_flag);
      uint8_t* vst = smem + L::kV + stage * L::kStageBytes;
      const int top = valid < kBN ? kBN - valid : 0, bottom = zlo > 0 ? min(zlo, kBN) : 0;
      const int n16 = (top + bottom) * L::kHalves * 8;
      for (int e = t; e < n16; e += kSmxThreads) {
        const int i = e / (L::kHalves * 8), c = (e / 8) % L::kHalves, q = e % 8;
        const int r = i < bottom ? i : valid + (i - bottom);
        *reinterpret_cast<uint4*>(vst + c * kChunk + r * 128 + q * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    mbar_arrive(&bars[kPFull]);
  }

  // Epilogue: combine the pair's row sums, normalise, write this row's half.
  // The P buffer is no longer read once the last P V is done: 2 KB of it per
  // warp stage the warp's 32 rows, 32 columns at a time (16-byte chunk q of
  // row r at r*64 + (q ^ ((r >> 1) & 3))*16: no bank conflicts either way),
  // so that a store instruction writes 8 rows x 64 contiguous bytes rather
  // than 32 rows x 16 bytes.
  wait_tc(&bars[kPVDone], (n_tiles - 1) & 1, abort_flag, p.err_flag);
  tc_fence_after();
  const int rb = n_tiles & 1;  // the reduction buffer not used by the last tile
  red[(rb * 2 + half) * kBM + row] = l;
  named_bar_sync(1, kSmxThreads);
  const float lt = l + red[(rb * 2 + (half ^ 1)) * kBM + row];
  const float inv = lt > 0.f ? 1.f / lt : 0.f;
  uint8_t* stg = smem + L::kP + warp * 2048;
  const int wrow0 = quad * 32;
  const long long ostride = static_cast<long long>(p.num_q_heads) * D;
  T* obase = static_cast<T*>(p.out) + (static_cast<long long>(tok0) + wrow0) * ostride + h * D +
             half * (D / 2);
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {  // two TMEM loads in flight per wait
    float v[32];
    tmem_ld16(lane_base + kTmemO + half * (D / 2) + c * 32, v);
    tmem_ld16(lane_base + kTmemO + half * (D / 2) + c * 32 + 16, v + 16);
    tmem_wait_ld();
    uint32_t w[16];
    float a, b;
#pragma unroll
    for (int k = 0; k < 16; ++k) w[k] = Pack<T>::run(v[2 * k] * inv, v[2 * k + 1] * inv, a, b);
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<uint4*>(stg + lane * 64 + ((q ^ ((lane >> 1) & 3)) * 16)) =
          make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    __syncwarp();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int r = i * 8 + (lane >> 2), q = lane & 3;
      const uint4 val =
          *reinterpret_cast<const uint4*>(stg + r * 64 + ((q ^ ((r >> 1) & 3)) * 16));
      if (wrow0 + r < q_rows) *reinterpret_cast<uint4*>(obase + r * ostride + c * 32 + q * 8) = val;
    }
    __syncwarp();
  }
  tc_fence_before();
}

template <typename T, int D, bool kBf16>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ TcPrefillParams p) {
  using L = TcLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  int* info = reinterpret_cast<int*>(smem + L::kMisc + 16);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x % p.num_q_heads;
  const int item = blockIdx.x / p.num_q_heads;

  if (warp == 0) {
    int s = 0, tile = 0, ctx = 0, len = 0;
    const bool found = tc_locate(p, item, lane, s, tile, ctx, len);
    if (lane == 0) {
      info[0] = found ? s : -1;
      info[1] = tile;
      info[2] = ctx;
      info[3] = len;
      const uint32_t counts[L::kNumBars] = {1, 1, 1, 1, 1, 1, 1, kSmxThreads, kSmxThreads,
                                            kSmxThreads, 1, 1, 1, 1, 1, 1};
      for (int i = 0; i < L::kNumBars; ++i) mbar_init(&bars[i], counts[i]);
      *abort_flag = 0;
      fence_barrier_init();
    }
  }
  __syncthreads();
  const int s = info[0];
  if (s < 0) return;  // grid slots beyond the real number of tiles
  const int q0 = info[1] * kBM, ctx = info[2], len = info[3];
  const int q_rows = min(kBM, len - q0);
  const int kv_len = ctx + len;
  if (kv_len > p.max_blocks * p.block_size) {  // table too short: flag, write nothing
    if (tid == 0) set_flag(p.err_flag, KVC_FLAG_LEN_RANGE);
    return;
  }
  // Key tiles j0 .. j0 + n_tiles - 1: from the tile holding the band start of
  // the first query row to the tile holding the last row.
  const int band0 = band_start(ctx + q0, p.window);
  const int j0 = band0 / kBN;
  const int n_tiles = (ctx + q0 + q_rows - 1) / kBN + 1 - j0;
  const int tok0 = p.cu_seqlens[s] + q0;

  uint32_t leader = 0;  // the MMA warp's issuing lane
  if (warp == kMmaWarp) {
    tmem_alloc(tslot, kTmemCols);
    leader = elect_one_sync();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp < kProducerWarp) {
    tc_softmax<T, D>(p, smem, bars, abort_flag, tmem, tid, j0, n_tiles, q0, ctx, kv_len, q_rows,
                     tok0, h);
  } else if (warp == kProducerWarp) {
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
    }
    tc_producer<D>(p, &tm_q, &tm_k, &tm_v, smem, bars, abort_flag, s, h, h / p.group, tok0, kv_len,
                   j0, n_tiles, band0, lane);
  } else {
    tc_mma<D, kBf16>(p, smem, bars, abort_flag, tmem, n_tiles, leader);
  }
  // Teardown: all tensor-core work done before TMEM is freed.
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
}

template <typename T, int D, bool kBf16>
kvc_status run_prefill_tc(const PrefillArgs& a) {
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(prefill_tc_kernel<T, D, kBf16>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize, TcLayout<D>::kTotal);
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
  if (!encode_tmap_16bit(&tq, a.dtype, 3, a.q, qdims, qstrides, qbox, true) ||
      !encode_tmap_16bit(&tk, a.dtype, 4, a.key_cache, dims, strides, box, true) ||
      !encode_tmap_16bit(&tv, a.dtype, 4, a.value_cache, dims, strides, box, true))
    return KVC_ERR_CUDA;
  TcPrefillParams p;
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
  // Upper bound of query tiles: sum ceil(L_s / BM) <= T / BM + S.
  const long long grid = (static_cast<long long>(a.num_tokens) / kBM + a.num_seqs) * a.num_q_heads;
  if (grid > 0x7fffffffLL) return KVC_ERR_UNSUPPORTED;
  prefill_tc_kernel<T, D, kBf16><<<static_cast<unsigned>(grid), kThreads, TcLayout<D>::kTotal,
                                   a.stream>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

}  // namespace

kvc_status launch_prefill_attention_tc(const PrefillArgs& a) {
  if (a.head_dim == 64)
    return a.dtype == KVC_BF16 ? run_prefill_tc<__nv_bfloat16, 64, true>(a)
                               : run_prefill_tc<__half, 64, false>(a);
  if (a.head_dim == 128)
    return a.dtype == KVC_BF16 ? run_prefill_tc<__nv_bfloat16, 128, true>(a)
                               : run_prefill_tc<__half, 128, false>(a);
  return KVC_ERR_UNSUPPORTED;
}

}  // namespace kvc
