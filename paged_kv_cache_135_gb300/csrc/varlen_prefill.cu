// Packed-varlen causal prefill over the paged cache (row a5 of the hot path).
//
// What it computes: the hotelren.com notes "Paged KV Cache + Packed
// Sequence" 3.1-3.3 -- sequences are packed along the token axis and
// delimited by cu_seqlens (seq_offset); every token attends causally to the
// tokens of its own sequence only, and the K/V it attends to are read back
// from the paged cache through the sequence's block_table (packed token ->
// request and offset -> logical block -> physical block).  The call first
// writes the chunk's own K/V rows into the cache at slot_mapping (ai6s.net
// KVCache article 4.2), as "external-cannbot-model-model-infer-kvcache" 3.6
// has every layer write its cache before FA reads it; causality is
// sparse_mode 3 of its Appendix C, with the diagonal included.
//
// GB300 design: one CTA per (sequence, 128-query tile, q head), heaviest
// tiles of a sequence first, heads fastest so that CTAs sharing K/V run
// together.  A producer warp loads the query tile once and streams 64-token
// K/V tiles through block_table with TMA into a 3-stage mbarrier ring
// (128-byte swizzled, the table entry is the box's block coordinate); eight
// consumer warps (16 query rows each) run S = Q K^T and O += P V with
// mma.sync m16n8k16 (fp32 accumulation), an online softmax in the log2 domain
// with the causal predicate computed from positions, and skip K/V tiles that
// lie wholly in their future.
#include <cuda_runtime.h>

#include <math.h>

#include <map>
#include <mutex>
#include <utility>

#include "kvc_device.cuh"
#include "kvc_host.h"

namespace kvc {

namespace {

constexpr int kBM = 128;            // query rows per CTA
constexpr int kBN = 64;             // kv positions per stage
constexpr int kWarps = kBM / 16;    // consumer warps
constexpr int kThreads = (kWarps + 1) * 32;
constexpr int kStages = 3;
constexpr int kHalfBytes = kBN * 128;  // one 64-element half of a K or V tile

struct PrefillParams {
  void* out;
  const int32_t* cu_seqlens;
  const int32_t* context_lens;  // may be null (all zero)
  const int32_t* block_table;
  uint32_t* err_flag;
  int num_seqs, num_tokens, num_q_heads, group;
  int block_size, log2_bs, max_blocks, num_blocks, box_tokens;
  float scale_log2;
};

template <int D>
struct PLayout {
  static constexpr int kHalves = D / 64;
  static constexpr int kQBytes = kHalves * kBM * 128;
  static constexpr int kKBytes = kHalves * kHalfBytes;
  static constexpr int kStageBytes = 2 * kKBytes;
  static constexpr int kStagesOff = kQBytes;
  static constexpr int kBarOff = kStagesOff + kStages * kStageBytes;  // qbar, full[], empty[]
  static constexpr int kInfoOff = kBarOff + (1 + 2 * kStages) * 8;    // s, tile, ctx, len
  static constexpr int kTotal = 1024 + kInfoOff + 64;
};

__device__ __forceinline__ uint32_t keep_rows(uint32_t x, int k, int valid) {
  const uint32_t lo = k < valid ? 0x0000FFFFu : 0u;
  const uint32_t hi = k + 1 < valid ? 0xFFFF0000u : 0u;
  return x & (lo | hi);
}

// Work item -> (sequence, query tile).  Items enumerate the tiles of each
// sequence from its last (heaviest under the causal mask) to its first.
// One warp scans cu_seqlens 32 sequences at a time.
__device__ __forceinline__ bool locate_item(const PrefillParams& p, int item, int lane, int& s,
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
    const int lo = before + x - n;  // first item of sequence i
    const unsigned hit = __ballot_sync(0xffffffffu, i < p.num_seqs && item >= lo && item < lo + n);
    if (hit) {
      const int src = __ffs(hit) - 1;
      s = base + src;
      const int k = item - __shfl_sync(0xffffffffu, lo, src);
      const int ns = __shfl_sync(0xffffffffu, n, src);
      tile = ns - 1 - k;
      len = __shfl_sync(0xffffffffu, L, src);
      ctx = p.context_lens ? p.context_lens[s] : 0;
      return true;
    }
    before += __shfl_sync(0xffffffffu, x, 31);
  }
  return false;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    varlen_prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ PrefillParams p) {
  using L = PLayout<D>;
  constexpr int kHalves = L::kHalves;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* qbar = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* full = qbar + 1;
  uint64_t* empty = full + kStages;
  int* info = reinterpret_cast<int*>(smem + L::kInfoOff);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x % p.num_q_heads;
  const int item = blockIdx.x / p.num_q_heads;
  const int g = h / p.group;

  if (warp == 0) {
    int s = 0, tile = 0, ctx = 0, len = 0;
    const bool found = locate_item(p, item, lane, s, tile, ctx, len);
    if (lane == 0) {
      info[0] = found ? s : -1;
      info[1] = tile;
      info[2] = ctx;
      info[3] = len;
      mbar_init(qbar, 1);
      for (int i = 0; i < kStages; ++i) {
        mbar_init(&full[i], 1);
        mbar_init(&empty[i], kWarps);
      }
      fence_barrier_init();
    }
  }
  __syncthreads();
  const int s = info[0];
  if (s < 0) return;  // grid slots beyond the real number of tiles
  const int tile = info[1], ctx = info[2], len = info[3];
  const int q0 = tile * kBM;                       // first query row (within the sequence)
  const int q_rows = min(kBM, len - q0);           // real query rows of this tile
  const int kv_len = ctx + len;                    // positions cached for this sequence
  if (kv_len > p.max_blocks * p.block_size) {      // table too short: flag, write nothing
    if (tid == 0) set_flag(p.err_flag, KVC_FLAG_LEN_RANGE);
    return;
  }
  const int pos_last = ctx + q0 + q_rows - 1;      // last query position of the tile
  const int n_kv_tiles = pos_last / kBN + 1;
  const int tok0 = p.cu_seqlens[s] + q0;           // packed index of the first query row

  if (warp == kWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      mbar_arrive_expect_tx(qbar, kHalves * kBM * 128);
#pragma unroll
      for (int hh = 0; hh < kHalves; ++hh)
        tma_load_3d(smem + hh * kBM * 128, &tm_q, qbar, hh * 64, h, tok0);
    }
    const int nsub = kBN / p.box_tokens;
    const uint32_t box_bytes = static_cast<uint32_t>(p.box_tokens) * 128u;
    for (int j = 0; j < n_kv_tiles; ++j) {
      const int stage = j % kStages;
      const uint32_t phase = (j / kStages) & 1;
      const int tok = j * kBN + lane * p.box_tokens;
      int pb = -1;
      if (lane < nsub && tok < kv_len)
        pb = __ldg(&p.block_table[static_cast<long long>(s) * p.max_blocks + (tok >> p.log2_bs)]);
      const bool ok = mbar_wait_bounded(&empty[stage], phase ^ 1, p.err_flag);
      bool valid = false;
      if (lane < nsub && tok < kv_len) {
        if (pb < 0 || pb >= p.num_blocks) set_flag(p.err_flag, KVC_FLAG_BLOCK_ID_RANGE);
        else valid = true;
      }
      valid = valid && ok;
      const uint32_t nvalid = __popc(__ballot_sync(0xffffffffu, valid));
      if (lane == 0) mbar_arrive_expect_tx(&full[stage], nvalid * box_bytes * kHalves * 2);
      __syncwarp();
      if (valid) {
        uint8_t* kdst = smem + L::kStagesOff + stage * L::kStageBytes + lane * box_bytes;
        const int in_blk = tok & (p.block_size - 1);
#pragma unroll
        for (int hh = 0; hh < kHalves; ++hh) {
          tma_load_4d(kdst + hh * kHalfBytes, &tm_k, &full[stage], hh * 64, g, in_blk, pb);
          tma_load_4d(kdst + L::kKBytes + hh * kHalfBytes, &tm_v, &full[stage], hh * 64, g,
                      in_blk, pb);
        }
      }
    }
    // Drain: wait for the last copies before shared memory can go away.
    for (int j = max(0, n_kv_tiles - kStages); j < n_kv_tiles; ++j)
      mbar_wait_bounded(&full[j % kStages], (j / kStages) & 1, p.err_flag);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int mi = lane >> 3, rr = lane & 7, c0 = 2 * (lane & 3);
  const int wrow0 = warp * 16;                                // first row of this warp
  const int pos_r0 = ctx + q0 + wrow0 + (lane >> 2);          // position of row lane/4
  const int pos_r1 = pos_r0 + 8;
  const int warp_pos_max = ctx + q0 + wrow0 + 15;
  const bool warp_active = wrow0 < q_rows;  // warps wholly past the sequence do nothing

  // Query fragments stay in registers for the whole CTA.
  const bool q_ok = mbar_wait_bounded(qbar, 0, p.err_flag);
  uint32_t qa[D / 16][4];
  {
    const uint32_t qb = smem_u32(smem);
    const int qr = wrow0 + (mi & 1) * 8 + rr;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      ldsm_x4(qb + (kk >> 2) * (kBM * 128) + swz128(qr, (kk & 3) * 2 + (mi >> 1)), qa[kk][0],
              qa[kk][1], qa[kk][2], qa[kk][3]);
  }
  float o[D / 8][4], m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
#pragma unroll
  for (int n = 0; n < D / 8; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[n][e] = 0.f;

  const uint32_t sbase = smem_u32(smem + L::kStagesOff);
  bool alive = q_ok;
  for (int j = 0; j < n_kv_tiles; ++j) {
    const int stage = j % kStages;
    const uint32_t phase = (j / kStages) & 1;
    if (alive) alive = mbar_wait_bounded(&full[stage], phase, p.err_flag);
    const int kv0 = j * kBN;
    if (alive && warp_active && kv0 <= warp_pos_max) {
      const uint32_t kb = sbase + stage * L::kStageBytes, vb = kb + L::kKBytes;
      float sc[kBN / 8][4];
#pragma unroll
      for (int n = 0; n < kBN / 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[n][e] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int dcol = kk * 16 + (mi & 1) * 8;
#pragma unroll
        for (int np = 0; np < kBN / 16; ++np) {
          const int tok = np * 16 + (mi >> 1) * 8 + rr;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(kb + (dcol >> 6) * kHalfBytes + swz128(tok, (dcol & 63) >> 3), b0, b1, b2, b3);
          MmaOp<T>::run(sc[2 * np], qa[kk], b0, b1);
          MmaOp<T>::run(sc[2 * np + 1], qa[kk], b2, b3);
        }
      }
      // causal + length mask, then the online softmax update
      const bool need_mask = kv0 + kBN - 1 > ctx + q0 + wrow0 || kv0 + kBN > kv_len;
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int n = 0; n < kBN / 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = kv0 + n * 8 + c0 + (e & 1);
          const int pr = e < 2 ? pos_r0 : pos_r1;
          float v = sc[n][e] * p.scale_log2;
          if (need_mask && (key > pr || key >= kv_len)) v = -INFINITY;
          sc[n][e] = v;
        }
#pragma unroll
      for (int n = 0; n < kBN / 8; ++n) {
        mx0 = fmaxf(mx0, fmaxf(sc[n][0], sc[n][1]));
        mx1 = fmaxf(mx1, fmaxf(sc[n][2], sc[n][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
      // A row can see no key of this tile while having seen earlier ones (never
      // none at all: position 0 is always visible); keep exp2 arguments finite.
      const float ms0 = mn0 == -INFINITY ? 0.f : mn0, ms1 = mn1 == -INFINITY ? 0.f : mn1;
      const float corr0 = fast_exp2(m[0] - ms0), corr1 = fast_exp2(m[1] - ms1);
      m[0] = mn0;
      m[1] = mn1;
      uint32_t pa[kBN / 16][4];
      float rs0 = 0.f, rs1 = 0.f, ra, rb;
#pragma unroll
      for (int ks = 0; ks < kBN / 16; ++ks) {
        pa[ks][0] = Pack<T>::run(fast_exp2(sc[2 * ks][0] - ms0), fast_exp2(sc[2 * ks][1] - ms0),
                                 ra, rb);
        rs0 += ra + rb;
        pa[ks][1] = Pack<T>::run(fast_exp2(sc[2 * ks][2] - ms1), fast_exp2(sc[2 * ks][3] - ms1),
                                 ra, rb);
        rs1 += ra + rb;
        pa[ks][2] = Pack<T>::run(fast_exp2(sc[2 * ks + 1][0] - ms0),
                                 fast_exp2(sc[2 * ks + 1][1] - ms0), ra, rb);
        rs0 += ra + rb;
        pa[ks][3] = Pack<T>::run(fast_exp2(sc[2 * ks + 1][2] - ms1),
                                 fast_exp2(sc[2 * ks + 1][3] - ms1), ra, rb);
        rs1 += ra + rb;
      }
      l[0] = l[0] * corr0 + rs0;
      l[1] = l[1] * corr1 + rs1;
#pragma unroll
      for (int n = 0; n < D / 8; ++n) {
        o[n][0] *= corr0;
        o[n][1] *= corr0;
        o[n][2] *= corr1;
        o[n][3] *= corr1;
      }
      const int kv_valid = kv_len - kv0;  // rows of this tile that hold cached tokens
#pragma unroll
      for (int ks = 0; ks < kBN / 16; ++ks) {
        const int tok = ks * 16 + (mi & 1) * 8 + rr;
#pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          const int dcol = dp * 16 + (mi >> 1) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vb + (dcol >> 6) * kHalfBytes + swz128(tok, (dcol & 63) >> 3), b0, b1, b2,
                    b3);
          if (kv_valid < kBN) {
            b0 = keep_rows(b0, ks * 16 + c0, kv_valid);
            b1 = keep_rows(b1, ks * 16 + 8 + c0, kv_valid);
            b2 = keep_rows(b2, ks * 16 + c0, kv_valid);
            b3 = keep_rows(b3, ks * 16 + 8 + c0, kv_valid);
          }
          MmaOp<T>::run(o[2 * dp], pa[ks], b0, b1);
          MmaOp<T>::run(o[2 * dp + 1], pa[ks], b2, b3);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
  }

  // Normalise and write this warp's real rows.
  float l0 = l[0], l1 = l[1];
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
  T* out = static_cast<T*>(p.out);
  const int r0 = wrow0 + (lane >> 2), r1 = r0 + 8;
  const long long row_stride = static_cast<long long>(p.num_q_heads) * D;
  float ra, rb;
#pragma unroll
  for (int n = 0; n < D / 8; ++n) {
    if (r0 < q_rows)
      *reinterpret_cast<uint32_t*>(out + (tok0 + r0) * row_stride + h * D + n * 8 + c0) =
          Pack<T>::run(o[n][0] * inv0, o[n][1] * inv0, ra, rb);
    if (r1 < q_rows)
      *reinterpret_cast<uint32_t*>(out + (tok0 + r1) * row_stride + h * D + n * 8 + c0) =
          Pack<T>::run(o[n][2] * inv1, o[n][3] * inv1, ra, rb);
  }
}

template <typename T, int D>
kvc_status run_prefill(const PrefillArgs& a) {
  static std::once_flag once;
  std::call_once(once, [] {
    cudaFuncSetAttribute(varlen_prefill_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         PLayout<D>::kTotal);
  });
  const int G = a.num_q_heads / a.num_kv_heads;
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
  PrefillParams p;
  p.out = a.out;
  p.cu_seqlens = a.cu_seqlens;
  p.context_lens = a.context_lens;
  p.block_table = a.block_table;
  p.err_flag = a.err_flag;
  p.num_seqs = a.num_seqs;
  p.num_tokens = a.num_tokens;
  p.num_q_heads = a.num_q_heads;
  p.group = G;
  p.block_size = a.block_size;
  p.log2_bs = ilog2(a.block_size);
  p.max_blocks = a.max_blocks_per_seq;
  p.num_blocks = a.num_blocks;
  p.box_tokens = box_tokens;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  // Upper bound of query tiles: sum ceil(L_s / BM) <= T / BM + S.
  const long long items = static_cast<long long>(a.num_tokens) / kBM + a.num_seqs;
  const long long grid = items * a.num_q_heads;
  if (grid > 0x7fffffffLL) return KVC_ERR_UNSUPPORTED;
  varlen_prefill_kernel<T, D><<<static_cast<unsigned>(grid), kThreads, PLayout<D>::kTotal,
                                a.stream>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

}  // namespace

kvc_status launch_varlen_prefill(const PrefillArgs& a) {
  // 1. The chunk's own K/V rows go into the cache (bit-exact row copies).
  kvc_status st = launch_reshape_and_cache(a.key, a.value, a.key_cache, a.value_cache,
                                           a.slot_mapping, a.num_tokens, a.num_kv_heads,
                                           a.head_dim, a.head_dim, a.block_size, a.num_blocks,
                                           a.err_flag, a.stream);
  if (st != KVC_OK) return st;
  // 2. Causal attention of every packed token over its sequence's cache.
  if (a.head_dim == 64)
    return a.dtype == KVC_BF16 ? run_prefill<__nv_bfloat16, 64>(a) : run_prefill<__half, 64>(a);
  if (a.head_dim == 128)
    return a.dtype == KVC_BF16 ? run_prefill<__nv_bfloat16, 128>(a) : run_prefill<__half, 128>(a);
  return KVC_ERR_UNSUPPORTED;
}

}  // namespace kvc
