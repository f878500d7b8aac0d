// Paged decode attention with split-KV and its in-kernel merge.
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
//    the CTA that finishes its share last (an atomic arrival counter per
//    split segment) merges them in a fixed order -- no second kernel, no
//    spin-wait, deterministic and independent of physical block IDs.
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
// Pipeline depth: 3 stages of ~33 KB (16-bit cache) or 4 of ~17 KB (INT8,
// whose stages also hold scales; 4 keeps two CTAs per SM).
template <bool kI8>
constexpr int stages_of() { return kI8 ? 4 : 3; }
constexpr int kMaxBatch = 1024;
constexpr int kHalfBytes = kTile * 128;  // one 64-element half of a K or V tile
constexpr int kMaxPieces = 62;           // split shares merged from a shared-memory list
// INT8 cache: a tile's per-token scales arrive as one TMA box per physical
// block (min(block_size, 64) floats); each box gets its own 128-byte slot.
constexpr int kScaleBytes = (kTile / 8) * 128;

struct DecodeParams {
  const void* q;
  void* out;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int* ws_cnt;   // [P][2] arrival counters of split segments (zero between calls)
  float* ws_o;   // [P][2][G][D] unnormalised partial outputs
  float* ws_ml;  // [P][2][G][2] partial (max, sum) in the log2 domain
  uint32_t* err_flag;
  // Appending variant (null = plain decode): the new token of sequence b sits
  // at position seq_lens[b] - 1; its K/V rows come from new_k / new_v
  // [B, Hkv, D] and are written into k_cache / v_cache by the CTA that loads
  // that position, before it loads it; slot_out[b] (nullable) gets its slot.
  const void* new_k;
  const void* new_v;
  void* k_cache;
  void* v_cache;
  int32_t* slot_out;
  int batch, num_q_heads, num_kv_heads, group, head_dim;
  int block_size, log2_bs, max_blocks, num_blocks, box_tokens, log2_box;
  int window;  // band of the last `window` cached tokens (0: the whole sequence)
  float scale_log2;
};

__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

// Dynamic shared memory of the decode kernel.  A stage holds the K tile, the
// V tile and the query rows of the tile's (b, g) (all 128-byte swizzled, each
// 1024-byte aligned as the TMA swizzle requires); every other region starts
// on a 16-byte boundary.  Over an INT8 cache (kI8) the K and V tiles hold the
// int8 codes (one 128-byte row per token), the stage also holds the tile's
// per-token K and V scales, and each consumer warp owns a staging tile for
// its 16 value rows converted to 16 bits.
template <int D, bool kI8>
struct Layout {
  static constexpr int kHalves = D / 64;  // 64-element halves of a 16-bit row
  static constexpr int kKBytes = kI8 ? kTile * D : kHalves * kHalfBytes;  // one K or V tile
  int q_half;   // bytes of one 64-wide half of the G query rows (1024-aligned)
  int scales;   // INT8: K scales then V scales of the stage, kTile floats each
  int qoff;     // query rows of the stage (1024-aligned)
  int vstg;     // INT8: per consumer warp, its 16 value rows as 16-bit values
  int qfrag;    // INT8: the segment's fp16 query fragments, [D/16][32 lanes][4 words]
  int stage;    // K tile, V tile, (scales), query rows
  static constexpr int kStages = stages_of<kI8>();
  int bar;      // full[kStages], empty[kStages]
  int flags;    // abort, last, npieces
  int pieces;   // int[kMaxPieces]
  int lens;     // int[batch]
  int cum;      // int[batch + 1]
  int cmb;      // cross-warp combine: m[4G], l[4G], o[4G][D]
  int total;    // bytes to request (with 1024 bytes of alignment slack)
  __host__ __device__ Layout(int batch, int group) {
    q_half = align_up(group * 128, 1024);
    scales = 2 * kKBytes;
    qoff = kI8 ? align_up(scales + 2 * kScaleBytes, 1024) : 2 * kKBytes;
    stage = qoff + kHalves * q_half;
    bar = kStages * stage;
    flags = bar + 2 * kStages * 8;
    pieces = align_up(flags + 12, 16);
    lens = align_up(pieces + kMaxPieces * 4, 16);
    cum = align_up(lens + batch * 4, 16);
    cmb = align_up(cum + (batch + 1) * 4, 16);
    vstg = align_up(cmb + kConsumerWarps * group * (D + 2) * 4, 1024);
    qfrag = vstg + kConsumerWarps * 16 * D * 2;
    total = 1024 + (kI8 ? qfrag + (D / 16) * 32 * 16
                        : cmb + kConsumerWarps * group * (D + 2) * 4);
  }
};

// Arrival counters at the head of the workspace, padded to 256 bytes.
__host__ __device__ inline size_t counter_bytes(int ctas) {
  return (static_cast<size_t>(ctas) * 2 * sizeof(int) + 255) & ~static_cast<size_t>(255);
}

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

// Rows k and k + 1 of a value fragment (low and high 16 bits) kept if they lie
// in [vlo, valid), zeroed otherwise.
__device__ __forceinline__ uint32_t keep_rows(uint32_t x, int k, int vlo, int valid) {
  const uint32_t lo = k >= vlo && k < valid ? 0x0000FFFFu : 0u;
  const uint32_t hi = k + 1 >= vlo && k + 1 < valid ? 0xFFFF0000u : 0u;
  return x & (lo | hi);
}

// Band attention (sliding window): a sequence of L cached tokens attends to
// positions band_lo .. L-1 only, the last `window` of them (0: all).  Its
// tiles start at the 64-token tile holding band_lo.
__device__ __forceinline__ int band_lo(int L, int window) {
  return window > 0 && L > window ? L - window : 0;
}
__device__ __forceinline__ int first_tile(int L, int window) { return band_lo(L, window) / kTile; }

// out[0..3] = v * inv, rounded to T (one 8-byte store).
template <typename T>
__device__ __forceinline__ void store4(T* dst, float4 v, float inv) {
  float a, b;
  uint2 w;
  w.x = Pack<T>::run(v.x * inv, v.y * inv, a, b);
  w.y = Pack<T>::run(v.z * inv, v.w * inv, a, b);
  *reinterpret_cast<uint2*>(dst) = w;
}

// One warp's 16 tokens of a stage: S = Q K^T, online softmax, O += P V.
template <typename T, int D>
__device__ __forceinline__ void attend_16(uint32_t kbase, uint32_t vbase, int warp, int lane,
                                          int vlo, int valid, float scale_log2, uint32_t qbase,
                                          int q_half, int group, float (&o)[D / 8][4],
                                          float (&m)[2], float (&l)[2]) {
  const int mi = lane >> 3, rr = lane & 7;
  float s[2][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) s[i][e] = 0.f;
  {
    const int tok = warp * 16 + (mi >> 1) * 8 + rr;
    // Query rows >= G are padding: they read row 0 and their results are dropped.
    const int qr = (mi & 1) * 8 + rr < group ? (mi & 1) * 8 + rr : 0;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int dcol = kk * 16 + (mi & 1) * 8;
      uint32_t a[4], b0, b1, b2, b3;
      ldsm_x4(qbase + (kk >> 2) * q_half + swz128(qr, (kk & 3) * 2 + (mi >> 1)), a[0], a[1],
              a[2], a[3]);
      ldsm_x4(kbase + (dcol >> 6) * kHalfBytes + swz128(tok, (dcol & 63) >> 3), b0, b1, b2, b3);
      MmaOp<T>::run(s[0], a, b0, b1);
      MmaOp<T>::run(s[1], a, b2, b3);
    }
  }
  const int c0 = 2 * (lane & 3);
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int k = nt * 8 + c0 + (e & 1);
      s[nt][e] = k >= vlo && k < valid ? s[nt][e] * scale_log2 : -INFINITY;
    }
  float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
  float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
  const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
  const bool grew = mn0 != m[0] || mn1 != m[1];
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
  if (__any_sync(0xffffffffu, grew)) {  // O keeps its scale while no row max grows
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      o[n][0] *= corr0;
      o[n][1] *= corr0;
      o[n][2] *= corr1;
      o[n][3] *= corr1;
    }
  }
  const int tok = warp * 16 + (mi & 1) * 8 + rr;
#pragma unroll
  for (int dp = 0; dp < D / 16; ++dp) {
    const int dcol = dp * 16 + (mi >> 1) * 8;
    uint32_t b0, b1, b2, b3;
    ldsm_x4_t(vbase + (dcol >> 6) * kHalfBytes + swz128(tok, (dcol & 63) >> 3), b0, b1, b2, b3);
    if (valid < 16 || vlo > 0) {
      b0 = keep_rows(b0, c0, vlo, valid);
      b1 = keep_rows(b1, 8 + c0, vlo, valid);
      b2 = keep_rows(b2, c0, vlo, valid);
      b3 = keep_rows(b3, 8 + c0, vlo, valid);
    }
    MmaOp<T>::run(o[2 * dp], pa, b0, b1);
    MmaOp<T>::run(o[2 * dp + 1], pa, b2, b3);
  }
}

// ---- INT8 cache: codes to 16-bit values, scales, and one warp's 16 tokens.

__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ void sts_v4(uint32_t a, uint32_t x, uint32_t y, uint32_t z,
                                       uint32_t w) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z),
               "r"(w)
               : "memory");
}
__device__ __forceinline__ float lds_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}

// Four int8 codes (one 32-bit word, byte k = element k) as two fp16 pairs,
// exactly: each code c (|c| <= 127) is biased to the byte c + 128, placed as
// the low mantissa byte of the fp16 1024 + (c + 128), and 1152 is subtracted
// (both steps exact).  lo = elements 0, 1; hi = elements 2, 3.
__device__ __forceinline__ void i8x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t x = w ^ 0x80808080u;
  const uint32_t a = __byte_perm(x, 0x64646464u, 0x4140u);
  const uint32_t b = __byte_perm(x, 0x64646464u, 0x4342u);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  const __half2 ra = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
  const __half2 rb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
  lo = *reinterpret_cast<const uint32_t*>(&ra);
  hi = *reinterpret_cast<const uint32_t*>(&rb);
}

// A pair of 16-bit query values as an fp16 pair: unchanged for fp16; for bf16
// exact whenever the values lie in fp16's normal range (|q| in [2^-14, 65504]),
// since a bf16 significand (8 bits) fits fp16's (11 bits).
template <typename T>
__device__ __forceinline__ uint32_t q_pair_f16(uint32_t w);
template <>
__device__ __forceinline__ uint32_t q_pair_f16<__half>(uint32_t w) { return w; }
template <>
__device__ __forceinline__ uint32_t q_pair_f16<__nv_bfloat16>(uint32_t w) {
  const __half2 h = __floats2half2_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Address of token t's scale in a stage's scale region (one 128-byte slot per
// TMA box of 2^log2_box tokens).
__device__ __forceinline__ uint32_t scale_addr(uint32_t base, int t, int log2_box) {
  return base + ((t >> log2_box) << 7) + ((t & ((1 << log2_box) - 1)) << 2);
}

// The query fragments of S = Q K^T over an INT8 cache, in fp16 and with the
// 16 dims of every k-step permuted: lane (g = lane/4, c = lane%4) holds dims
// 16kk + 4c .. 4c+3 of query rows g and g + 8, so that its key operand is the
// 4 contiguous codes at the same dims (one 32-bit load).  The dot product does
// not depend on the order of its terms.  Rows >= G are padding and read row
// 0.  They are the same for every consumer warp and every tile of a (b, g)
// segment: at the segment's first tile each warp builds two k-steps of them
// (from the stage's query rows) into shared memory, [kk][lane] as 16 bytes.
template <typename T, int D>
__device__ __forceinline__ void build_q_i8(uint32_t qbase, int q_half, int group, int warp,
                                           int lane, uint32_t qfrag) {
  const int g = lane >> 2, c = lane & 3;
  const int r0 = g < group ? g : 0, r1 = g + 8 < group ? g + 8 : 0;
#pragma unroll
  for (int i = 0; i < D / 16 / kConsumerWarps; ++i) {
    const int kk = warp * (D / 16 / kConsumerWarps) + i;
    const uint32_t off = (kk >> 2) * q_half;
    const int chunk = (kk & 3) * 2 + (c >> 1), byte = (c & 1) * 8;
    uint32_t w0, w1, w2, w3;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                 : "=r"(w0), "=r"(w1) : "r"(qbase + off + swz128(r0, chunk) + byte));
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                 : "=r"(w2), "=r"(w3) : "r"(qbase + off + swz128(r1, chunk) + byte));
    // a0: row g dims 4c, 4c+1; a1: row g+8 same; a2: row g dims 4c+2, 4c+3; a3: row g+8 same
    sts_v4(qfrag + (kk * 32 + lane) * 16, q_pair_f16<T>(w0), q_pair_f16<T>(w2), q_pair_f16<T>(w1),
           q_pair_f16<T>(w3));
  }
}

// One warp's 16 tokens of a stage over an INT8 cache.  A cached row is
// code * scale, so q . k = scale_k * (q . codes_k) and sum_j p_j v_j =
// sum_j (p_j * scale_v_j) codes_v_j.  Both products run on the tensor cores
// in fp16 with fp32 accumulation: the codes are exact in fp16, the queries
// are (qa, see load_q_i8), and the weights p * scale_v keep 11 bits (l sums
// the plain p, so the weights are not renormalised after rounding).  Each
// score column is multiplied by its key scale.  The warp's 16 value rows are
// first converted into `vst`, in the layout of a 16-bit tile, so P V reads
// them with ldmatrix.trans as the 16-bit path does.
template <int D>
__device__ __forceinline__ void attend_16_i8(uint32_t kbase, uint32_t vbase, uint32_t kscale,
                                             uint32_t vscale, int log2_box, int warp, int lane,
                                             int vlo, int valid, float scale_log2,
                                             uint32_t qfrag, uint32_t vst,
                                             float (&o)[D / 8][4], float (&m)[2],
                                             float (&l)[2]) {
  static_assert(D == 128, "one 128-byte code row per token");
  const int mi = lane >> 3, rr = lane & 7;
  const int c0 = 2 * (lane & 3);
  // Shared-memory loads are issued in groups ahead of their use (the asm
  // statements keep program order), so their latencies overlap.
  float ksr[2][2], vsr[2][2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int t = warp * 16 + nt * 8 + c0 + e;
      ksr[nt][e] = lds_f32(scale_addr(kscale, t, log2_box));
      vsr[nt][e] = lds_f32(scale_addr(vscale, t, log2_box));
    }
  {  // value codes -> fp16: lane converts 64 codes of row lane / 2
    const int row = lane >> 1, tok = warp * 16 + row;
    uint4 u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) u[i] = lds_v4(vbase + swz128(tok, (lane & 1) * 4 + i));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = (lane & 1) * 4 + i;  // 16 dims
      uint32_t w[8];
      i8x4_to_f16(u[i].x, w[0], w[1]);
      i8x4_to_f16(u[i].y, w[2], w[3]);
      i8x4_to_f16(u[i].z, w[4], w[5]);
      i8x4_to_f16(u[i].w, w[6], w[7]);
      const uint32_t half = vst + (c >> 2) * (16 * 128);
      sts_v4(half + swz128(row, (c & 3) * 2), w[0], w[1], w[2], w[3]);
      sts_v4(half + swz128(row, (c & 3) * 2 + 1), w[4], w[5], w[6], w[7]);
    }
    __syncwarp();
  }
  // Key operands: token lane/4 of each octet, codes at dims 16kk + 4c .. 4c+3.
  uint32_t kw[D / 16][2];
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int tk = warp * 16 + nt * 8 + (lane >> 2);
      asm volatile("ld.shared.u32 %0, [%1];"
                   : "=r"(kw[kk][nt])
                   : "r"(kbase + swz128(tk, kk) + 4 * (lane & 3)));
    }
  float s[2][4];
#pragma unroll
  for (int i = 0; i < 2; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) s[i][e] = 0.f;
  uint4 qn = lds_v4(qfrag + lane * 16);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t qa[4] = {qn.x, qn.y, qn.z, qn.w};
    if (kk + 1 < D / 16) qn = lds_v4(qfrag + ((kk + 1) * 32 + lane) * 16);
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      uint32_t b0, b1;
      i8x4_to_f16(kw[kk][nt], b0, b1);
      MmaOp<__half>::run(s[nt], qa, b0, b1);
    }
  }
  float vsc[2][2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int k = nt * 8 + c0 + e;
      const bool in = k >= vlo && k < valid;
      // Stale stage contents outside [vlo, valid) never enter arithmetic.
      const float ks = in ? ksr[nt][e] : 0.f;
      vsc[nt][e] = in ? vsr[nt][e] : 0.f;
      s[nt][e] = in ? s[nt][e] * (scale_log2 * ks) : -INFINITY;
      s[nt][e + 2] = in ? s[nt][e + 2] * (scale_log2 * ks) : -INFINITY;
    }
  float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
  float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
  const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
  const bool grew = mn0 != m[0] || mn1 != m[1];
  const float corr0 = fast_exp2(m[0] - mn0), corr1 = fast_exp2(m[1] - mn1);
  m[0] = mn0;
  m[1] = mn1;
  float p[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    p[nt][0] = fast_exp2(s[nt][0] - mn0);
    p[nt][1] = fast_exp2(s[nt][1] - mn0);
    p[nt][2] = fast_exp2(s[nt][2] - mn1);
    p[nt][3] = fast_exp2(s[nt][3] - mn1);
  }
  l[0] = l[0] * corr0 + (p[0][0] + p[0][1] + p[1][0] + p[1][1]);
  l[1] = l[1] * corr1 + (p[0][2] + p[0][3] + p[1][2] + p[1][3]);
  uint32_t pa[4];
  float ra, rb;
  pa[0] = Pack<__half>::run(p[0][0] * vsc[0][0], p[0][1] * vsc[0][1], ra, rb);
  pa[1] = Pack<__half>::run(p[0][2] * vsc[0][0], p[0][3] * vsc[0][1], ra, rb);
  pa[2] = Pack<__half>::run(p[1][0] * vsc[1][0], p[1][1] * vsc[1][1], ra, rb);
  pa[3] = Pack<__half>::run(p[1][2] * vsc[1][0], p[1][3] * vsc[1][1], ra, rb);
  if (__any_sync(0xffffffffu, grew)) {  // O keeps its scale while no row max grows
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      o[n][0] *= corr0;
      o[n][1] *= corr0;
      o[n][2] *= corr1;
      o[n][3] *= corr1;
    }
  }
  const int tok = (mi & 1) * 8 + rr;  // row of the warp's staging tile
  uint32_t vb[D / 16][4];
#pragma unroll
  for (int dp = 0; dp < D / 16; ++dp) {
    const int dcol = dp * 16 + (mi >> 1) * 8;
    ldsm_x4_t(vst + (dcol >> 6) * (16 * 128) + swz128(tok, (dcol & 63) >> 3), vb[dp][0],
              vb[dp][1], vb[dp][2], vb[dp][3]);
  }
  // Codes are finite, and the weights outside [vlo, valid) are exact zeros,
  // so no value row needs masking here.
#pragma unroll
  for (int dp = 0; dp < D / 16; ++dp) {
    MmaOp<__half>::run(o[2 * dp], pa, vb[dp][0], vb[dp][1]);
    MmaOp<__half>::run(o[2 * dp + 1], pa, vb[dp][2], vb[dp][3]);
  }
  __syncwarp();  // the staging tile is rewritten by the warp's next tile
}

// The end of one segment share (cold path, kept out of line to spare the
// main loop's registers): merge the four consumer warps' states held in
// shared memory, then write the output (whole segment) or publish a partial
// state; for a split segment the last-arriving CTA merges all partials.
// Each thread handles four consecutive head-dim elements of one query row.
template <typename T, int D>
__device__ __noinline__ void finish_share(const DecodeParams& p, const float* cmb_m,
                                          const float* cmb_l, float* cmb_o,
                                          volatile int* last_flag, volatile int* npieces,
                                          int* pieces, int ctid, int b, int g,
                                          bool complete, int c, int slot, long long seg0,
                                          int seg_tiles, long long N, int P) {
  constexpr int kQuads = D / 4;
  const int G = p.group;
  T* out = static_cast<T*>(p.out);
  const long long row0 = static_cast<long long>(b) * p.num_q_heads + g * G;
  for (int e4 = ctid; e4 < G * kQuads; e4 += kConsumerWarps * 32) {
    const int r = e4 / kQuads, d = (e4 - r * kQuads) * 4;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, cmb_m[w * G + r]);
    float Ls = 0.f;
    float4 Os = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float mw = cmb_m[w * G + r];
      const float f = mw == -INFINITY ? 0.f : fast_exp2(mw - M);
      Ls += f * cmb_l[w * G + r];
      const float4 v = *reinterpret_cast<const float4*>(&cmb_o[(w * G + r) * D + d]);
      Os.x += f * v.x; Os.y += f * v.y; Os.z += f * v.z; Os.w += f * v.w;
    }
    if (complete) {
      store4<T>(out + (row0 + r) * D + d, Os, Ls > 0.f ? 1.f / Ls : 0.f);
    } else {
      const long long ws_row = (static_cast<long long>(c) * 2 + slot) * G + r;
      *reinterpret_cast<float4*>(&p.ws_o[ws_row * D + d]) = Os;
      if (d == 0) *reinterpret_cast<float2*>(&p.ws_ml[ws_row * 2]) = make_float2(M, Ls);
    }
  }
  if (complete) return;

  // Split segment: count arrivals with one acq_rel atomic per CTA (after a CTA
  // barrier, so it releases every thread's partial writes); the CTA that
  // arrives last merges all shares in ascending CTA order and resets the
  // counter -- no second kernel and no waiting.
  named_bar_sync(1, kConsumerWarps * 32);
  const int cfirst = cta_of(seg0, N, P), clast = cta_of(seg0 + seg_tiles - 1, N, P);
  const int slot0 = tile_begin(cfirst, N, P) == seg0 ? 0 : 1;
  if (ctid == 0) {
    // Workspace rows (cta * 2 + slot) of every non-empty share, in CTA order.
    int n = 0;
    long long tb = tile_begin(cfirst, N, P);
    for (int cc = cfirst; cc <= clast; ++cc) {
      const long long te = tile_begin(cc + 1, N, P);
      if (tb < te) {
        if (n < kMaxPieces) pieces[n] = cc * 2 + (cc == cfirst ? slot0 : 0);
        ++n;
      }
      tb = te;
    }
    *npieces = n;
    *last_flag = atomic_add_acq_rel(&p.ws_cnt[cfirst * 2 + slot0], 1) == n - 1 ? 1 : 0;
  }
  named_bar_sync(1, kConsumerWarps * 32);
  if (!*last_flag) return;
  const int n = *npieces;
  if (n <= kMaxPieces) {
    // (m, l) of every share and row, loaded in parallel into the (now free)
    // combine buffer, then one float4 of each share per thread.
    float2* ml = reinterpret_cast<float2*>(cmb_o);
    for (int i = ctid; i < n * G; i += kConsumerWarps * 32)
      ml[i] = __ldcg(reinterpret_cast<const float2*>(
          &p.ws_ml[(static_cast<long long>(pieces[i / G]) * G + i % G) * 2]));
    named_bar_sync(1, kConsumerWarps * 32);
    for (int e4 = ctid; e4 < G * kQuads; e4 += kConsumerWarps * 32) {
      const int r = e4 / kQuads, d = (e4 - r * kQuads) * 4;
      float M = -INFINITY;
      for (int i = 0; i < n; ++i) M = fmaxf(M, ml[i * G + r].x);
      float Ls = 0.f;
      float4 Os = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
      for (int i = 0; i < n; ++i) {
        const float f = fast_exp2(ml[i * G + r].x - M);
        Ls += f * ml[i * G + r].y;
        const float4 v = __ldcg(reinterpret_cast<const float4*>(
            &p.ws_o[(static_cast<long long>(pieces[i]) * G + r) * D + d]));
        Os.x += f * v.x; Os.y += f * v.y; Os.z += f * v.z; Os.w += f * v.w;
      }
      store4<T>(out + (row0 + r) * D + d, Os, Ls > 0.f ? 1.f / Ls : 0.f);
    }
  } else {
    // Very many CTAs per segment (num_ctas far above the tile count).
    for (int e = ctid; e < G * D; e += kConsumerWarps * 32) {
      const int r = e / D, d = e - r * D;
      float M = -INFINITY, Ls = 0.f, Os = 0.f;
      for (int cc = cfirst; cc <= clast; ++cc) {
        if (tile_begin(cc, N, P) == tile_begin(cc + 1, N, P)) continue;
        const long long row = (static_cast<long long>(cc) * 2 + (cc == cfirst ? slot0 : 0)) * G + r;
        M = fmaxf(M, __ldcg(&p.ws_ml[row * 2]));
      }
      for (int cc = cfirst; cc <= clast; ++cc) {
        if (tile_begin(cc, N, P) == tile_begin(cc + 1, N, P)) continue;
        const long long row = (static_cast<long long>(cc) * 2 + (cc == cfirst ? slot0 : 0)) * G + r;
        const float f = fast_exp2(__ldcg(&p.ws_ml[row * 2]) - M);
        Ls += f * __ldcg(&p.ws_ml[row * 2 + 1]);
        Os += f * __ldcg(&p.ws_o[row * D + d]);
      }
      out[(row0 + r) * D + d] = Pack<T>::cvt(Ls > 0.f ? Os / Ls : 0.f);
    }
  }
  if (ctid == 0) p.ws_cnt[cfirst * 2 + slot0] = 0;
}

// tm_ks / tm_vs: the INT8 cache's K and V scales (unused for a 16-bit cache).
template <typename T, int D, bool kI8>
__global__ void __launch_bounds__(kThreads, 2)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_ks,
                        const __grid_constant__ CUtensorMap tm_vs,
                        const __grid_constant__ DecodeParams p) {
  constexpr int kHalves = Layout<D, kI8>::kHalves;
  constexpr int kKBytes = Layout<D, kI8>::kKBytes;
  constexpr int kStages = Layout<D, kI8>::kStages;
  const Layout<D, kI8> L(p.batch, p.group);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L.bar);
  uint64_t* empty = full + kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.flags);
  volatile int* last_flag = abort_flag + 1;
  int* lens = reinterpret_cast<int*>(smem + L.lens);
  int* cum = reinterpret_cast<int*>(smem + L.cum);
  float* cmb_m = reinterpret_cast<float*>(smem + L.cmb);
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
    prefetch_tmap(&tm_q);
    if constexpr (kI8) {
      prefetch_tmap(&tm_ks);
      prefetch_tmap(&tm_vs);
    }
  }
  // Plan: clamped lengths and the prefix sum of 64-token tiles per sequence.
  for (int i = tid; i < B; i += kThreads) lens[i] = clamp_len(p.seq_lens[i], cap, p.err_flag);
  __syncthreads();
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < B; base += 32) {
      const int i = base + lane;
      const int n = i < B ? (lens[i] + kTile - 1) / kTile - first_tile(lens[i], p.window) : 0;
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
  // Sequences with no cached token get a row of zeros (CTA b % P writes them)
  // and, when appending, no slot (-1): there is no new token to write.
  {
    T* out = static_cast<T*>(p.out);
    const int row_elems = p.num_q_heads * D;
    for (int b = c; b < B; b += P)
      if (lens[b] == 0) {
        for (int e = tid; e < row_elems; e += kThreads)
          out[static_cast<long long>(b) * row_elems + e] = Pack<T>::cvt(0.f);
        if (tid == 0 && p.slot_out) p.slot_out[b] = -1;
      }
  }
  const long long t_begin = tile_begin(c, N, P), t_end = tile_begin(c + 1, N, P);
  if (t_begin >= t_end) return;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    Cursor cur;
    cur.locate(t_begin, cum, B, hkv);
    const int nsub = kTile / p.box_tokens;
    // Bytes of one box: a 64-element half of box_tokens 16-bit rows, or
    // box_tokens whole 128-byte code rows.
    const uint32_t box_bytes = static_cast<uint32_t>(p.box_tokens) * 128u;
    const uint32_t q_bytes = static_cast<uint32_t>(G) * 128u * kHalves;
    int it = 0;
    for (long long t = t_begin; t < t_end; ++t, ++it) {
      const int stage = it % kStages;
      const uint32_t phase = (it / kStages) & 1;
      // Look up this tile's physical blocks first: the table load's latency
      // overlaps the wait for a free stage.
      const int Lb = lens[cur.b];
      const int tok = (first_tile(Lb, p.window) + cur.j) * kTile + lane * p.box_tokens;
      // A box wholly below the band is not fetched (its rows are masked).
      const bool wanted = lane < nsub && tok < Lb && tok + p.box_tokens > band_lo(Lb, p.window);
      int pb = -1;
      if (wanted)
        pb = __ldg(&p.block_table[static_cast<long long>(cur.b) * p.max_blocks +
                                  (tok >> p.log2_bs)]);
      if (!kI8 && p.new_k != nullptr && cur.j == cur.n - 1) {
        // The last tile of segment (b, g) holds the new token: write its K/V
        // rows for head g (16 bytes per lane), make the writes visible to the
        // TMA unit, then load the tile as usual.  No other CTA reads them.
        const int pos = Lb - 1;
        const int pbn = __ldg(&p.block_table[static_cast<long long>(cur.b) * p.max_blocks +
                                             (pos >> p.log2_bs)]);
        constexpr int kChunks = D * 2 / 16;  // 16-byte pieces of one row
        if (pbn >= 0 && pbn < p.num_blocks) {
          if (lane < 2 * kChunks) {
            const bool is_v = lane >= kChunks;
            const int q16 = lane - (is_v ? kChunks : 0);
            const long long src_row = static_cast<long long>(cur.b) * p.num_kv_heads + cur.g;
            const long long dst_row =
                (static_cast<long long>(pbn) * p.block_size + (pos & (p.block_size - 1))) *
                    p.num_kv_heads + cur.g;
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(
                                      static_cast<const T*>(is_v ? p.new_v : p.new_k) + src_row * D) +
                                  q16);
            *(reinterpret_cast<uint4*>(static_cast<T*>(is_v ? p.v_cache : p.k_cache) + dst_row * D) +
              q16) = v;
            asm volatile("fence.proxy.async.global;" ::: "memory");
          }
          if (lane == 0 && cur.g == 0 && p.slot_out)
            p.slot_out[cur.b] = pbn * p.block_size + (pos & (p.block_size - 1));
        } else if (lane == 0) {
          set_flag(p.err_flag, KVC_FLAG_BLOCK_ID_RANGE);
          if (cur.g == 0 && p.slot_out) p.slot_out[cur.b] = -1;
        }
        __syncwarp();
        if (lane == 0) asm volatile("fence.proxy.async.global;" ::: "memory");
      }
      bool ok = !*abort_flag && mbar_wait_bounded(&empty[stage], phase ^ 1, p.err_flag);
      if (!ok) {
        *abort_flag = 1;
      } else {
        bool valid = false;
        if (wanted) {
          if (pb < 0 || pb >= p.num_blocks) set_flag(p.err_flag, KVC_FLAG_BLOCK_ID_RANGE);
          else valid = true;
        }
        const uint32_t nvalid = __popc(__ballot_sync(0xffffffffu, valid));
        uint8_t* st = smem + stage * L.stage;
        if (lane == 0) {
          const uint32_t per_box =
              kI8 ? box_bytes * 2 + static_cast<uint32_t>(p.box_tokens) * 8u
                  : box_bytes * kHalves * 2;
          mbar_arrive_expect_tx(&full[stage], nvalid * per_box + q_bytes);
#pragma unroll
          for (int h = 0; h < kHalves; ++h)
            tma_load_3d(st + L.qoff + h * L.q_half, &tm_q, &full[stage], h * 64, cur.g * G,
                        cur.b);
        }
        __syncwarp();
        if (valid) {
          uint8_t* kdst = st + lane * box_bytes;
          const int in_blk = tok & (p.block_size - 1);
          if constexpr (kI8) {
            tma_load_4d(kdst, &tm_k, &full[stage], 0, cur.g, in_blk, pb);
            tma_load_4d(kdst + kKBytes, &tm_v, &full[stage], 0, cur.g, in_blk, pb);
            uint8_t* sdst = st + L.scales + lane * 128;
            tma_load_3d(sdst, &tm_ks, &full[stage], in_blk, cur.g, pb);
            tma_load_3d(sdst + kScaleBytes, &tm_vs, &full[stage], in_blk, cur.g, pb);
          } else {
#pragma unroll
            for (int h = 0; h < kHalves; ++h) {
              tma_load_4d(kdst + h * kHalfBytes, &tm_k, &full[stage], h * 64, cur.g, in_blk, pb);
              tma_load_4d(kdst + kKBytes + h * kHalfBytes, &tm_v, &full[stage], h * 64, cur.g,
                          in_blk, pb);
            }
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
  Cursor cur;
  cur.locate(t_begin, cum, B, hkv);
  const int ctid = warp * 32 + lane;
  float o[D / 8][4], m[2], l[2];
  auto reset = [&]() {
#pragma unroll
    for (int n = 0; n < D / 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[n][e] = 0.f;
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
  };
  reset();
  bool need_q = true;  // INT8: the segment's query fragments are still to be built
  int seg_first_j = cur.j;
  int slot = 0;  // 0 for the first segment this CTA touches, 1 afterwards
  const uint32_t sbase = smem_u32(smem);
  int it = 0;
  for (long long t = t_begin; t < t_end; ++t, ++it) {
    const int stage = it % kStages;
    const uint32_t phase = (it / kStages) & 1;
    bool ok = !*abort_flag && mbar_wait_bounded(&full[stage], phase, p.err_flag);
    if (!ok) *abort_flag = 1;
    if constexpr (kI8) {
      // Every consumer warp reaches this point at the same tile (need_q is
      // set at the same segment boundaries for all of them), whether or not
      // its tokens are attended, so the barrier always completes; after a
      // failed wait the stage's query rows are stale but still in bounds.
      if (need_q) {
        build_q_i8<T, D>(sbase + stage * L.stage + L.qoff, L.q_half, G, warp, lane,
                         sbase + L.qfrag);
        named_bar_sync(2, kConsumerWarps * 32);
        need_q = false;
      }
    }
    const int Lc = lens[cur.b];
    const int row0 = (first_tile(Lc, p.window) + cur.j) * kTile + warp * 16;
    const int valid = min(16, Lc - row0);                     // rows [vlo, valid) of the
    const int vlo = max(0, band_lo(Lc, p.window) - row0);     // warp's 16 are attended
    if (ok && valid > vlo) {
      const uint32_t kb = sbase + stage * L.stage;
      if constexpr (kI8)
        attend_16_i8<D>(kb, kb + kKBytes, kb + L.scales, kb + L.scales + kScaleBytes,
                        p.log2_box, warp, lane, vlo, valid, p.scale_log2, sbase + L.qfrag,
                        sbase + L.vstg + warp * 16 * D * 2, o, m, l);
      else
        attend_16<T, D>(kb, kb + kKBytes, warp, lane, vlo, valid, p.scale_log2, kb + L.qoff,
                        L.q_half, G, o, m, l);
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
      finish_share<T, D>(p, cmb_m, cmb_l, cmb_o, last_flag, abort_flag + 2,
                         reinterpret_cast<int*>(smem + L.pieces), ctid, cur.b, cur.g,
                         complete, c, slot,
                         static_cast<long long>(hkv) * cum[cur.b] +
                             static_cast<long long>(cur.g) * cur.n,
                         cur.n, N, P);
      named_bar_sync(1, kConsumerWarps * 32);
      slot = 1;
      cur.advance(cum, B, hkv);
      reset();
      need_q = true;
      seg_first_j = cur.j;
    } else {
      cur.advance(cum, B, hkv);
    }
  }
}

template <typename T, int D, bool kI8>
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
    cudaFuncSetAttribute(paged_decode_kernel<T, D, kI8>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                         Layout<D, kI8>(kMaxBatch, 16).total);
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, paged_decode_kernel<T, D, kI8>,
                                                      kThreads, smem) != cudaSuccess ||
        occ < 1)
      occ = 1;
    cache[{dev, smem}] = occ;
    return occ;
  }
};

template <typename T, int D, bool kI8>
kvc_status run_decode(const DecodeArgs& a) {
  const int G = a.num_q_heads / a.num_kv_heads;
  const size_t smem = Layout<D, kI8>(a.batch, G).total;
  const int occ = DecodeKernel<T, D, kI8>::occupancy(smem);  // also sets the smem limit
  const int P = a.num_ctas > 0 ? a.num_ctas : device_sm_count() * occ;
  if (a.workspace_bytes < paged_decode_workspace_bytes(G, D, P) || a.workspace == nullptr)
    return KVC_ERR_WORKSPACE;

  const int box_tokens = a.block_size < kTile ? a.block_size : kTile;
  const uint64_t elt = kI8 ? 1 : 2;
  const uint64_t dims[4] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.num_kv_heads),
                            static_cast<uint64_t>(a.block_size),
                            static_cast<uint64_t>(a.num_blocks)};
  const uint64_t strides[3] = {static_cast<uint64_t>(D) * elt,
                               static_cast<uint64_t>(a.num_kv_heads) * D * elt,
                               static_cast<uint64_t>(a.block_size) * a.num_kv_heads * D * elt};
  // 16-bit cache: boxes of one 64-element (128-byte) half of box_tokens rows;
  // INT8 cache: boxes of box_tokens whole 128-byte code rows.
  const uint32_t box[4] = {kI8 ? static_cast<uint32_t>(D) : 64u, 1,
                           static_cast<uint32_t>(box_tokens), 1};
  const CUtensorMapDataType cache_type =
      kI8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
          : (a.dtype == KVC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16);
  CUtensorMap tk, tv, tks, tvs;
  if (!encode_tmap(&tk, cache_type, 4, a.key_cache, dims, strides, box, true) ||
      !encode_tmap(&tv, cache_type, 4, a.value_cache, dims, strides, box, true))
    return KVC_ERR_CUDA;
  if constexpr (kI8) {
    // Scales [num_blocks, Hkv, block_size] fp32: a box = one head's scales of
    // the box_tokens tokens of one block.
    const uint64_t sdims[3] = {static_cast<uint64_t>(a.block_size),
                               static_cast<uint64_t>(a.num_kv_heads),
                               static_cast<uint64_t>(a.num_blocks)};
    const uint64_t sstrides[2] = {static_cast<uint64_t>(a.block_size) * 4,
                                  static_cast<uint64_t>(a.num_kv_heads) * a.block_size * 4};
    const uint32_t sbox[3] = {static_cast<uint32_t>(box_tokens), 1, 1};
    if (!encode_tmap(&tks, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.key_scales, sdims, sstrides,
                     sbox, false) ||
        !encode_tmap(&tvs, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.value_scales, sdims, sstrides,
                     sbox, false))
      return KVC_ERR_CUDA;
  } else {
    tks = tk;  // not read
    tvs = tv;
  }
  // Query [B, Hq, D]: one box = the G rows of a query group, 64 elements wide.
  CUtensorMap tq;
  const uint64_t qdims[3] = {static_cast<uint64_t>(D), static_cast<uint64_t>(a.num_q_heads),
                             static_cast<uint64_t>(a.batch)};
  const uint64_t qstrides[2] = {static_cast<uint64_t>(D) * 2,
                                static_cast<uint64_t>(a.num_q_heads) * D * 2};
  const uint32_t qbox[3] = {64, static_cast<uint32_t>(G), 1};
  if (!encode_tmap_16bit(&tq, a.dtype, 3, a.q, qdims, qstrides, qbox, true)) return KVC_ERR_CUDA;

  DecodeParams p;
  p.q = a.q;
  p.out = a.out;
  p.block_table = a.block_table;
  p.seq_lens = a.seq_lens;
  p.ws_cnt = static_cast<int*>(a.workspace);
  p.ws_o = reinterpret_cast<float*>(static_cast<char*>(a.workspace) + counter_bytes(P));
  p.ws_ml = p.ws_o + static_cast<size_t>(P) * 2 * G * D;
  p.err_flag = a.err_flag;
  p.new_k = a.new_key;
  p.new_v = a.new_value;
  p.k_cache = const_cast<void*>(a.key_cache);
  p.v_cache = const_cast<void*>(a.value_cache);
  p.slot_out = a.slot_out;
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
  p.log2_box = ilog2(box_tokens);
  p.window = a.window;
  p.scale_log2 = a.scale * 1.4426950408889634f;

  paged_decode_kernel<T, D, kI8><<<P, kThreads, smem, a.stream>>>(tk, tv, tq, tks, tvs, p);
  return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

template <bool kI8>
int num_ctas_for(int group, int head_dim, kvc_dtype dtype) {
  const int sms = device_sm_count();
  if (sms <= 0) return 0;
  // The smallest batch needs the least shared memory, hence the most CTAs.
  if (head_dim == 64 && !kI8) {
    const size_t smem = Layout<64, false>(1, group).total;
    return sms * (dtype == KVC_BF16 ? DecodeKernel<__nv_bfloat16, 64, false>::occupancy(smem)
                                    : DecodeKernel<__half, 64, false>::occupancy(smem));
  }
  if (head_dim == 128) {
    const size_t smem = Layout<128, kI8>(1, group).total;
    return sms * (dtype == KVC_BF16 ? DecodeKernel<__nv_bfloat16, 128, kI8>::occupancy(smem)
                                    : DecodeKernel<__half, 128, kI8>::occupancy(smem));
  }
  return 0;
}

}  // namespace

size_t paged_decode_workspace_bytes(int group, int head_dim, int ctas) {
  return counter_bytes(ctas) + static_cast<size_t>(ctas) * 2 * group * (head_dim + 2) * sizeof(float);
}

int paged_decode_num_ctas(int group, int head_dim, kvc_dtype dtype, int num_ctas, bool int8) {
  if (num_ctas > 0) return num_ctas;
  return int8 ? num_ctas_for<true>(group, head_dim, dtype)
              : num_ctas_for<false>(group, head_dim, dtype);
}

kvc_status launch_paged_decode(const DecodeArgs& a) {
  if (a.key_scales != nullptr) {  // INT8 cache (head_dim 128, plain decode)
    if (a.head_dim != 128 || a.new_key != nullptr) return KVC_ERR_UNSUPPORTED;
    return a.dtype == KVC_BF16 ? run_decode<__nv_bfloat16, 128, true>(a)
                               : run_decode<__half, 128, true>(a);
  }
  if (a.head_dim == 64)
    return a.dtype == KVC_BF16 ? run_decode<__nv_bfloat16, 64, false>(a)
                               : run_decode<__half, 64, false>(a);
  if (a.head_dim == 128)
    return a.dtype == KVC_BF16 ? run_decode<__nv_bfloat16, 128, false>(a)
                               : run_decode<__half, 128, false>(a);
  return KVC_ERR_UNSUPPORTED;
}

}  // namespace kvc
