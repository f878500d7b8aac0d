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
//  * Work unit = a 64-token tile (INT8: 128) of one (sequence b, kv head g) segment.
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
//  * Over an INT8 cache (codes + one fp32 scale per row) the same kernel
//    runs with 128-token tiles of codes and scales, each consumer warp taking
//    two 16-token sub-tiles under one softmax update, and the products
//    transposed (S^T = K Q^T, O^T = V^T P^T: the tokens are the M side, the
//    query group the N side), the codes widened to fp16 exactly in registers.
#include <cuda_runtime.h>

#include <math.h>

#include <map>
#include <mutex>
#include <utility>

#include "kvc_device.cuh"
#include "kvc_host.h"

namespace kvc {

namespace {

constexpr int kTile = 64;            // tokens per pipeline stage over a 16-bit cache
constexpr int kConsumerWarps = 4;    // 16 tokens each
constexpr int kThreads = (kConsumerWarps + 1) * 32;
// Over an INT8 cache each consumer warp takes kI8Sub 16-token sub-tiles of a
// stage under one online-softmax update: with 2, a stage holds 128 tokens
// (the bytes of a 64-token stage of a 16-bit cache) and the per-tile work of
// a warp (waits, cursor, masks, the softmax update) is paid per 32 tokens.
constexpr int kI8Sub = 2;
template <bool kI8>
constexpr int tile_of() { return kI8 ? 64 * kI8Sub : kTile; }
// Pipeline depth: 3 stages of ~33 KB over a 16-bit cache; over an INT8 cache
// 2 stages of ~38 KB (128-token tiles, two CTAs per SM) or 3 of ~20 KB
// (64-token tiles, three CTAs per SM).
template <bool kI8>
constexpr int stages_of() { return kI8 && kI8Sub == 2 ? 2 : 3; }
// Resident CTAs per SM the kernel is compiled for (register budget).
template <int kQ>
constexpr int min_ctas_of() { return kQ == 1 && kI8Sub == 1 ? 3 : 2; }
constexpr int kMaxBatch = 1024;
// Work split: each (sequence, kv head) segment counts seg_units_of<kI8>()
// units of work beyond its tiles, for its end-of-segment finish (combine,
// partial state, arrival, merge), so that CTAs whose shares end more
// segments get fewer tiles.  The units are virtual: no role visits them.
// Measured: over an INT8 cache, whose 128-token tiles carry the same finish
// cost per segment as 64-token 16-bit ones, 1 unit is 5 % faster than none
// (2 is between); over a 16-bit cache 3 units gained 0.2-0.5 % on the GQA
// 8B shape but cost 2.5 % on the MHA shape's many short segments, so none.
constexpr int kSegUnits16 = 0;  // 16-bit cache
constexpr int kSegUnitsI8 = 1;  // INT8 cache
template <bool kI8>
constexpr int seg_units_of() { return kI8 ? kSegUnitsI8 : kSegUnits16; }
constexpr int kHalfBytes = kTile * 128;  // one 64-element half of a K or V tile
constexpr int kMaxPieces = 62;           // split shares merged from a shared-memory list
// INT8 cache: a tile's per-token scales arrive as one TMA box per box of
// codes (min(block_size, 64) floats); each box gets its own slot of
// max(128, 4 * box) bytes, so every TMA destination is 128-byte aligned.
constexpr int kScaleBytes = (tile_of<true>() / 8) * 128;

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
  // Over an INT8 cache the new rows are quantised (quantize_row_int8) into
  // the code arrays k_cache / v_cache and their scales into k_scales /
  // v_scales [num_blocks, Hkv, block_size].
  const void* new_k;
  const void* new_v;
  void* k_cache;
  void* v_cache;
  float* k_scales;
  float* v_scales;
  int32_t* slot_out;
  int batch, num_q_heads, num_kv_heads, group, head_dim;
  int block_size, log2_bs, max_blocks, num_blocks, box_tokens, log2_box;
  int log2_sslot;  // INT8: log2 of a scale box's slot in the stage (>= 7)
  int window;  // band of the last `window` cached tokens (0: the whole sequence)
  float scale_log2;
};

__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

// Dynamic shared memory of the decode kernel.  A stage holds the K tile, the
// V tile and the query rows of the tile's (b, g) (all 128-byte swizzled, each
// 1024-byte aligned as the TMA swizzle requires); every other region starts
// on a 16-byte boundary.  Over an INT8 cache (kI8) the K and V tiles hold the
// int8 codes (one 128-byte row per token) and the stage also holds the tile's
// per-token K and V scales.
template <int D, bool kI8>
struct Layout {
  static constexpr int kHalves = D / 64;  // 64-element halves of a 16-bit row
  static constexpr int kKBytes = kI8 ? tile_of<true>() * D : kHalves * kHalfBytes;  // K or V tile
  int q_half;   // bytes of one 64-wide half of the G query rows (1024-aligned)
  int scales;   // INT8: K scales then V scales of the stage, kScaleBytes each
  int qoff;     // query rows of the stage (1024-aligned)
  int stage;    // K tile, V tile, (scales), query rows
  static constexpr int kStages = stages_of<kI8>();
  int bar;      // full[kStages], empty[kStages]
  int flags;    // abort, last, npieces
  int pieces;   // int[kMaxPieces]
  int lens;     // int[batch]
  int cum;      // int[batch + 1]: tiles per kv head before each sequence
  int ucum;     // int[batch + 1]: work units (tiles + seg_units_of) per kv head before it
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
    ucum = align_up(cum + (batch + 1) * 4, 16);
    cmb = align_up(ucum + (batch + 1) * 4, 16);
    total = 1024 + cmb + kConsumerWarps * group * (D + 2) * 4;
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
  // The first tile at or after work unit t (units: ucum, seg_units virtual
  // units before each segment's tiles; tiles: cum).
  __device__ __forceinline__ void locate(long long t, const int* cum, const int* ucum, int batch,
                                         int hkv, int seg_units) {
    int lo = 0, hi = batch - 1;  // largest b with hkv*ucum[b] <= t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (static_cast<long long>(hkv) * ucum[mid] <= t) lo = mid; else hi = mid - 1;
    }
    b = lo;
    n = cum[b + 1] - cum[b];
    const long long r = t - static_cast<long long>(hkv) * ucum[b];
    g = static_cast<int>(r / (n + seg_units));
    const int jj = static_cast<int>(r - static_cast<long long>(g) * (n + seg_units)) - seg_units;
    j = jj > 0 ? jj : 0;
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
// tiles start at the kT-token tile holding band_lo.
__device__ __forceinline__ int band_lo(int L, int window) {
  return window > 0 && L > window ? L - window : 0;
}
template <int kT>
__device__ __forceinline__ int first_tile(int L, int window) { return band_lo(L, window) / kT; }

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

// Over an INT8 cache the products run transposed, S^T = K Q^T and
// O^T = V^T P^T (mma m16n8k16, fp16 operands, fp32 accumulation): the warp's
// 16 tokens are the M side of the score product and the K side of the value
// product, and the query group is the N side, NT tiles of 8 query rows (rows
// >= G are zero queries whose results are dropped).  For G <= 8 this is half
// the tensor ops and half the accumulator registers of padding the group to
// 16 rows.
//
// Score product, k-step kk (dims 16kk .. 16kk+15, permuted): lane (g =
// lane/4, c = lane%4) holds dims 16kk + 4c .. 4c+3 of tokens g and g+8 (one
// 32-bit word of codes each) and of query row g of each tile, in the slots
// of k = 2c, 2c+1, 2c+8, 2c+9; a dot product does not depend on the order of
// its terms.  Value product, dims 16ch .. 16ch+15 (m-tile ch of O^T): lane
// (g, c) holds the codes of tokens 2c, 2c+1 (and 2c+8, 2c+9) at dims
// 16ch + 2g and 2g+1, and the m-tile's output rows are permuted to match:
// row g is dim 16ch + 2g, row g+8 dim 16ch + 2g + 1.

// The segment's query fragments (B of the score product) from the stage's
// query rows, as fp16: qb[kk][nt] = dims 16kk + 4c .. 4c+3 of row 8nt + g.
template <typename T, int D, int NT>
__device__ __forceinline__ void load_q_i8(uint32_t qbase, int q_half, int group, int lane,
                                          uint32_t (&qb)[D / 16][NT][2]) {
  const int g = lane >> 2, c = lane & 3;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int r = nt * 8 + g;
      uint32_t w0 = 0, w1 = 0;
      if (r < group)
        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                     : "=r"(w0), "=r"(w1)
                     : "r"(qbase + (kk >> 2) * q_half + swz128(r, (kk & 3) * 2 + (c >> 1)) +
                           (c & 1) * 8));
      qb[kk][nt][0] = q_pair_f16<T>(w0);
      qb[kk][nt][1] = q_pair_f16<T>(w1);
    }
}

// Per-lane shared-memory offsets of the INT8 consumer, the same for every
// tile (relative to a stage's K or V tile and scale region).  A consumer
// warp takes kI8Sub 16-token sub-tiles of a stage (2048 bytes apart).  With the 128-byte swizzle a row r's chunk x sits at
// r * 128 + ((x ^ (r % 8)) << 4), and the sub-tiles start at multiples of 8
// rows.  Codes are read with ldmatrix (8 rows of 16 bytes per matrix):
// without .trans lane (g, c) receives bytes 4c .. 4c+3 of row g, with .trans
// (16-bit elements) bytes 2g, 2g+1 of rows 2c and 2c+1.
struct I8Lane {
  // ldmatrix.x4 row addresses: lane L gives row (L / 8 % 2) * 8 + L % 8 of
  // a 16-token sub-tile in chunk x + L / 16, at row_ofs + ((x << 4) ^ xr) for
  // an even chunk x.
  uint32_t row_ofs;
  uint32_t xr;
  uint32_t sc[2 * kI8Sub];  // scales of the warp's tokens g, g+8, (g+16, g+24) (one slot of
                     // 2^log2_slot bytes per TMA box of 2^log2_box tokens)
  __device__ __forceinline__ I8Lane(int warp, int lane, int log2_box, int log2_slot) {
    const int g = lane >> 2;
    const int t0 = warp * 16 * kI8Sub + g;
    const int r = lane & 7;
    row_ofs = static_cast<uint32_t>((warp * 16 * kI8Sub + ((lane >> 3) & 1) * 8 + r) * 128);
    xr = static_cast<uint32_t>(((lane >> 4) ^ r) << 4);
    const int box = 1 << log2_box;
#pragma unroll
    for (int i = 0; i < 2 * kI8Sub; ++i) {
      const int t = t0 + 8 * i;
      sc[i] = static_cast<uint32_t>(((t >> log2_box) << log2_slot) + ((t & (box - 1)) << 2));
    }
  }
};

// One warp's 16 kI8Sub tokens of a stage over an INT8 cache: kI8Sub
// sub-tiles of 16 sharing one online-softmax update.  A cached row is code * scale, so
// q . k = scale_k * (q . codes_k) and sum_j p_j v_j = sum_j (p_j * scale_v_j)
// codes_v_j.  The codes are exact in fp16, the queries are (load_q_i8), and
// the weights p * scale_v keep 11 bits (l sums the plain p, so the weights
// are not renormalised after rounding).  State per lane: m, l and O for
// query rows 8nt + 2c and 8nt + 2c + 1; l is this lane's share (tokens g and
// g+8 of each sub-tile), summed over the 8 lanes of a query at the end of
// the segment.  Rows [vlo, valid) of the warp's 16 kI8Sub are attended.
template <int D, int NT>
__device__ __forceinline__ void attend_i8(uint32_t kbase, uint32_t vbase, uint32_t kscale,
                                          uint32_t vscale, const I8Lane& ofs, int lane, int vlo,
                                          int valid, float scale_log2,
                                          const uint32_t (&qb)[D / 16][NT][2],
                                          float (&o)[NT][D / 16][4], float (&m)[NT][2],
                                          float (&l)[NT][2]) {
  static_assert(D == 128, "one 128-byte code row per token");
  const int g = lane >> 2, c = lane & 3;
  // All shared-memory loads first (the asm statements keep program order),
  // so their latencies overlap.  Row +8 is +1024 bytes with the same
  // swizzle; row 2c+1 is row 2c + 128 bytes with chunk bit 0 flipped.
  float ks[2 * kI8Sub], vs[2 * kI8Sub];
#pragma unroll
  for (int i = 0; i < 2 * kI8Sub; ++i) ks[i] = lds_f32(kscale + ofs.sc[i]);
#pragma unroll
  for (int i = 0; i < 2 * kI8Sub; ++i) vs[i] = lds_f32(vscale + ofs.sc[i]);
  // K: one ldmatrix.x4 per two k-steps gives a lane its codes at dims
  // 16kk + 4c .. 4c+3 of tokens g and g+8 for kk and kk+1.  V: one
  // ldmatrix.x4.trans per two 16-dim chunks gives a lane, per chunk, the codes
  // of tokens 2c, 2c+1 (and 2c+8, 2c+9) at dims 16 ch + 2g, 2g+1.
  // With two query tiles (NT = 2) the V loads wait until the scores are done,
  // to keep the live registers within the two-CTAs-per-SM budget.
  uint32_t kw[kI8Sub][D / 16][2], vw[kI8Sub][D / 16][2];
  auto load_v = [&]() {
#pragma unroll
    for (int sub = 0; sub < kI8Sub; ++sub)
#pragma unroll
      for (int ch = 0; ch < D / 16; ch += 2)
        ldsm_x4_t(vbase + ofs.row_ofs + sub * 2048 + ((ch << 4) ^ ofs.xr), vw[sub][ch][0],
                  vw[sub][ch][1], vw[sub][ch + 1][0], vw[sub][ch + 1][1]);
  };
#pragma unroll
  for (int sub = 0; sub < kI8Sub; ++sub)
#pragma unroll
    for (int kk = 0; kk < D / 16; kk += 2)
      ldsm_x4(kbase + ofs.row_ofs + sub * 2048 + ((kk << 4) ^ ofs.xr), kw[sub][kk][0],
              kw[sub][kk][1], kw[sub][kk + 1][0], kw[sub][kk + 1][1]);
  if constexpr (NT == 1) load_v();
  float s[kI8Sub][NT][4];
#pragma unroll
  for (int sub = 0; sub < kI8Sub; ++sub)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[sub][nt][e] = 0.f;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk)
#pragma unroll
    for (int sub = 0; sub < kI8Sub; ++sub) {
      uint32_t a[4];
      i8x4_to_f16(kw[sub][kk][0], a[0], a[2]);
      i8x4_to_f16(kw[sub][kk][1], a[1], a[3]);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        MmaOp<__half>::run(s[sub][nt], a, qb[kk][nt][0], qb[kk][nt][1]);
    }
  if constexpr (NT != 1) load_v();
  // s[sub][nt][0, 1]: token 16 sub + g, queries 2c, 2c+1; [2, 3]: token 16 sub
  // + g + 8.  Stale stage contents outside [vlo, valid) never enter arithmetic.
  bool in[2 * kI8Sub];
  float f[2 * kI8Sub], w[2 * kI8Sub];
#pragma unroll
  for (int i = 0; i < 2 * kI8Sub; ++i) {  // token 8 i + g of the warp's
    in[i] = 8 * i + g >= vlo && 8 * i + g < valid;
    f[i] = in[i] ? scale_log2 * ks[i] : 0.f;
    w[i] = in[i] ? vs[i] : 0.f;
  }
  bool grew = false;
  float corr[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int sub = 0; sub < kI8Sub; ++sub) {
      const int i0 = 2 * sub, i1 = 2 * sub + 1;
      s[sub][nt][0] = in[i0] ? s[sub][nt][0] * f[i0] : -INFINITY;
      s[sub][nt][1] = in[i0] ? s[sub][nt][1] * f[i0] : -INFINITY;
      s[sub][nt][2] = in[i1] ? s[sub][nt][2] * f[i1] : -INFINITY;
      s[sub][nt][3] = in[i1] ? s[sub][nt][3] * f[i1] : -INFINITY;
    }
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float mx = fmaxf(s[0][nt][e], s[0][nt][e + 2]);
#pragma unroll
      for (int sub = 1; sub < kI8Sub; ++sub)
        mx = fmaxf(mx, fmaxf(s[sub][nt][e], s[sub][nt][e + 2]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float mn = fmaxf(m[nt][e], mx);
      grew |= mn != m[nt][e];
      corr[nt][e] = fast_exp2(m[nt][e] - mn);
      m[nt][e] = mn;
    }
  }
  // The B fragments of P^T: lane (g, c) needs the weights of query row 8nt+g
  // at tokens 2c, 2c+1 of a sub-tile (lanes 8c + g/2 and 8c + 4 + g/2 hold
  // them, as the low or high half of their packed pair) and at tokens 2c+8,
  // 2c+9 (the same lanes' second pair).
  const int src_a = 8 * c + (g >> 1), src_b = src_a + 4;
  const uint32_t sel = (g & 1) ? 0x7632u : 0x5410u;
  uint32_t pb[kI8Sub][NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
    for (int sub = 0; sub < kI8Sub; ++sub) {
      const float p0 = fast_exp2(s[sub][nt][0] - m[nt][0]);
      const float p1 = fast_exp2(s[sub][nt][1] - m[nt][1]);
      const float p2 = fast_exp2(s[sub][nt][2] - m[nt][0]);
      const float p3 = fast_exp2(s[sub][nt][3] - m[nt][1]);
      ls0 += p0 + p2;
      ls1 += p1 + p3;
      float ra, rb;
      const uint32_t x = Pack<__half>::run(p0 * w[2 * sub], p1 * w[2 * sub], ra, rb);
      const uint32_t y = Pack<__half>::run(p2 * w[2 * sub + 1], p3 * w[2 * sub + 1], ra, rb);
      const uint32_t xa = __shfl_sync(0xffffffffu, x, src_a);
      const uint32_t xb = __shfl_sync(0xffffffffu, x, src_b);
      const uint32_t ya = __shfl_sync(0xffffffffu, y, src_a);
      const uint32_t yb = __shfl_sync(0xffffffffu, y, src_b);
      pb[sub][nt][0] = __byte_perm(xa, xb, sel);
      pb[sub][nt][1] = __byte_perm(ya, yb, sel);
    }
    l[nt][0] = l[nt][0] * corr[nt][0] + ls0;
    l[nt][1] = l[nt][1] * corr[nt][1] + ls1;
  }
  if (__any_sync(0xffffffffu, grew)) {  // O keeps its scale while no row max grows
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int dm = 0; dm < D / 16; ++dm) {
        o[nt][dm][0] *= corr[nt][0];
        o[nt][dm][1] *= corr[nt][1];
        o[nt][dm][2] *= corr[nt][0];
        o[nt][dm][3] *= corr[nt][1];
      }
  }
  // Codes are finite, and the weights outside [vlo, valid) are exact zeros,
  // so no value row needs masking here.  m-tile ch of O^T: row g is dim
  // 16 ch + 2g, row g+8 dim 16 ch + 2g + 1.
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
#pragma unroll
  for (int sub = 0; sub < kI8Sub; ++sub)
#pragma unroll
    for (int ch = 0; ch < D / 16; ++ch) {
      const uint32_t x0 = vw[sub][ch][0] ^ 0x80808080u, x1 = vw[sub][ch][1] ^ 0x80808080u;
      const uint32_t t[4] = {__byte_perm(x0, 0x64646464u, 0x4240u),
                             __byte_perm(x0, 0x64646464u, 0x4341u),
                             __byte_perm(x1, 0x64646464u, 0x4240u),
                             __byte_perm(x1, 0x64646464u, 0x4341u)};
      uint32_t a[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const __half2 v = __hsub2(*reinterpret_cast<const __half2*>(&t[i]), bias);
        a[i] = *reinterpret_cast<const uint32_t*>(&v);
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        MmaOp<__half>::run(o[nt][ch], a, pb[sub][nt][0], pb[sub][nt][1]);
    }
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
                                          int seg_tiles, int seg_units, long long N, int P) {
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
  // seg0: the work unit of the segment's first tile (seg_units virtual units
  // precede it).  The segment is the first one of CTA cfirst's share iff that
  // share starts within the segment's units.
  const int cfirst = cta_of(seg0, N, P), clast = cta_of(seg0 + seg_tiles - 1, N, P);
  const int slot0 = tile_begin(cfirst, N, P) >= seg0 - seg_units ? 0 : 1;
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
// kQ = 0: 16-bit cache; kQ = 1, 2: INT8 cache, query group of at most 8 kQ rows.
template <typename T, int D, int kQ>
__global__ void __launch_bounds__(kThreads, min_ctas_of<kQ>())
    paged_decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_ks,
                        const __grid_constant__ CUtensorMap tm_vs,
                        const __grid_constant__ DecodeParams p) {
  constexpr bool kI8 = kQ > 0;
  constexpr int kNT = kI8 ? kQ : 1;
  constexpr int kT = tile_of<kI8>();  // tokens per stage
  constexpr int kSegUnits = seg_units_of<kI8>();
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
  int* ucum = reinterpret_cast<int*>(smem + L.ucum);
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
  // Plan: clamped lengths and the prefix sum of kT-token tiles per sequence.
  for (int i = tid; i < B; i += kThreads) lens[i] = clamp_len(p.seq_lens[i], cap, p.err_flag);
  __syncthreads();
  if (warp == 0) {
    int carry = 0, ucarry = 0;
    for (int base = 0; base < B; base += 32) {
      const int i = base + lane;
      const int n = i < B ? (lens[i] + kT - 1) / kT - first_tile<kT>(lens[i], p.window) : 0;
      const int u = n > 0 ? n + kSegUnits : 0;
      int x = n, y = u;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int xs = __shfl_up_sync(0xffffffffu, x, off);
        const int ys = __shfl_up_sync(0xffffffffu, y, off);
        if (lane >= off) { x += xs; y += ys; }
      }
      if (i < B) { cum[i] = carry + x - n; ucum[i] = ucarry + y - u; }
      carry += __shfl_sync(0xffffffffu, x, 31);
      ucarry += __shfl_sync(0xffffffffu, y, 31);
    }
    if (lane == 0) { cum[B] = carry; ucum[B] = ucarry; }
  }
  __syncthreads();

  const long long N = static_cast<long long>(hkv) * ucum[B];  // work units
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
  // This CTA's share: units [t_begin, t_end), n_real tiles of them.
  const long long t_begin = tile_begin(c, N, P), t_end = tile_begin(c + 1, N, P);
  auto tiles_before = [&](long long x) -> long long {
    if (x >= N) return static_cast<long long>(hkv) * cum[B];
    int lo = 0, hi = B - 1;  // largest b with hkv*ucum[b] <= x
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (static_cast<long long>(hkv) * ucum[mid] <= x) lo = mid; else hi = mid - 1;
    }
    const int nb = cum[lo + 1] - cum[lo];
    const long long r = x - static_cast<long long>(hkv) * ucum[lo];
    const long long g = r / (nb + kSegUnits);
    const long long jj = r - g * (nb + kSegUnits) - kSegUnits;
    return static_cast<long long>(hkv) * cum[lo] + g * nb + (jj < 0 ? 0 : (jj > nb ? nb : jj));
  };
  const int n_real = t_begin < t_end ? static_cast<int>(tiles_before(t_end) - tiles_before(t_begin))
                                     : 0;
  if (n_real <= 0) return;

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    Cursor cur;
    cur.locate(t_begin, cum, ucum, B, hkv, kSegUnits);
    const int nsub = kT / p.box_tokens;
    // Bytes of one box: a 64-element half of box_tokens 16-bit rows, or
    // box_tokens whole 128-byte code rows.
    const uint32_t box_bytes = static_cast<uint32_t>(p.box_tokens) * 128u;
    const uint32_t q_bytes = static_cast<uint32_t>(G) * 128u * kHalves;
    // Appending: the lane's 16-byte piece of the new K row (lanes < kChunks)
    // or V row (lanes kChunks .. 2 kChunks - 1) of segment (b, g), loaded one
    // tile before the segment's last tile so its latency is off the path.
    constexpr int kChunks = D * 2 / 16;
    const bool new_is_v = lane >= kChunks;
    const int new_q16 = lane - (new_is_v ? kChunks : 0);
    uint4 new_piece = make_uint4(0u, 0u, 0u, 0u);
    bool new_ready = false;
    auto load_new_piece = [&](const Cursor& at) {
      if (lane < 2 * kChunks)
        new_piece = __ldg(reinterpret_cast<const uint4*>(
                              static_cast<const T*>(new_is_v ? p.new_v : p.new_k) +
                              (static_cast<long long>(at.b) * p.num_kv_heads + at.g) * D) +
                          new_q16);
      new_ready = true;
    };
    int it = 0;
    for (; it < n_real; ++it) {
      const int stage = it % kStages;
      const uint32_t phase = (it / kStages) & 1;
      // Look up this tile's physical blocks first: the table load's latency
      // overlaps the wait for a free stage.
      const int Lb = lens[cur.b];
      const int tok = (first_tile<kT>(Lb, p.window) + cur.j) * kT + lane * p.box_tokens;
      // A box wholly below the band is not fetched (its rows are masked).
      const bool wanted = lane < nsub && tok < Lb && tok + p.box_tokens > band_lo(Lb, p.window);
      int pb = -1;
      if (wanted)
        pb = __ldg(&p.block_table[static_cast<long long>(cur.b) * p.max_blocks +
                                  (tok >> p.log2_bs)]);
      if (p.new_k != nullptr && cur.j + 2 == cur.n) load_new_piece(cur);
      if (p.new_k != nullptr && cur.j == cur.n - 1) {
        // The last tile of segment (b, g) holds the new token: write its K/V
        // rows for head g, make the writes visible to the TMA unit, then load
        // the tile as usual.  No other CTA reads them.
        if (!new_ready) load_new_piece(cur);
        new_ready = false;
        const int pos = Lb - 1;
        const int pbn = __ldg(&p.block_table[static_cast<long long>(cur.b) * p.max_blocks +
                                             (pos >> p.log2_bs)]);
        if (pbn >= 0 && pbn < p.num_blocks) {
          const int in_blk = pos & (p.block_size - 1);
          const long long dst_row =
              (static_cast<long long>(pbn) * p.block_size + in_blk) * p.num_kv_heads + cur.g;
          if constexpr (kI8) {
            // Lanes 0-15 quantise the K row, lanes 16-31 the V row, 8
            // elements each (the arithmetic of kvc_reshape_and_cache_int8).
            static_assert(D == 128, "8 elements per lane, 16 lanes per row");
            const bool is_v = new_is_v;
            const int l16 = new_q16;
            const T* pv = reinterpret_cast<const T*>(&new_piece);
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = static_cast<float>(pv[e]);
            uint32_t packed[2];
            float sc;
            quantize_row_int8<8, 16>(x, packed, sc);
            reinterpret_cast<uint2*>(static_cast<int8_t*>(is_v ? p.v_cache : p.k_cache) +
                                     dst_row * D)[l16] = make_uint2(packed[0], packed[1]);
            if (l16 == 0)
              (is_v ? p.v_scales : p.k_scales)[(static_cast<long long>(pbn) * p.num_kv_heads +
                                                cur.g) * p.block_size + in_blk] = sc;
            asm volatile("fence.proxy.async.global;" ::: "memory");
          } else {
            if (lane < 2 * kChunks) {
              *(reinterpret_cast<uint4*>(static_cast<T*>(new_is_v ? p.v_cache : p.k_cache) +
                                         dst_row * D) + new_q16) = new_piece;
              asm volatile("fence.proxy.async.global;" ::: "memory");
            }
          }
          if (lane == 0 && cur.g == 0 && p.slot_out)
            p.slot_out[cur.b] = pbn * p.block_size + in_blk;
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
            uint8_t* sdst = st + L.scales + (lane << p.log2_sslot);
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
  cur.locate(t_begin, cum, ucum, B, hkv, kSegUnits);
  const int ctid = warp * 32 + lane;
  // 16-bit cache: o, m, l of query rows g, g+8 (mma M side).  INT8 cache:
  // o8, m8, l8 of query rows 8nt + 2c, 2c+1 (N side), qb the query fragments.
  float o[kI8 ? 1 : D / 8][4], m[2], l[2];
  float o8[kNT][kI8 ? D / 16 : 1][4], m8[kNT][2], l8[kNT][2];
  uint32_t qb[kI8 ? D / 16 : 1][kNT][2];
  auto reset = [&]() {
    if constexpr (kI8) {
#pragma unroll
      for (int nt = 0; nt < kNT; ++nt) {
#pragma unroll
        for (int n = 0; n < D / 16; ++n)
#pragma unroll
          for (int e = 0; e < 4; ++e) o8[nt][n][e] = 0.f;
        m8[nt][0] = m8[nt][1] = -INFINITY;
        l8[nt][0] = l8[nt][1] = 0.f;
      }
    } else {
#pragma unroll
      for (int n = 0; n < D / 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[n][e] = 0.f;
      m[0] = m[1] = -INFINITY;
      l[0] = l[1] = 0.f;
    }
  };
  reset();
  bool need_q = true;  // INT8: the segment's query fragments are still to be loaded
  const I8Lane i8ofs(warp, lane, p.log2_box, p.log2_sslot);
  int seg_first_j = cur.j;
  int slot = 0;  // 0 for the first segment this CTA touches, 1 afterwards
  const uint32_t sbase = smem_u32(smem);
  int it = 0;
  for (; it < n_real; ++it) {
    const int stage = it % kStages;
    const uint32_t phase = (it / kStages) & 1;
    bool ok = !*abort_flag && mbar_wait_bounded(&full[stage], phase, p.err_flag);
    if (!ok) *abort_flag = 1;
    if constexpr (kI8) {
      // The first tile of a segment share: its query rows into registers
      // (after a failed wait they are stale but still in bounds).
      if (need_q) {
        load_q_i8<T, D, kNT>(sbase + stage * L.stage + L.qoff, L.q_half, G, lane, qb);
        need_q = false;
      }
    }
    const int Lc = lens[cur.b];
    constexpr int kRows = kT / kConsumerWarps;                // the warp's rows: 16 or 32
    const int row0 = (first_tile<kT>(Lc, p.window) + cur.j) * kT + warp * kRows;
    const int valid = min(kRows, Lc - row0);                  // rows [vlo, valid) of the
    const int vlo = max(0, band_lo(Lc, p.window) - row0);     // warp's are attended
    if (ok && valid > vlo) {
      const uint32_t kb = sbase + stage * L.stage;
      if constexpr (kI8)
        attend_i8<D, kNT>(kb, kb + kKBytes, kb + L.scales, kb + L.scales + kScaleBytes,
                             i8ofs, lane, vlo, valid, p.scale_log2, qb, o8, m8, l8);
      else
        attend_16<T, D>(kb, kb + kKBytes, warp, lane, vlo, valid, p.scale_log2, kb + L.qoff,
                        L.q_half, G, o, m, l);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);

    const bool last_of_seg = cur.j == cur.n - 1;
    if (last_of_seg || it == n_real - 1) {
      // ---- finalize this segment's share: merge the 4 warps' states.
      const bool complete = seg_first_j == 0 && last_of_seg;
      if constexpr (kI8) {
        // l: sum the 8 lanes (g) of each query; m is already the same there.
        // Lane (g, c) holds dims 16ch + 2g, 2g+1 of query rows 8nt + 2c + e.
        const int g8 = lane >> 2, c8 = lane & 3;
#pragma unroll
        for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float x = l8[nt][e];
            x += __shfl_xor_sync(0xffffffffu, x, 4);
            x += __shfl_xor_sync(0xffffffffu, x, 8);
            x += __shfl_xor_sync(0xffffffffu, x, 16);
            const int r = nt * 8 + 2 * c8 + e;
            if (r < G) {
              if (g8 == 0) {
                cmb_m[warp * G + r] = m8[nt][e];
                cmb_l[warp * G + r] = x;
              }
#pragma unroll
              for (int ch = 0; ch < D / 16; ++ch)
                *reinterpret_cast<float2*>(&cmb_o[(warp * G + r) * D + 16 * ch + 2 * g8]) =
                    make_float2(o8[nt][ch][e], o8[nt][ch][e + 2]);
            }
          }
      } else {
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
      }
      named_bar_sync(1, kConsumerWarps * 32);
      finish_share<T, D>(p, cmb_m, cmb_l, cmb_o, last_flag, abort_flag + 2,
                         reinterpret_cast<int*>(smem + L.pieces), ctid, cur.b, cur.g,
                         complete, c, slot,
                         static_cast<long long>(hkv) * ucum[cur.b] +
                             static_cast<long long>(cur.g) * (cur.n + kSegUnits) + kSegUnits,
                         cur.n, kSegUnits, N, P);
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

template <typename T, int D, int kQ>
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
    cudaFuncSetAttribute(paged_decode_kernel<T, D, kQ>,
                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                         Layout<D, (kQ > 0)>(kMaxBatch, 16).total);
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, paged_decode_kernel<T, D, kQ>,
                                                      kThreads, smem) != cudaSuccess ||
        occ < 1)
      occ = 1;
    cache[{dev, smem}] = occ;
    return occ;
  }
};

template <typename T, int D, int kQ>
kvc_status run_decode(const DecodeArgs& a) {
  constexpr bool kI8 = kQ > 0;
  const int G = a.num_q_heads / a.num_kv_heads;
  const size_t smem = Layout<D, kI8>(a.batch, G).total;
  const int occ = DecodeKernel<T, D, kQ>::occupancy(smem);  // also sets the smem limit
  const int P = a.num_ctas > 0 ? a.num_ctas : device_sm_count() * occ;
  if (a.workspace_bytes < paged_decode_workspace_bytes(G, D, P) || a.workspace == nullptr)
    return KVC_ERR_WORKSPACE;

  // Boxes of at most 64 tokens: a box wholly past a sequence's end is not
  // fetched, so the tail of its last tile costs less than 64 rows.
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
  p.k_scales = const_cast<float*>(a.key_scales);
  p.v_scales = const_cast<float*>(a.value_scales);
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
  p.log2_sslot = p.log2_box + 2 > 7 ? p.log2_box + 2 : 7;
  p.window = a.window;
  p.scale_log2 = a.scale * 1.4426950408889634f;

  paged_decode_kernel<T, D, kQ><<<P, kThreads, smem, a.stream>>>(tk, tv, tq, tks, tvs, p);
  return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

template <int kQ>
int num_ctas_for(int group, int head_dim, kvc_dtype dtype) {
  constexpr bool kI8 = kQ > 0;
  const int sms = device_sm_count();
  if (sms <= 0) return 0;
  // The smallest batch needs the least shared memory, hence the most CTAs.
  if (head_dim == 64 && !kI8) {
    const size_t smem = Layout<64, false>(1, group).total;
    return sms * (dtype == KVC_BF16 ? DecodeKernel<__nv_bfloat16, 64, 0>::occupancy(smem)
                                    : DecodeKernel<__half, 64, 0>::occupancy(smem));
  }
  if (head_dim == 128) {
    const size_t smem = Layout<128, kI8>(1, group).total;
    return sms * (dtype == KVC_BF16 ? DecodeKernel<__nv_bfloat16, 128, kQ>::occupancy(smem)
                                    : DecodeKernel<__half, 128, kQ>::occupancy(smem));
  }
  return 0;
}

}  // namespace

size_t paged_decode_workspace_bytes(int group, int head_dim, int ctas) {
  return counter_bytes(ctas) + static_cast<size_t>(ctas) * 2 * group * (head_dim + 2) * sizeof(float);
}

int paged_decode_num_ctas(int group, int head_dim, kvc_dtype dtype, int num_ctas, bool int8) {
  if (num_ctas > 0) return num_ctas;
  if (!int8) return num_ctas_for<0>(group, head_dim, dtype);
  return group <= 8 ? num_ctas_for<1>(group, head_dim, dtype)
                    : num_ctas_for<2>(group, head_dim, dtype);
}

kvc_status launch_paged_decode(const DecodeArgs& a) {
  if (a.key_scales != nullptr) {  // INT8 cache (head_dim 128)
    if (a.head_dim != 128) return KVC_ERR_UNSUPPORTED;
    const bool wide = a.num_q_heads / a.num_kv_heads > 8;  // two 8-row query tiles
    if (a.dtype == KVC_BF16)
      return wide ? run_decode<__nv_bfloat16, 128, 2>(a) : run_decode<__nv_bfloat16, 128, 1>(a);
    return wide ? run_decode<__half, 128, 2>(a) : run_decode<__half, 128, 1>(a);
  }
  if (a.head_dim == 64)
    return a.dtype == KVC_BF16 ? run_decode<__nv_bfloat16, 64, 0>(a)
                               : run_decode<__half, 64, 0>(a);
  if (a.head_dim == 128)
    return a.dtype == KVC_BF16 ? run_decode<__nv_bfloat16, 128, 0>(a)
                               : run_decode<__half, 128, 0>(a);
  return KVC_ERR_UNSUPPORTED;
}

}  // namespace kvc
