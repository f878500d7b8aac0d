// Slot-mapping construction and the paged cache write.
//
// Slot formula: "external-cannbot-model-model-infer-kvcache", 3.1 Mapping
// Formula (logical block = pos / block_size, offset = pos % block_size,
// slot = block_table[seq][logical] * block_size + offset) and 3.3
// slot_mapping Construction; the packed form follows the hotelren.com notes
// "Paged KV Cache + Packed Sequence" 3.3 (packed token -> request and offset
// -> logical block -> physical block).
// Cache write: ai6s.net KVCache article 4.2 -- each new row is copied,
// unchanged, to its cache position.
// INT8 cache write: the same placement, with each row quantised as the
// KVCache skill's quantized-KV parameters imply (codes plus dequantisation
// scales; the article's FP16 -> INT8 halving of the bytes).  The pages fix no
// scheme; this library stores one symmetric fp32 scale per written row
// (token, kv head), its codes decided in IEEE fp32: amax = max|x|, inv = 127 /
// amax, scale = amax / 127 (round-to-nearest divisions), code = x * inv
// (round-to-nearest product) rounded half to even and clamped to +-127; a
// zero row has scale 0 and codes 0.  Codes keep the 16-bit cache's layout
// [num_blocks, block_size, Hkv, D]; scales are [num_blocks, Hkv, block_size].
#include <cuda_runtime.h>

#include <type_traits>

#include "kvc_device.cuh"
#include "kvc_host.h"

namespace kvc {

namespace {

__global__ void slot_mapping_kernel(const int32_t* __restrict__ block_table, int max_blocks,
                                    const int32_t* __restrict__ cu_seqlens,
                                    const int32_t* __restrict__ start_pos, int num_seqs,
                                    int num_tokens, int block_size, int num_blocks,
                                    int32_t* __restrict__ slot_mapping, uint32_t* err_flag) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= num_tokens) return;
  int s, pos;
  if (cu_seqlens == nullptr) {
    s = t;
    pos = start_pos[s];
  } else {
    // Sequence owning packed token t: the last s with cu_seqlens[s] <= t.
    int lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cu_seqlens[mid] <= t) lo = mid; else hi = mid - 1;
    }
    s = lo;
    pos = start_pos[s] + (t - cu_seqlens[s]);
  }
  int32_t slot = -1;
  const int lb = pos >= 0 ? pos / block_size : -1;
  if (lb < 0 || lb >= max_blocks) {
    set_flag(err_flag, KVC_FLAG_LEN_RANGE);
  } else {
    const int pb = block_table[static_cast<int64_t>(s) * max_blocks + lb];
    if (pb < 0 || pb >= num_blocks) {
      set_flag(err_flag, KVC_FLAG_BLOCK_ID_RANGE);
    } else {
      slot = pb * block_size + (pos - lb * block_size);
    }
  }
  slot_mapping[t] = slot;
}

// One thread per 16-byte chunk; consecutive threads copy consecutive chunks
// of one token row, so both the read of key/value and the write into the
// cache row are fully coalesced.  K chunks come first, then V chunks.
__global__ void reshape_and_cache_kernel(const uint4* __restrict__ key,
                                         const uint4* __restrict__ value,
                                         uint4* __restrict__ key_cache,
                                         uint4* __restrict__ value_cache,
                                         const int32_t* __restrict__ slot_mapping,
                                         int num_tokens, int chunks_k, int chunks_v,
                                         int64_t num_slots, uint32_t* err_flag) {
  const int per_tok = chunks_k + chunks_v;
  const int64_t total = static_cast<int64_t>(num_tokens) * per_tok;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / per_tok);
    const int c = static_cast<int>(i - static_cast<int64_t>(t) * per_tok);
    const int32_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (c == 0) set_flag(err_flag, KVC_FLAG_SLOT_RANGE);
      continue;
    }
    if (c < chunks_k) {
      key_cache[static_cast<int64_t>(slot) * chunks_k + c] =
          key[static_cast<int64_t>(t) * chunks_k + c];
    } else {
      const int cv = c - chunks_k;
      value_cache[static_cast<int64_t>(slot) * chunks_v + cv] =
          value[static_cast<int64_t>(t) * chunks_v + cv];
    }
  }
}

// Copy-on-write block copies: pair i copies block src[i] to block dst[i], as
// 16-byte chunks (one thread per chunk, consecutive threads on consecutive
// chunks, so reads and writes are coalesced).  K chunks of a pair come first,
// then V chunks.  A pair with src < 0 is skipped; an id outside the pool is
// skipped and flagged.
__global__ void copy_blocks_kernel(uint4* __restrict__ key_cache, uint4* __restrict__ value_cache,
                                   const int32_t* __restrict__ src,
                                   const int32_t* __restrict__ dst, int num_pairs,
                                   int64_t chunks_k, int64_t chunks_v, int num_blocks,
                                   uint32_t* err_flag) {
  const int64_t per_pair = chunks_k + chunks_v;
  const int64_t total = static_cast<int64_t>(num_pairs) * per_pair;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int pair = static_cast<int>(i / per_pair);
    const int64_t c = i - static_cast<int64_t>(pair) * per_pair;
    const int32_t s = src[pair], d = dst[pair];
    if (s < 0) continue;
    if (s >= num_blocks || d < 0 || d >= num_blocks) {
      if (c == 0) set_flag(err_flag, KVC_FLAG_BLOCK_ID_RANGE);
      continue;
    }
    if (c < chunks_k) {
      key_cache[d * chunks_k + c] = key_cache[s * chunks_k + c];
    } else {
      const int64_t cv = c - chunks_k;
      value_cache[d * chunks_v + cv] = value_cache[s * chunks_v + cv];
    }
  }
}

__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }

// One warp per (token, kv head, K or V) row of D elements: lane l holds D/32
// consecutive elements, amax is a warp max, and the lane writes its codes.
template <typename T, int D>
__global__ void reshape_and_cache_int8_kernel(const T* __restrict__ key,
                                              const T* __restrict__ value,
                                              int8_t* __restrict__ key_codes,
                                              int8_t* __restrict__ value_codes,
                                              float* __restrict__ key_scales,
                                              float* __restrict__ value_scales,
                                              const int32_t* __restrict__ slot_mapping,
                                              int num_tokens, int num_kv_heads, int block_size,
                                              int64_t num_slots, uint32_t* err_flag) {
  constexpr int E = D / 32;  // elements per lane: 2 (D 64) or 4 (D 128)
  const int lane = threadIdx.x & 31;
  const int64_t w0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  const int64_t rows = static_cast<int64_t>(num_tokens) * num_kv_heads * 2;
  for (int64_t r = w0; r < rows; r += nw) {
    const int is_v = static_cast<int>(r & 1);
    const int64_t th = r >> 1;  // token * Hkv + head
    const int t = static_cast<int>(th / num_kv_heads);
    const int h = static_cast<int>(th - static_cast<int64_t>(t) * num_kv_heads);
    const int32_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_slots) {
      if (lane == 0 && is_v == 0 && h == 0) set_flag(err_flag, KVC_FLAG_SLOT_RANGE);
      continue;
    }
    const T* src = (is_v ? value : key) + th * D + lane * E;
    float x[E];
    if constexpr (E == 4) {
      const uint2 u = *reinterpret_cast<const uint2*>(src);
      const T* pv = reinterpret_cast<const T*>(&u);
#pragma unroll
      for (int e = 0; e < 4; ++e) x[e] = to_f32(pv[e]);
    } else {
      const uint32_t u = *reinterpret_cast<const uint32_t*>(src);
      const T* pv = reinterpret_cast<const T*>(&u);
#pragma unroll
      for (int e = 0; e < 2; ++e) x[e] = to_f32(pv[e]);
    }
    uint32_t packed[1];
    float scale;
    quantize_row_int8<E, 32>(x, packed, scale);
    const int64_t blk = slot / block_size, in_blk = slot - blk * block_size;
    int8_t* dst = (is_v ? value_codes : key_codes) +
                  (static_cast<int64_t>(slot) * num_kv_heads + h) * D + lane * E;
    if constexpr (E == 4) *reinterpret_cast<uint32_t*>(dst) = packed[0];
    else *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(packed[0]);
    if (lane == 0)
      (is_v ? value_scales : key_scales)[(blk * num_kv_heads + h) * block_size + in_blk] = scale;
  }
}

}  // namespace

kvc_status launch_reshape_and_cache_int8(const void* key, const void* value, void* key_codes,
                                         void* value_codes, float* key_scales,
                                         float* value_scales, const int32_t* slot_mapping,
                                         int num_tokens, int num_kv_heads, int head_dim,
                                         int block_size, int num_blocks, kvc_dtype dtype,
                                         uint32_t* err_flag, cudaStream_t stream) {
  if (num_tokens == 0) return KVC_OK;
  const int64_t rows = static_cast<int64_t>(num_tokens) * num_kv_heads * 2;
  const int threads = 256;  // 8 rows per CTA pass
  const int64_t want = (rows * 32 + threads - 1) / threads;
  const int cap = device_sm_count() * 16;
  const int grid = static_cast<int>(want < cap ? want : cap);
  const int64_t ns = static_cast<int64_t>(num_blocks) * block_size;
  auto go = [&](auto tag, auto dim) {
    using T = decltype(tag);
    constexpr int D = decltype(dim)::value;
    reshape_and_cache_int8_kernel<T, D><<<grid, threads, 0, stream>>>(
        static_cast<const T*>(key), static_cast<const T*>(value),
        static_cast<int8_t*>(key_codes), static_cast<int8_t*>(value_codes), key_scales,
        value_scales, slot_mapping, num_tokens, num_kv_heads, block_size, ns, err_flag);
  };
  using D64 = std::integral_constant<int, 64>;
  using D128 = std::integral_constant<int, 128>;
  if (dtype == KVC_BF16) {
    if (head_dim == 128) go(__nv_bfloat16(), D128()); else go(__nv_bfloat16(), D64());
  } else {
    if (head_dim == 128) go(__half(), D128()); else go(__half(), D64());
  }
  return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

kvc_status launch_copy_blocks(void* key_cache, void* value_cache, const int32_t* src,
                              const int32_t* dst, int num_pairs, int64_t block_bytes_k,
                              int64_t block_bytes_v, int num_blocks, uint32_t* err_flag,
                              cudaStream_t stream) {
  if (num_pairs == 0) return KVC_OK;
  const int64_t chunks_k = block_bytes_k / 16;
  const int64_t chunks_v = value_cache ? block_bytes_v / 16 : 0;
  const int64_t total = static_cast<int64_t>(num_pairs) * (chunks_k + chunks_v);
  const int threads = 256;
  const int64_t want = (total + threads - 1) / threads;
  const int cap = device_sm_count() * 8;
  const int grid = static_cast<int>(want < cap ? want : cap);
  copy_blocks_kernel<<<grid, threads, 0, stream>>>(
      static_cast<uint4*>(key_cache), static_cast<uint4*>(value_cache), src, dst, num_pairs,
      chunks_k, chunks_v, num_blocks, err_flag);
  return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

kvc_status launch_slot_mapping(const int32_t* block_table, int max_blocks_per_seq,
                               const int32_t* cu_seqlens, const int32_t* start_pos, int num_seqs,
                               int num_tokens, int block_size, int num_blocks,
                               int32_t* slot_mapping, uint32_t* err_flag, cudaStream_t stream) {
  if (num_tokens == 0) return KVC_OK;
  const int threads = 256;
  const int grid = (num_tokens + threads - 1) / threads;
  slot_mapping_kernel<<<grid, threads, 0, stream>>>(block_table, max_blocks_per_seq, cu_seqlens,
                                                    start_pos, num_seqs, num_tokens, block_size,
                                                    num_blocks, slot_mapping, err_flag);
  return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

kvc_status launch_reshape_and_cache(const void* key, const void* value, void* key_cache,
                                    void* value_cache, const int32_t* slot_mapping,
                                    int num_tokens, int num_kv_heads, int head_dim_k,
                                    int head_dim_v, int block_size, int num_blocks,
                                    uint32_t* err_flag, cudaStream_t stream) {
  if (num_tokens == 0) return KVC_OK;
  const int chunks_k = num_kv_heads * head_dim_k * 2 / 16;
  const int chunks_v = value ? num_kv_heads * head_dim_v * 2 / 16 : 0;
  const int64_t total = static_cast<int64_t>(num_tokens) * (chunks_k + chunks_v);
  const int threads = 256;
  const int64_t want = (total + threads - 1) / threads;
  const int cap = device_sm_count() * 16;
  const int grid = static_cast<int>(want < cap ? want : cap);
  reshape_and_cache_kernel<<<grid, threads, 0, stream>>>(
      static_cast<const uint4*>(key), static_cast<const uint4*>(value),
      static_cast<uint4*>(key_cache), static_cast<uint4*>(value_cache), slot_mapping, num_tokens,
      chunks_k, chunks_v, static_cast<int64_t>(num_blocks) * block_size, err_flag);
  return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

}  // namespace kvc
