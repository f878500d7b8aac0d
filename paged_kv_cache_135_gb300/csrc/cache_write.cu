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
#include <cuda_runtime.h>

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

}  // namespace

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
