// Host-side internals of the kvc library: argument checks, device queries,
// TMA descriptor encoding and the per-kernel launchers the C ABI calls.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/kvc.h"

namespace kvc {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
inline int ilog2(int x) {
  int r = 0;
  while ((1 << r) < x) ++r;
  return r;
}

// SM count of the current device (cached per device ordinal).
int device_sm_count();

// Encode a tiled TMA descriptor over a 16-bit tensor of rank `rank`.
// dims/strides follow cuTensorMapEncodeTiled (dims innermost first, strides
// in bytes for dims 1..rank-1).  Returns false if the driver rejects it.
bool encode_tmap_16bit(CUtensorMap* map, kvc_dtype dtype, int rank, const void* base,
                       const uint64_t* dims, const uint64_t* strides_bytes,
                       const uint32_t* box, bool swizzle128);
// The same for any element type.  The L2 promotion is the widest of 64 / 128 /
// 256 bytes that the box's contiguous bytes fill (none below 64).
bool encode_tmap(CUtensorMap* map, CUtensorMapDataType type, int rank, const void* base,
                 const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                 bool swizzle128);

kvc_status launch_slot_mapping(const int32_t* block_table, int max_blocks_per_seq,
                               const int32_t* cu_seqlens, const int32_t* start_pos, int num_seqs,
                               int num_tokens, int block_size, int num_blocks,
                               int32_t* slot_mapping, uint32_t* err_flag, cudaStream_t stream);

kvc_status launch_reshape_and_cache(const void* key, const void* value, void* key_cache,
                                    void* value_cache, const int32_t* slot_mapping,
                                    int num_tokens, int num_kv_heads, int head_dim_k,
                                    int head_dim_v, int block_size, int num_blocks,
                                    uint32_t* err_flag, cudaStream_t stream);

kvc_status launch_copy_blocks(void* key_cache, void* value_cache, const int32_t* src,
                              const int32_t* dst, int num_pairs, int64_t block_bytes_k,
                              int64_t block_bytes_v, int num_blocks, uint32_t* err_flag,
                              cudaStream_t stream);

kvc_status launch_reshape_and_cache_int8(const void* key, const void* value, void* key_codes,
                                         void* value_codes, float* key_scales,
                                         float* value_scales, const int32_t* slot_mapping,
                                         int num_tokens, int num_kv_heads, int head_dim,
                                         int block_size, int num_blocks, kvc_dtype dtype,
                                         uint32_t* err_flag, cudaStream_t stream);

kvc_status launch_rope_table(float* cos_sin, int max_position, int rope_dim, float base,
                             cudaStream_t stream);
kvc_status launch_rmsnorm_rope_cache(const void* kv, const void* gamma, float eps,
                                     const float* cos_sin, int max_position,
                                     const int32_t* positions, const int32_t* slot_mapping,
                                     void* cache_norm, void* cache_rope, int num_tokens,
                                     int num_heads, int d_norm, int d_rope, int block_size,
                                     int num_blocks, kvc_dtype dtype, uint32_t* err_flag,
                                     cudaStream_t stream);

struct DecodeArgs {
  const void* q;
  const void* key_cache;
  const void* value_cache;
  const int32_t* block_table;
  const int32_t* seq_lens;
  void* out;
  int batch, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks;
  float scale;
  kvc_dtype dtype;
  int num_ctas;
  void* workspace;
  size_t workspace_bytes;
  uint32_t* err_flag;
  cudaStream_t stream;
  // Appending decode (all null for plain decode): see kvc_paged_decode_append.
  const void* new_key = nullptr;
  const void* new_value = nullptr;
  int32_t* slot_out = nullptr;
  // Band decode: attend to the last `window` tokens only (0: all of them).
  int window = 0;
  // INT8 cache (null for a 16-bit cache): key_cache / value_cache hold int8
  // codes, these the fp32 scales [num_blocks, Hkv, block_size].
  const float* key_scales = nullptr;
  const float* value_scales = nullptr;
};

// The arguments of kvc_paged_decode gathered into a DecodeArgs.
DecodeArgs make_decode_args(const void* q, const void* key_cache, const void* value_cache,
                            const int32_t* block_table, const int32_t* seq_lens, void* out,
                            int batch, int num_q_heads, int num_kv_heads, int head_dim,
                            int block_size, int max_blocks_per_seq, int num_blocks, float scale,
                            kvc_dtype dtype, int num_ctas, void* workspace,
                            size_t workspace_bytes, uint32_t* err_flag, kvc_stream_t stream);
// Host-side checks shared by the decode entry points (every check except the
// workspace size); *empty is set for a batch of 0, which has nothing to do.
kvc_status check_decode_args(const DecodeArgs& a, bool* empty);

// Persistent CTAs the decode kernel would use for this shape (num_ctas <= 0
// means "auto").  Returns 0 for an unsupported shape.
int paged_decode_num_ctas(int group, int head_dim, kvc_dtype dtype, int num_ctas,
                          bool int8 = false);
size_t paged_decode_workspace_bytes(int group, int head_dim, int ctas);
kvc_status launch_paged_decode(const DecodeArgs& a);

struct PrefillArgs {
  const void* q;
  const void* key;
  const void* value;
  const int32_t* cu_seqlens;
  const int32_t* context_lens;
  const int32_t* slot_mapping;
  const int32_t* block_table;
  void* key_cache;
  void* value_cache;
  void* out;
  int num_seqs, num_tokens, max_seqlen_q, num_q_heads, num_kv_heads, head_dim;
  int block_size, max_blocks_per_seq, num_blocks;
  float scale;
  kvc_dtype dtype;
  uint32_t* err_flag;
  cudaStream_t stream;
  // Band: a query at position p sees p - window + 1 .. p only (0: 0 .. p).
  int window = 0;
};

// Cache write of the chunk's K/V rows, then the causal attention kernel.
kvc_status launch_varlen_prefill(const PrefillArgs& a);
// The causal attention part alone (tcgen05 kernel).
kvc_status launch_prefill_attention_tc(const PrefillArgs& a);
// Two query heads per CTA; requires an even GQA group size.
kvc_status launch_prefill_attention_tc2(const PrefillArgs& a);
// The cache write and the attention in one launch, for chunks without cached
// context (context_lens null): K/V tiles come from the packed input and a
// writer warp stores the chunk's rows at slot_mapping; even GQA group size.
kvc_status launch_prefill_fused_tc2(const PrefillArgs& a);

struct MlaArgs {
  const void* q_nope;
  const void* q_rope;
  const void* cache_nope;
  const void* cache_rope;
  const int32_t* block_table;
  const int32_t* seq_lens;
  void* out;
  int batch, block_size, max_blocks_per_seq, num_blocks;
  float scale;
  kvc_dtype dtype;
  int num_ctas;
  void* workspace;
  size_t workspace_bytes;
  uint32_t* err_flag;
  cudaStream_t stream;
  // Appending decode (all null for plain decode): see kvc_mla_paged_decode_append.
  const void* new_nope = nullptr;
  const void* new_rope = nullptr;
  int32_t* slot_out = nullptr;
};

// CTAs (an even number: pairs) the MLA kernel runs with (num_ctas <= 0: auto).
int mla_decode_num_ctas(int num_ctas);
size_t mla_decode_workspace_bytes(int ctas);
kvc_status launch_mla_decode(const MlaArgs& a);

}  // namespace kvc
