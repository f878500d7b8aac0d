// The library's C ABI (include/kvc.h): host-side validation, then launches.
// Every check here runs before anything is enqueued, so a rejected call has
// no effect on the device.
#include <cuda.h>
#include <cuda_runtime.h>

#include <math.h>
#include <mutex>

#include "../../include/kvc.h"
#include "kvc_host.h"

namespace kvc {

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  int& c = cached[dev & 63];
  if (c == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    c = n;
  }
  return c;
}

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

bool encode_tmap_16bit(CUtensorMap* map, kvc_dtype dtype, int rank, const void* base,
                       const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                       bool swizzle128) {
  return encode_tmap(map,
                     dtype == KVC_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                     rank, base, dims, strides_bytes, box, swizzle128);
}

bool encode_tmap(CUtensorMap* map, CUtensorMapDataType type, int rank, const void* base,
                 const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                 bool swizzle128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  // L2 promotion no wider than the contiguous bytes a box covers: one row of
  // dimension 0, or box[1] such rows when they are adjacent and the box spans
  // the whole row.  A wider promotion fetches the neighbouring row (another
  // head's 128-byte code row of an INT8 cache, say), which the box does not use.
  const uint64_t elt = type == CU_TENSOR_MAP_DATA_TYPE_UINT8 ? 1
                       : type == CU_TENSOR_MAP_DATA_TYPE_FLOAT32 ? 4 : 2;
  uint64_t span = dims[0] * elt;
  if (rank > 1 && box[0] == dims[0] && strides_bytes[0] == span) span *= box[1];
  const CUtensorMapL2promotion promo = span >= 256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                                       : span >= 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                       : span >= 64 ? CU_TENSOR_MAP_L2_PROMOTION_L2_64B
                                                    : CU_TENSOR_MAP_L2_PROMOTION_NONE;
  const CUresult r = fn(map, type, static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, s,
                        b, e,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                        promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

DecodeArgs make_decode_args(const void* q, const void* key_cache, const void* value_cache,
                            const int32_t* block_table, const int32_t* seq_lens, void* out,
                            int batch, int num_q_heads, int num_kv_heads, int head_dim,
                            int block_size, int max_blocks_per_seq, int num_blocks, float scale,
                            kvc_dtype dtype, int num_ctas, void* workspace,
                            size_t workspace_bytes, uint32_t* err_flag, kvc_stream_t stream) {
  DecodeArgs a;
  a.q = q;
  a.key_cache = key_cache;
  a.value_cache = value_cache;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.out = out;
  a.batch = batch;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.scale = scale;
  a.dtype = dtype;
  a.num_ctas = num_ctas;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.err_flag = err_flag;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  return a;
}

kvc_status check_decode_args(const DecodeArgs& a, bool* empty) {
  *empty = false;
  if (a.dtype != KVC_F16 && a.dtype != KVC_BF16) return KVC_ERR_INVALID_ARG;
  if (a.batch < 0 || a.num_q_heads <= 0 || a.num_kv_heads <= 0 || a.head_dim <= 0 ||
      a.block_size <= 0 || a.max_blocks_per_seq <= 0 || a.num_blocks <= 0 || a.num_ctas < 0 ||
      a.window < 0)
    return KVC_ERR_INVALID_ARG;
  if (a.num_q_heads % a.num_kv_heads) return KVC_ERR_INVALID_ARG;
  if (!isfinite(a.scale)) return KVC_ERR_INVALID_ARG;
  if (a.num_q_heads / a.num_kv_heads > 16) return KVC_ERR_UNSUPPORTED;
  if (a.head_dim != 64 && a.head_dim != 128) return KVC_ERR_UNSUPPORTED;
  if (!is_pow2(a.block_size) || a.block_size < 8) return KVC_ERR_UNSUPPORTED;
  if (a.batch > 1024) return KVC_ERR_UNSUPPORTED;
  if (static_cast<long long>(a.max_blocks_per_seq) * a.block_size > 0x7fffffffLL)
    return KVC_ERR_UNSUPPORTED;
  if (a.batch == 0) {
    *empty = true;
    return KVC_OK;
  }
  if (!a.q || !a.key_cache || !a.value_cache || !a.block_table || !a.seq_lens || !a.out)
    return KVC_ERR_INVALID_ARG;
  if (!aligned16(a.q) || !aligned16(a.out) || !aligned16(a.key_cache) ||
      !aligned16(a.value_cache) || !aligned16(a.workspace))
    return KVC_ERR_INVALID_ARG;
  return KVC_OK;
}

}  // namespace kvc

using kvc::aligned16;
using kvc::is_pow2;

extern "C" {

const char* kvc_status_string(kvc_status s) {
  switch (s) {
    case KVC_OK: return "KVC_OK";
    case KVC_ERR_INVALID_ARG: return "KVC_ERR_INVALID_ARG";
    case KVC_ERR_UNSUPPORTED: return "KVC_ERR_UNSUPPORTED";
    case KVC_ERR_CUDA: return "KVC_ERR_CUDA";
    case KVC_ERR_WORKSPACE: return "KVC_ERR_WORKSPACE";
    case KVC_ERR_OUT_OF_BLOCKS: return "KVC_ERR_OUT_OF_BLOCKS";
  }
  return "KVC_UNKNOWN_STATUS";
}

int kvc_version(void) { return 100; }

kvc_status kvc_build_slot_mapping(const int32_t* block_table, int max_blocks_per_seq,
                                  const int32_t* cu_seqlens, const int32_t* start_pos,
                                  int num_seqs, int num_tokens, int block_size, int num_blocks,
                                  int32_t* slot_mapping, uint32_t* err_flag,
                                  kvc_stream_t stream) {
  if (num_seqs < 0 || num_tokens < 0 || block_size <= 0 || num_blocks <= 0 ||
      max_blocks_per_seq <= 0)
    return KVC_ERR_INVALID_ARG;
  if (static_cast<long long>(num_blocks) * block_size > 0x7fffffffLL) return KVC_ERR_UNSUPPORTED;
  if (num_tokens == 0) return KVC_OK;
  if (num_seqs == 0 || !block_table || !start_pos || !slot_mapping) return KVC_ERR_INVALID_ARG;
  if (!cu_seqlens && num_tokens != num_seqs) return KVC_ERR_INVALID_ARG;
  return kvc::launch_slot_mapping(block_table, max_blocks_per_seq, cu_seqlens, start_pos,
                                  num_seqs, num_tokens, block_size, num_blocks, slot_mapping,
                                  err_flag, reinterpret_cast<cudaStream_t>(stream));
}

kvc_status kvc_reshape_and_cache(const void* key, const void* value, void* key_cache,
                                 void* value_cache, const int32_t* slot_mapping, int num_tokens,
                                 int num_kv_heads, int head_dim_k, int head_dim_v,
                                 int block_size, int num_blocks, kvc_dtype dtype,
                                 uint32_t* err_flag, kvc_stream_t stream) {
  if (dtype != KVC_F16 && dtype != KVC_BF16) return KVC_ERR_INVALID_ARG;
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim_k <= 0 || block_size <= 0 ||
      num_blocks <= 0)
    return KVC_ERR_INVALID_ARG;
  if ((value == nullptr) != (value_cache == nullptr)) return KVC_ERR_INVALID_ARG;
  if (value && head_dim_v <= 0) return KVC_ERR_INVALID_ARG;
  if (head_dim_k % 8 || (value && head_dim_v % 8)) return KVC_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_blocks) * block_size > 0x7fffffffLL) return KVC_ERR_UNSUPPORTED;
  if (num_tokens == 0) return KVC_OK;
  if (!key || !key_cache || !slot_mapping) return KVC_ERR_INVALID_ARG;
  if (!aligned16(key) || !aligned16(key_cache) || (value && (!aligned16(value) ||
                                                             !aligned16(value_cache))))
    return KVC_ERR_INVALID_ARG;
  return kvc::launch_reshape_and_cache(key, value, key_cache, value_cache, slot_mapping,
                                       num_tokens, num_kv_heads, head_dim_k, head_dim_v,
                                       block_size, num_blocks, err_flag,
                                       reinterpret_cast<cudaStream_t>(stream));
}

kvc_status kvc_copy_blocks(void* key_cache, void* value_cache, const int32_t* src_blocks,
                           const int32_t* dst_blocks, int num_pairs, long long block_bytes_k,
                           long long block_bytes_v, int num_blocks, uint32_t* err_flag,
                           kvc_stream_t stream) {
  if (num_pairs < 0 || num_blocks <= 0 || block_bytes_k <= 0 || block_bytes_k % 16)
    return KVC_ERR_INVALID_ARG;
  if (value_cache && (block_bytes_v <= 0 || block_bytes_v % 16)) return KVC_ERR_INVALID_ARG;
  if (num_pairs == 0) return KVC_OK;
  if (!key_cache || !src_blocks || !dst_blocks) return KVC_ERR_INVALID_ARG;
  if (!aligned16(key_cache) || (value_cache && !aligned16(value_cache)))
    return KVC_ERR_INVALID_ARG;
  return kvc::launch_copy_blocks(key_cache, value_cache, src_blocks, dst_blocks, num_pairs,
                                 block_bytes_k, block_bytes_v, num_blocks, err_flag,
                                 reinterpret_cast<cudaStream_t>(stream));
}

kvc_status kvc_rope_cos_sin_table(float* cos_sin, int max_position, int rope_dim, float base,
                                  kvc_stream_t stream) {
  if (max_position <= 0 || rope_dim <= 0 || rope_dim % 2 || !(base > 0.f) || !isfinite(base))
    return KVC_ERR_INVALID_ARG;
  if (!cos_sin) return KVC_ERR_INVALID_ARG;
  return kvc::launch_rope_table(cos_sin, max_position, rope_dim, base,
                                reinterpret_cast<cudaStream_t>(stream));
}

kvc_status kvc_rmsnorm_rope_cache(const void* kv, const void* gamma, float eps,
                                  const float* cos_sin, int max_position,
                                  const int32_t* positions, const int32_t* slot_mapping,
                                  void* cache_norm, void* cache_rope, int num_tokens,
                                  int num_heads, int d_norm, int d_rope, int block_size,
                                  int num_blocks, kvc_dtype dtype, uint32_t* err_flag,
                                  kvc_stream_t stream) {
  if (dtype != KVC_F16 && dtype != KVC_BF16) return KVC_ERR_INVALID_ARG;
  if (num_tokens < 0 || num_heads <= 0 || d_norm <= 0 || d_rope <= 0 || block_size <= 0 ||
      num_blocks <= 0 || max_position <= 0 || !(eps >= 0.f) || !isfinite(eps))
    return KVC_ERR_INVALID_ARG;
  if (d_norm % 8 || d_rope % 8) return KVC_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_blocks) * block_size > 0x7fffffffLL) return KVC_ERR_UNSUPPORTED;
  if (num_tokens == 0) return KVC_OK;
  if (!kv || !gamma || !cos_sin || !positions || !slot_mapping || !cache_norm || !cache_rope)
    return KVC_ERR_INVALID_ARG;
  if (!aligned16(kv) || !aligned16(gamma) || !aligned16(cache_norm) || !aligned16(cache_rope))
    return KVC_ERR_INVALID_ARG;
  return kvc::launch_rmsnorm_rope_cache(kv, gamma, eps, cos_sin, max_position, positions,
                                        slot_mapping, cache_norm, cache_rope, num_tokens,
                                        num_heads, d_norm, d_rope, block_size, num_blocks, dtype,
                                        err_flag, reinterpret_cast<cudaStream_t>(stream));
}

size_t kvc_paged_decode_workspace_size(int num_q_heads, int num_kv_heads, int head_dim,
                                       int num_ctas) {
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads) return 0;
  const int group = num_q_heads / num_kv_heads;
  if (group > 16 || (head_dim != 64 && head_dim != 128)) return 0;
  // Enough for every variant (dtype, 16-bit or INT8 cache): the automatic
  // CTA count may differ between them.
  int ctas = 0;
  for (const kvc_dtype dt : {KVC_F16, KVC_BF16})
    for (const bool i8 : {false, true}) {
      if (i8 && head_dim != 128) continue;
      const int c = kvc::paged_decode_num_ctas(group, head_dim, dt, num_ctas, i8);
      if (c > ctas) ctas = c;
    }
  return kvc::paged_decode_workspace_bytes(group, head_dim, ctas);
}

kvc_status kvc_paged_decode(const void* q, const void* key_cache, const void* value_cache,
                            const int32_t* block_table, const int32_t* seq_lens, void* out,
                            int batch, int num_q_heads, int num_kv_heads, int head_dim,
                            int block_size, int max_blocks_per_seq, int num_blocks, float scale,
                            kvc_dtype dtype, int num_ctas, void* workspace,
                            size_t workspace_bytes, uint32_t* err_flag, kvc_stream_t stream) {
  const kvc::DecodeArgs a = kvc::make_decode_args(
      q, key_cache, value_cache, block_table, seq_lens, out, batch, num_q_heads, num_kv_heads,
      head_dim, block_size, max_blocks_per_seq, num_blocks, scale, dtype, num_ctas, workspace,
      workspace_bytes, err_flag, stream);
  bool empty = false;
  const kvc_status st = kvc::check_decode_args(a, &empty);
  if (st != KVC_OK || empty) return st;
  return kvc::launch_paged_decode(a);
}

kvc_status kvc_paged_decode_append(const void* q, const void* new_key, const void* new_value,
                                   void* key_cache, void* value_cache, const int32_t* block_table,
                                   const int32_t* seq_lens, int32_t* slot_mapping, void* out,
                                   int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, int max_blocks_per_seq, int num_blocks,
                                   float scale, kvc_dtype dtype, int num_ctas, void* workspace,
                                   size_t workspace_bytes, uint32_t* err_flag,
                                   kvc_stream_t stream) {
  if (batch > 0 && (!new_key || !new_value || !aligned16(new_key) || !aligned16(new_value)))
    return KVC_ERR_INVALID_ARG;
  kvc::DecodeArgs a = kvc::make_decode_args(
      q, key_cache, value_cache, block_table, seq_lens, out, batch, num_q_heads, num_kv_heads,
      head_dim, block_size, max_blocks_per_seq, num_blocks, scale, dtype, num_ctas, workspace,
      workspace_bytes, err_flag, stream);
  a.new_key = new_key;
  a.new_value = new_value;
  a.slot_out = slot_mapping;
  bool empty = false;
  const kvc_status st = kvc::check_decode_args(a, &empty);
  if (st != KVC_OK || empty) return st;
  return kvc::launch_paged_decode(a);
}

kvc_status kvc_paged_decode_window(const void* q, const void* key_cache, const void* value_cache,
                                   const int32_t* block_table, const int32_t* seq_lens, void* out,
                                   int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, int max_blocks_per_seq, int num_blocks,
                                   float scale, int window, kvc_dtype dtype, int num_ctas,
                                   void* workspace, size_t workspace_bytes, uint32_t* err_flag,
                                   kvc_stream_t stream) {
  if (window < 1) return KVC_ERR_INVALID_ARG;
  kvc::DecodeArgs a = kvc::make_decode_args(
      q, key_cache, value_cache, block_table, seq_lens, out, batch, num_q_heads, num_kv_heads,
      head_dim, block_size, max_blocks_per_seq, num_blocks, scale, dtype, num_ctas, workspace,
      workspace_bytes, err_flag, stream);
  a.window = window;
  bool empty = false;
  const kvc_status st = kvc::check_decode_args(a, &empty);
  if (st != KVC_OK || empty) return st;
  return kvc::launch_paged_decode(a);
}

kvc_status kvc_reshape_and_cache_int8(const void* key, const void* value, int8_t* key_codes,
                                      int8_t* value_codes, float* key_scales,
                                      float* value_scales, const int32_t* slot_mapping,
                                      int num_tokens, int num_kv_heads, int head_dim,
                                      int block_size, int num_blocks, kvc_dtype dtype,
                                      uint32_t* err_flag, kvc_stream_t stream) {
  if (dtype != KVC_F16 && dtype != KVC_BF16) return KVC_ERR_INVALID_ARG;
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
    return KVC_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return KVC_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_blocks) * block_size > 0x7fffffffLL) return KVC_ERR_UNSUPPORTED;
  if (num_tokens == 0) return KVC_OK;
  if (!key || !value || !key_codes || !value_codes || !key_scales || !value_scales ||
      !slot_mapping)
    return KVC_ERR_INVALID_ARG;
  if (!aligned16(key) || !aligned16(value) || !aligned16(key_codes) || !aligned16(value_codes) ||
      !aligned16(key_scales) || !aligned16(value_scales))
    return KVC_ERR_INVALID_ARG;
  return kvc::launch_reshape_and_cache_int8(key, value, key_codes, value_codes, key_scales,
                                            value_scales, slot_mapping, num_tokens, num_kv_heads,
                                            head_dim, block_size, num_blocks, dtype, err_flag,
                                            reinterpret_cast<cudaStream_t>(stream));
}

kvc_status kvc_paged_decode_int8(const void* q, const int8_t* key_codes,
                                 const int8_t* value_codes, const float* key_scales,
                                 const float* value_scales, const int32_t* block_table,
                                 const int32_t* seq_lens, void* out, int batch, int num_q_heads,
                                 int num_kv_heads, int head_dim, int block_size,
                                 int max_blocks_per_seq, int num_blocks, float scale,
                                 kvc_dtype dtype, int num_ctas, void* workspace,
                                 size_t workspace_bytes, uint32_t* err_flag,
                                 kvc_stream_t stream) {
  kvc::DecodeArgs a = kvc::make_decode_args(
      q, key_codes, value_codes, block_table, seq_lens, out, batch, num_q_heads, num_kv_heads,
      head_dim, block_size, max_blocks_per_seq, num_blocks, scale, dtype, num_ctas, workspace,
      workspace_bytes, err_flag, stream);
  bool empty = false;
  const kvc_status st = kvc::check_decode_args(a, &empty);
  if (st != KVC_OK || empty) return st;
  if (head_dim != 128) return KVC_ERR_UNSUPPORTED;
  if (!key_scales || !value_scales || !aligned16(key_scales) || !aligned16(value_scales))
    return KVC_ERR_INVALID_ARG;
  a.key_scales = key_scales;
  a.value_scales = value_scales;
  return kvc::launch_paged_decode(a);
}

kvc_status kvc_paged_decode_int8_append(const void* q, const void* new_key,
                                        const void* new_value, int8_t* key_codes,
                                        int8_t* value_codes, float* key_scales,
                                        float* value_scales, const int32_t* block_table,
                                        const int32_t* seq_lens, int32_t* slot_mapping,
                                        void* out, int batch, int num_q_heads, int num_kv_heads,
                                        int head_dim, int block_size, int max_blocks_per_seq,
                                        int num_blocks, float scale, kvc_dtype dtype,
                                        int num_ctas, void* workspace, size_t workspace_bytes,
                                        uint32_t* err_flag, kvc_stream_t stream) {
  if (batch > 0 && (!new_key || !new_value || !aligned16(new_key) || !aligned16(new_value)))
    return KVC_ERR_INVALID_ARG;
  kvc::DecodeArgs a = kvc::make_decode_args(
      q, key_codes, value_codes, block_table, seq_lens, out, batch, num_q_heads, num_kv_heads,
      head_dim, block_size, max_blocks_per_seq, num_blocks, scale, dtype, num_ctas, workspace,
      workspace_bytes, err_flag, stream);
  bool empty = false;
  const kvc_status st = kvc::check_decode_args(a, &empty);
  if (st != KVC_OK || empty) return st;
  if (head_dim != 128) return KVC_ERR_UNSUPPORTED;
  if (!key_scales || !value_scales || !aligned16(key_scales) || !aligned16(value_scales))
    return KVC_ERR_INVALID_ARG;
  a.key_scales = key_scales;
  a.value_scales = value_scales;
  a.new_key = new_key;
  a.new_value = new_value;
  a.slot_out = slot_mapping;
  return kvc::launch_paged_decode(a);
}

namespace {
kvc_status varlen_prefill(const void* q, const void* key, const void* value,
                          const int32_t* cu_seqlens, const int32_t* context_lens,
                          const int32_t* slot_mapping, const int32_t* block_table,
                          void* key_cache, void* value_cache, void* out, int num_seqs,
                          int num_tokens, int max_seqlen_q, int num_q_heads, int num_kv_heads,
                          int head_dim, int block_size, int max_blocks_per_seq, int num_blocks,
                          float scale, int window, kvc_dtype dtype, uint32_t* err_flag,
                          kvc_stream_t stream) {
  if (dtype != KVC_F16 && dtype != KVC_BF16) return KVC_ERR_INVALID_ARG;
  if (num_seqs < 0 || num_tokens < 0 || max_seqlen_q < 0 || num_q_heads <= 0 ||
      num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || max_blocks_per_seq <= 0 ||
      num_blocks <= 0)
    return KVC_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads) return KVC_ERR_INVALID_ARG;
  if (!isfinite(scale)) return KVC_ERR_INVALID_ARG;
  if (head_dim != 64 && head_dim != 128) return KVC_ERR_UNSUPPORTED;
  if (!is_pow2(block_size) || block_size < 8) return KVC_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_blocks) * block_size > 0x7fffffffLL ||
      static_cast<long long>(max_blocks_per_seq) * block_size > 0x7fffffffLL)
    return KVC_ERR_UNSUPPORTED;
  if (num_tokens == 0 || num_seqs == 0) return KVC_OK;
  if (!q || !key || !value || !cu_seqlens || !slot_mapping || !block_table || !key_cache ||
      !value_cache || !out)
    return KVC_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(key) || !aligned16(value) || !aligned16(key_cache) ||
      !aligned16(value_cache) || !aligned16(out))
    return KVC_ERR_INVALID_ARG;
  kvc::PrefillArgs a;
  a.q = q;
  a.key = key;
  a.value = value;
  a.cu_seqlens = cu_seqlens;
  a.context_lens = context_lens;
  a.slot_mapping = slot_mapping;
  a.block_table = block_table;
  a.key_cache = key_cache;
  a.value_cache = value_cache;
  a.out = out;
  a.num_seqs = num_seqs;
  a.num_tokens = num_tokens;
  a.max_seqlen_q = max_seqlen_q;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.scale = scale;
  a.dtype = dtype;
  a.err_flag = err_flag;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  a.window = window;
  return kvc::launch_varlen_prefill(a);
}
}  // namespace

kvc_status kvc_varlen_prefill_paged(const void* q, const void* key, const void* value,
                                    const int32_t* cu_seqlens, const int32_t* context_lens,
                                    const int32_t* slot_mapping, const int32_t* block_table,
                                    void* key_cache, void* value_cache, void* out, int num_seqs,
                                    int num_tokens, int max_seqlen_q, int num_q_heads,
                                    int num_kv_heads, int head_dim, int block_size,
                                    int max_blocks_per_seq, int num_blocks, float scale,
                                    kvc_dtype dtype, uint32_t* err_flag, kvc_stream_t stream) {
  return varlen_prefill(q, key, value, cu_seqlens, context_lens, slot_mapping, block_table,
                        key_cache, value_cache, out, num_seqs, num_tokens, max_seqlen_q,
                        num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                        num_blocks, scale, 0, dtype, err_flag, stream);
}

kvc_status kvc_varlen_prefill_paged_window(
    const void* q, const void* key, const void* value, const int32_t* cu_seqlens,
    const int32_t* context_lens, const int32_t* slot_mapping, const int32_t* block_table,
    void* key_cache, void* value_cache, void* out, int num_seqs, int num_tokens,
    int max_seqlen_q, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
    int max_blocks_per_seq, int num_blocks, float scale, int window, kvc_dtype dtype,
    uint32_t* err_flag, kvc_stream_t stream) {
  if (window < 1) return KVC_ERR_INVALID_ARG;
  return varlen_prefill(q, key, value, cu_seqlens, context_lens, slot_mapping, block_table,
                        key_cache, value_cache, out, num_seqs, num_tokens, max_seqlen_q,
                        num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                        num_blocks, scale, window, dtype, err_flag, stream);
}

size_t kvc_mla_paged_decode_workspace_size(int num_heads, int d_nope, int d_rope, int num_ctas) {
  if (num_heads != 128 || d_nope != 512 || d_rope != 64 || num_ctas < 0) return 0;
  const int ctas = kvc::mla_decode_num_ctas(num_ctas);
  return ctas >= 2 ? kvc::mla_decode_workspace_bytes(ctas) : 0;
}

namespace {
kvc_status mla_decode(const void* q_nope, const void* q_rope, const void* new_nope,
                      const void* new_rope, const void* cache_nope, const void* cache_rope,
                      const int32_t* block_table, const int32_t* seq_lens, int32_t* slot_mapping,
                      void* out, int batch, int num_heads, int d_nope, int d_rope,
                      int block_size, int max_blocks_per_seq, int num_blocks, float scale,
                      kvc_dtype dtype, int num_ctas, void* workspace, size_t workspace_bytes,
                      uint32_t* err_flag, kvc_stream_t stream) {
  if (dtype != KVC_F16 && dtype != KVC_BF16) return KVC_ERR_INVALID_ARG;
  if (batch < 0 || num_heads <= 0 || d_nope <= 0 || block_size <= 0 || max_blocks_per_seq <= 0 ||
      num_blocks <= 0 || num_ctas < 0 || num_ctas == 1)
    return KVC_ERR_INVALID_ARG;
  if (!isfinite(scale)) return KVC_ERR_INVALID_ARG;
  // query_rope and key_rope come together or not at all; rope D must be 64.
  if ((q_rope == nullptr) != (cache_rope == nullptr)) return KVC_ERR_INVALID_ARG;
  if (q_rope == nullptr || d_rope != 64) return KVC_ERR_UNSUPPORTED;
  if (num_heads != 128 || d_nope != 512) return KVC_ERR_UNSUPPORTED;
  if (!is_pow2(block_size) || block_size < 8) return KVC_ERR_UNSUPPORTED;
  if (batch > 1024) return KVC_ERR_UNSUPPORTED;
  if (static_cast<long long>(max_blocks_per_seq) * block_size > 0x7fffffffLL ||
      static_cast<long long>(num_blocks) * block_size > 0x7fffffffLL)
    return KVC_ERR_UNSUPPORTED;
  if (batch == 0) return KVC_OK;
  if (!q_nope || !cache_nope || !block_table || !seq_lens || !out) return KVC_ERR_INVALID_ARG;
  if (!aligned16(q_nope) || !aligned16(q_rope) || !aligned16(cache_nope) ||
      !aligned16(cache_rope) || !aligned16(out) || !aligned16(workspace))
    return KVC_ERR_INVALID_ARG;
  if ((new_nope == nullptr) != (new_rope == nullptr)) return KVC_ERR_INVALID_ARG;
  if (new_nope && (!aligned16(new_nope) || !aligned16(new_rope))) return KVC_ERR_INVALID_ARG;
  kvc::MlaArgs a;
  a.q_nope = q_nope;
  a.q_rope = q_rope;
  a.cache_nope = cache_nope;
  a.cache_rope = cache_rope;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.out = out;
  a.batch = batch;
  a.block_size = block_size;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.scale = scale;
  a.dtype = dtype;
  a.num_ctas = num_ctas;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.err_flag = err_flag;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  a.new_nope = new_nope;
  a.new_rope = new_rope;
  a.slot_out = slot_mapping;
  return kvc::launch_mla_decode(a);
}
}  // namespace

kvc_status kvc_mla_paged_decode(const void* q_nope, const void* q_rope, const void* cache_nope,
                                const void* cache_rope, const int32_t* block_table,
                                const int32_t* seq_lens, void* out, int batch, int num_heads,
                                int d_nope, int d_rope, int block_size, int max_blocks_per_seq,
                                int num_blocks, float scale, kvc_dtype dtype, int num_ctas,
                                void* workspace, size_t workspace_bytes, uint32_t* err_flag,
                                kvc_stream_t stream) {
  return mla_decode(q_nope, q_rope, nullptr, nullptr, cache_nope, cache_rope, block_table,
                    seq_lens, nullptr, out, batch, num_heads, d_nope, d_rope, block_size,
                    max_blocks_per_seq, num_blocks, scale, dtype, num_ctas, workspace,
                    workspace_bytes, err_flag, stream);
}

kvc_status kvc_mla_paged_decode_append(const void* q_nope, const void* q_rope,
                                       const void* new_nope, const void* new_rope,
                                       void* cache_nope, void* cache_rope,
                                       const int32_t* block_table, const int32_t* seq_lens,
                                       int32_t* slot_mapping, void* out, int batch,
                                       int num_heads, int d_nope, int d_rope, int block_size,
                                       int max_blocks_per_seq, int num_blocks, float scale,
                                       kvc_dtype dtype, int num_ctas, void* workspace,
                                       size_t workspace_bytes, uint32_t* err_flag,
                                       kvc_stream_t stream) {
  if (batch > 0 && (!new_nope || !new_rope)) return KVC_ERR_INVALID_ARG;
  return mla_decode(q_nope, q_rope, new_nope, new_rope, cache_nope, cache_rope, block_table,
                    seq_lens, slot_mapping, out, batch, num_heads, d_nope, d_rope, block_size,
                    max_blocks_per_seq, num_blocks, scale, dtype, num_ctas, workspace,
                    workspace_bytes, err_flag, stream);
}

}  // extern "C"
