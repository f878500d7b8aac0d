/*
 * kvc.h -- C ABI of the GB300 (sm_103a) paged KV-cache attention library.
 *
 * The operations restate the problem posed by these pages:
 *   [SKILL] "external-cannbot-model-model-infer-kvcache" (KVCache Optimization
 *           Skill): Mode 2 "Paged attention + FA fused operator", Mode 3 "MLA
 *           compressed cache", 3.1 "Physical Memory Layout and Logical
 *           Mapping", 3.3 "slot_mapping Construction", 3.4
 *           "actual_seq_lengths Construction", Appendix C "sparse_mode".
 *   [ATB]   ai6s.net KVCache article, section 4: cache allocation in the ND
 *           layout [num_blocks, block_size, num_heads, head_size] and the
 *           cache write loop.
 *   [NOTES] hotelren.com notes "Paged KV Cache + Packed Sequence", sections
 *           2.2 (index arithmetic), 3.1-3.3 (seq_offset / cu_seqlens, causal
 *           within a sequence, packed -> paged index chain).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor pointer is a DEVICE pointer to a contiguous row-major
 *   tensor, 16-byte aligned.  The caller owns every buffer (including the
 *   workspace); the library never allocates or frees device memory.
 * - Work is enqueued asynchronously on `stream` (NULL = legacy default
 *   stream); a call returns as soon as its kernels are launched.
 * - The KV cache layout is ND: [num_blocks, block_size, num_kv_heads,
 *   head_dim] ([ATB] section 4.1; [SKILL] 3.1).  block_table is int32
 *   [num_seqs, max_blocks_per_seq] ([SKILL] note 4); position p of sequence
 *   s lives at slot block_table[s][p / block_size] * block_size +
 *   p % block_size ([SKILL] 3.1 Mapping Formula).  Table entries past a
 *   sequence's length are never read.
 * - seq_lens[s] counts the cached tokens a decode attends to, INCLUDING the
 *   token written this step ([SKILL] 3.6: FA reads kv_len + 1).
 * - cu_seqlens has num_seqs + 1 entries with a leading 0 ([NOTES] 3.1
 *   seq_offset).  The pages' TND actual_seq_lengths is cu_seqlens[1:].
 * - q head h uses kv head h / (num_q_heads / num_kv_heads).
 * - `scale` multiplies q.k before the softmax and has no default ([SKILL]
 *   Appendix A warns that a silently defaulted scale of 1.0 corrupts results).
 * - Outputs are rounded to the input dtype with round-to-nearest-even; the
 *   softmax and all accumulation run in fp32.
 * - A sequence with no visible key produces a row of zeros.
 *
 * Errors
 * ------
 * - Bad arguments are rejected on the host before anything is launched:
 *   KVC_ERR_INVALID_ARG (null pointer, bad size, misalignment) or
 *   KVC_ERR_UNSUPPORTED (a legal shape this build does not implement).
 * - KVC_ERR_WORKSPACE: the workspace is smaller than the size query says.
 * - KVC_ERR_CUDA: a launch failed (cudaGetLastError after launch).
 * - KVC_ERR_OUT_OF_BLOCKS: the host block manager has no free block left
 *   (the call changed nothing).
 * - Data errors found on the device never trap.  The kernel skips the bad
 *   access and, if `err_flag` (a device uint32, may be NULL) is given, ORs
 *   one of the KVC_FLAG_* bits into it.  The caller reads it after syncing.
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t; the library's functions only pass it to kernel launches. */
struct CUstream_st;
typedef struct CUstream_st* kvc_stream_t;

typedef enum {
  KVC_OK = 0,
  KVC_ERR_INVALID_ARG = 1,
  KVC_ERR_UNSUPPORTED = 2,
  KVC_ERR_CUDA = 3,
  KVC_ERR_WORKSPACE = 4,
  KVC_ERR_OUT_OF_BLOCKS = 5
} kvc_status;

typedef enum { KVC_F16 = 0, KVC_BF16 = 1 } kvc_dtype;

/* Bits a kernel ORs into *err_flag. */
#define KVC_FLAG_BLOCK_ID_RANGE 0x1u /* block_table entry outside [0, num_blocks)        */
#define KVC_FLAG_SLOT_RANGE     0x2u /* slot >= num_blocks * block_size                   */
#define KVC_FLAG_LEN_RANGE      0x4u /* length < 0 or beyond max_blocks_per_seq*block_size */
#define KVC_FLAG_WAIT_TIMEOUT   0x8u /* a bounded on-chip wait gave up (kernel returned)   */

/* Human-readable name of a status code.  Never NULL. */
const char* kvc_status_string(kvc_status status);

/* Library ABI version (major * 100 + minor). */
int kvc_version(void);

/*
 * kvc_build_slot_mapping -- slot of every token to be written.
 * [SKILL] 3.1 Mapping Formula and 3.3 slot_mapping Construction; [NOTES] 2.2
 * (logical block, slot, flat offset) and 3.3 (packed token -> request ->
 * logical block -> physical block).
 *
 *   cu_seqlens == NULL (decode form): num_tokens == num_seqs; token s is the
 *     new token of sequence s at position start_pos[s] (its current kv_len).
 *   cu_seqlens != NULL (packed form): token t with cu_seqlens[s] <= t <
 *     cu_seqlens[s+1] sits at position start_pos[s] + (t - cu_seqlens[s]).
 *   slot_mapping[t] = block_table[s][p / block_size] * block_size
 *                     + p % block_size                                (int32)
 *
 * block_table: int32 [num_seqs, max_blocks_per_seq]; cu_seqlens: int32
 * [num_seqs + 1] or NULL; start_pos: int32 [num_seqs]; slot_mapping: int32
 * [num_tokens] (output).  A position past the table or a table entry outside
 * [0, num_blocks) yields slot -1 (skipped by the write) and sets
 * KVC_FLAG_LEN_RANGE / KVC_FLAG_BLOCK_ID_RANGE.
 */
kvc_status kvc_build_slot_mapping(const int32_t* block_table, int max_blocks_per_seq,
                                  const int32_t* cu_seqlens, const int32_t* start_pos,
                                  int num_seqs, int num_tokens, int block_size, int num_blocks,
                                  int32_t* slot_mapping, uint32_t* err_flag,
                                  kvc_stream_t stream);

/*
 * kvc_reshape_and_cache -- copy new K/V rows into the paged cache.
 * [ATB] section 4.2 (the KVCache operator copies each request's new rows into
 * the cache unchanged); [SKILL] 3.3 (slot_mapping drives cache writes).
 *
 *   key_cache[slot / block_size][slot % block_size][:][:] = key[t][:][:]
 *   value_cache[...]                                      = value[t][:][:]
 *
 * key: [num_tokens, num_kv_heads, head_dim_k]; value: [num_tokens,
 * num_kv_heads, head_dim_v] or NULL (then value_cache must be NULL too);
 * caches: [num_blocks, block_size, num_kv_heads, head_dim_*].  The copy is
 * bit-exact.  slot_mapping[t] < 0 skips token t; a slot >= num_blocks *
 * block_size is skipped and sets KVC_FLAG_SLOT_RANGE.  Duplicate slots in one
 * call leave the cache row unspecified.  head_dim_k and head_dim_v must be
 * multiples of 8 (16-byte rows); for MLA pass cache_nope as key and
 * cache_rope as value (head_dim_k = 512, head_dim_v = 64, num_kv_heads = 1).
 */
kvc_status kvc_reshape_and_cache(const void* key, const void* value, void* key_cache,
                                 void* value_cache, const int32_t* slot_mapping, int num_tokens,
                                 int num_kv_heads, int head_dim_k, int head_dim_v,
                                 int block_size, int num_blocks, kvc_dtype dtype,
                                 uint32_t* err_flag, kvc_stream_t stream);

/*
 * kvc_copy_blocks -- the copy-on-write copies of the host block manager.
 * [NOTES] 5.2 (sequences that share a prefix share its blocks, counted by
 * reference); a sequence about to write into a shared, partly filled block
 * first gets a private copy of it (kvc_bm_append / kvc_bm_step report the
 * pair: this library's reading, the notes are silent on it).
 *
 *   for each i < num_pairs with src_blocks[i] >= 0:
 *     key_cache block dst_blocks[i]   <- key_cache block src_blocks[i]
 *     value_cache block dst_blocks[i] <- value_cache block src_blocks[i]
 *
 * Whole blocks are copied bit for bit (rows past the shared prefix are
 * rewritten before any read).  src_blocks, dst_blocks: device int32
 * [num_pairs] -- the cow_src / cow_dst arrays of kvc_bm_step, -1 meaning "no
 * copy".  block_bytes_k / block_bytes_v: bytes of one block of each cache
 * (block_size * num_kv_heads * head_dim * element size), multiples of 16;
 * value_cache may be NULL.  Any cache whose blocks are contiguous works (16-bit
 * caches, INT8 codes, scale arrays).  A block id outside [0, num_blocks) skips
 * the pair and sets KVC_FLAG_BLOCK_ID_RANGE.  The pairs of one call must not
 * overlap (no block both a source and a destination).
 */
kvc_status kvc_copy_blocks(void* key_cache, void* value_cache, const int32_t* src_blocks,
                           const int32_t* dst_blocks, int num_pairs, long long block_bytes_k,
                           long long block_bytes_v, int num_blocks, uint32_t* err_flag,
                           kvc_stream_t stream);

/*
 * kvc_rope_cos_sin_table -- the angle table kvc_rmsnorm_rope_cache reads.
 *   cos_sin[p][i] = cos(p * theta_i), cos_sin[p][rope_dim/2 + i] = sin(p * theta_i),
 *   theta_i = base^(-2i / rope_dim), 0 <= p < max_position, 0 <= i < rope_dim / 2.
 * Computed in fp64 on the device and stored as fp32.  cos_sin: device float
 * [max_position, rope_dim], caller-owned; rope_dim even, base > 0.  Built once.
 */
kvc_status kvc_rope_cos_sin_table(float* cos_sin, int max_position, int rope_dim, float base,
                                  kvc_stream_t stream);

/*
 * kvc_rmsnorm_rope_cache -- fused RMSNorm + RoPE + paged cache write.
 * [SKILL] Mode 2 step 3 and Appendix D (a fused write operator, "RMSNorm +
 * RoPE + Cache write", driven by slot_mapping, beside the plain write), Mode 3
 * (the MLA latent stored as a non-positional cache_nope and a positional
 * cache_rope), 3.5 (kv_len drives the RoPE positions); [NOTES] 3.1 (packed
 * position ids restart at 0 per sequence).  The pages fix neither the norm's
 * form nor the RoPE convention; this library's reading:
 *
 *   row = kv[t][h] = [x (d_norm) | y (d_rope)],  p = positions[t]
 *   cache_norm[slot / bs][slot % bs][h] = x / sqrt(mean(x^2) + eps) * gamma
 *   cache_rope[slot / bs][slot % bs][h][2i, 2i+1] = rotation of (y[2i], y[2i+1])
 *       by the angle p * theta_i, read from cos_sin (kvc_rope_cos_sin_table)
 *
 * kv: [num_tokens, num_heads, d_norm + d_rope] (for MLA: the latent row
 * [compressed kv 512 | key rope 64], num_heads 1); gamma: [d_norm] of the
 * same dtype; cos_sin: fp32 [max_position, d_rope]; positions: int32
 * [num_tokens] (decode: seq_lens - 1; packed prefill: context + offset in the
 * sequence); slot_mapping: int32 [num_tokens]; cache_norm: [num_blocks,
 * block_size, num_heads, d_norm]; cache_rope: [num_blocks, block_size,
 * num_heads, d_rope].  fp32 arithmetic, one rounding per stored element.
 * d_norm and d_rope multiples of 8.  slot < 0 skips the token; a slot beyond
 * the pool (KVC_FLAG_SLOT_RANGE) or a position outside [0, max_position)
 * (KVC_FLAG_LEN_RANGE) skips it and sets the flag.
 */
kvc_status kvc_rmsnorm_rope_cache(const void* kv, const void* gamma, float eps,
                                  const float* cos_sin, int max_position,
                                  const int32_t* positions, const int32_t* slot_mapping,
                                  void* cache_norm, void* cache_rope, int num_tokens,
                                  int num_heads, int d_norm, int d_rope, int block_size,
                                  int num_blocks, kvc_dtype dtype, uint32_t* err_flag,
                                  kvc_stream_t stream);

/*
 * Bytes of workspace kvc_paged_decode needs for this head shape when it runs
 * with `num_ctas` persistent CTAs (0 = the automatic choice for the current
 * device: SM count x resident CTAs per SM).  Independent of batch and lengths.
 * The same size serves the band, appending and INT8 decode calls of this
 * shape (with num_ctas 0 it covers the largest of their automatic choices);
 * kvc_paged_decode_no_alloc checks its own scratch against it.
 */
size_t kvc_paged_decode_workspace_size(int num_q_heads, int num_kv_heads, int head_dim,
                                       int num_ctas);

/*
 * kvc_paged_decode -- one query token per sequence against the paged cache.
 * [SKILL] Mode 2 (FA with block_table, block_size, actual_seq_kvlen,
 * num_query_heads / num_key_value_heads) with sparse_mode 0 (no mask,
 * Appendix C); [NOTES] 4.2 (the kernel walks the physical blocks of its
 * sequence).
 *
 *   out[b][h][:] = sum_{j < seq_lens[b]} softmax_j(scale * q[b][h] . K_b[j][g])
 *                  V_b[j][g],   g = h / (num_q_heads / num_kv_heads),
 *   K_b[j] = key_cache[block_table[b][j / block_size]][j % block_size].
 *
 * q, out: [batch, num_q_heads, head_dim]; caches: [num_blocks, block_size,
 * num_kv_heads, head_dim]; block_table: int32 [batch, max_blocks_per_seq];
 * seq_lens: int32 [batch].
 * Supported: head_dim 64 or 128; num_q_heads / num_kv_heads <= 16; block_size
 * a power of two >= 8; batch <= 1024.
 * Long sequences are split across CTAs (split-KV); the partial softmax states
 * go to `workspace` (device, >= kvc_paged_decode_workspace_size bytes) and
 * the CTA that finishes a split sequence last merges them, inside the same
 * kernel.  The workspace must be zero-filled before its first use (for
 * example cudaMemsetAsync); every call leaves it zero-filled again, so it can
 * be reused without clearing.  After a call that raised
 * KVC_FLAG_WAIT_TIMEOUT, zero it again.  Calls that overlap on the GPU must
 * not share a workspace.  num_ctas = 0 picks
 * the device's resident capacity; any positive value is valid (tests use it
 * to force 1..many splits).  Results do not depend on the physical block IDs
 * and are bitwise reproducible for a fixed num_ctas.
 */
kvc_status kvc_paged_decode(const void* q, const void* key_cache, const void* value_cache,
                            const int32_t* block_table, const int32_t* seq_lens, void* out,
                            int batch, int num_q_heads, int num_kv_heads, int head_dim,
                            int block_size, int max_blocks_per_seq, int num_blocks, float scale,
                            kvc_dtype dtype, int num_ctas, void* workspace,
                            size_t workspace_bytes, uint32_t* err_flag, kvc_stream_t stream);

/*
 * kvc_paged_decode_window -- kvc_paged_decode restricted to a band: each
 * sequence attends to its last `window` cached tokens only.
 * [SKILL] Appendix C, sparse_mode 4 (band attention, named for sliding-window
 * models together with pre_tokens); ai6s.net KVCache article, section 3 item
 * 4 (a sliding window keeps only the most recent N tokens).  Neither fixes the
 * band's edges; this library's reading: the band ends at the query's own
 * position and holds `window` positions.
 *
 *   lo = max(0, seq_lens[b] - window)
 *   out[b][h][:] = sum_{lo <= j < seq_lens[b]} softmax_j(scale * q[b][h] . K_b[j][g]) V_b[j][g]
 *
 * window >= 1 (else KVC_ERR_INVALID_ARG); a window of at least seq_lens[b]
 * gives kvc_paged_decode's result, bit for bit.  Every other argument, the
 * workspace rules and the errors are those of kvc_paged_decode.  Blocks that
 * lie wholly before the band are never read (their table entries are not
 * looked up either).
 */
kvc_status kvc_paged_decode_window(const void* q, const void* key_cache, const void* value_cache,
                                   const int32_t* block_table, const int32_t* seq_lens, void* out,
                                   int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, int max_blocks_per_seq, int num_blocks,
                                   float scale, int window, kvc_dtype dtype, int num_ctas,
                                   void* workspace, size_t workspace_bytes, uint32_t* err_flag,
                                   kvc_stream_t stream);

/*
 * kvc_reshape_and_cache_int8 -- the cache write of an INT8 KV cache.
 * [ATB] section 4.2 (new rows go to their cache position) with the rows
 * quantised as [SKILL] 4 (quantized KV: codes plus antiquant / dequant
 * scales) and the article's section 3 (FP16 -> INT8 halves the bytes per
 * element) imply.  The pages fix no scheme; this library's reading: one
 * symmetric fp32 scale per written row (token, kv head), so a decode write
 * never re-quantises earlier tokens, decided in IEEE fp32:
 *
 *   amax = max_d |x[d]|;  inv = 127 / amax;  scale = amax / 127
 *   code[d] = clamp(round_half_even(x[d] * inv), -127, 127)
 *   (a row of zeros: scale 0, codes 0; both divisions and the product are
 *    single fp32 operations rounded to nearest)
 *   key_codes[slot / bs][slot % bs][h][:] = code;  key_scales[slot / bs][h][slot % bs] = scale
 *   (the same for value)
 *
 * key, value: [num_tokens, num_kv_heads, head_dim] fp16/bf16; key_codes,
 * value_codes: int8 [num_blocks, block_size, num_kv_heads, head_dim] (the
 * 16-bit cache's layout); key_scales, value_scales: fp32 [num_blocks,
 * num_kv_heads, block_size] (head-major inside a block, so one head's scales
 * of consecutive tokens are contiguous).  slot_mapping as for
 * kvc_reshape_and_cache (negative: skip; out of range: skip and
 * KVC_FLAG_SLOT_RANGE).  head_dim 64 or 128.
 */
kvc_status kvc_reshape_and_cache_int8(const void* key, const void* value, int8_t* key_codes,
                                      int8_t* value_codes, float* key_scales,
                                      float* value_scales, const int32_t* slot_mapping,
                                      int num_tokens, int num_kv_heads, int head_dim,
                                      int block_size, int num_blocks, kvc_dtype dtype,
                                      uint32_t* err_flag, kvc_stream_t stream);

/*
 * kvc_paged_decode_int8 -- kvc_paged_decode over an INT8 KV cache written by
 * kvc_reshape_and_cache_int8: every cached row is code * scale.
 * [SKILL] Mode 2 and 4 (FA over a quantized KV cache with its dequantisation
 * scales); ai6s.net KVCache article section 3 (INT8 halves the bytes).
 *
 *   out[b][h][:] = sum_{j < seq_lens[b]} softmax_j(scale * q[b][h] . Kd_b[j][g]) Vd_b[j][g]
 *   Kd_b[j][g][d] = key_codes[blk][off][g][d] * key_scales[blk][g][off]
 *   (blk = block_table[b][j / block_size], off = j % block_size; V alike)
 *
 * q, out: fp16/bf16 [batch, num_q_heads, 128] (`dtype`); the kernel reads the
 * codes and scales (about half the bytes of a 16-bit cache).  Its products
 * run on fp16 tensor-core operands with fp32 accumulation: the codes are
 * exact in fp16, bf16 queries are converted to fp16 (exact within fp16's
 * normal range), the scores are scaled in fp32, and the softmax weights
 * times the value scales are rounded to fp16 for the value product (the row
 * sums use the unrounded weights).  head_dim 128 only (KVC_ERR_UNSUPPORTED
 * otherwise); every other argument, the workspace (same size query) and the
 * errors are those of kvc_paged_decode.
 */
kvc_status kvc_paged_decode_int8(const void* q, const int8_t* key_codes,
                                 const int8_t* value_codes, const float* key_scales,
                                 const float* value_scales, const int32_t* block_table,
                                 const int32_t* seq_lens, void* out, int batch, int num_q_heads,
                                 int num_kv_heads, int head_dim, int block_size,
                                 int max_blocks_per_seq, int num_blocks, float scale,
                                 kvc_dtype dtype, int num_ctas, void* workspace,
                                 size_t workspace_bytes, uint32_t* err_flag,
                                 kvc_stream_t stream);

/*
 * kvc_paged_decode_int8_append -- one decode step over an INT8 cache in one
 * launch: identical in effect to kvc_build_slot_mapping (start_pos =
 * seq_lens - 1) + kvc_reshape_and_cache_int8 + kvc_paged_decode_int8 for every
 * sequence with seq_lens[b] >= 1.  [SKILL] 3.6 (the cache write before the
 * attention that reads it) and Mode 2 / 4 with the quantized cache of
 * Appendix A; not a separate operation on the pages: it exists so an INT8
 * decode step costs one launch.
 *
 *   p = seq_lens[b] - 1; slot = block_table[b][p / block_size] * block_size
 *   + p % block_size; the rows new_key[b][g] / new_value[b][g] are quantised
 *   exactly as kvc_reshape_and_cache_int8 does (codes into key_codes /
 *   value_codes at `slot`, scales into key_scales / value_scales);
 *   slot_mapping[b] = slot (or -1 when seq_lens[b] == 0: nothing is written);
 *   out = kvc_paged_decode_int8 over the updated cache.
 *
 * new_key, new_value: [batch, num_kv_heads, 128] in `dtype` (device, 16-byte
 * aligned); slot_mapping: int32 [batch] output, may be NULL; every other
 * argument, the workspace rules and the errors are those of
 * kvc_paged_decode_int8.  Each new row is written by the CTA that then reads
 * it, before it reads it.  A block_table entry outside [0, num_blocks) sets
 * KVC_FLAG_BLOCK_ID_RANGE and that row is not written.
 */
kvc_status kvc_paged_decode_int8_append(const void* q, const void* new_key,
                                        const void* new_value, int8_t* key_codes,
                                        int8_t* value_codes, float* key_scales,
                                        float* value_scales, const int32_t* block_table,
                                        const int32_t* seq_lens, int32_t* slot_mapping,
                                        void* out, int batch, int num_q_heads, int num_kv_heads,
                                        int head_dim, int block_size, int max_blocks_per_seq,
                                        int num_blocks, float scale, kvc_dtype dtype,
                                        int num_ctas, void* workspace, size_t workspace_bytes,
                                        uint32_t* err_flag, kvc_stream_t stream);

/*
 * kvc_paged_decode_append -- one decode step in one launch: the slot mapping,
 * the cache write of the new token and the paged decode with split-KV,
 * fused.  Identical in effect to kvc_build_slot_mapping (start_pos =
 * seq_lens - 1) + kvc_reshape_and_cache + kvc_paged_decode for every sequence
 * with seq_lens[b] >= 1: the pages describe the cache write before the
 * attention that reads it ([SKILL] 3.6, [ATB] 4.2).  Not a separate operation
 * on the pages; it exists so a decode step costs one launch.
 *
 *   p = seq_lens[b] - 1 (seq_lens includes the new token);
 *   slot = block_table[b][p / block_size] * block_size + p % block_size;
 *   key_cache / value_cache row `slot` (all kv heads) <- new_key[b] / new_value[b];
 *   slot_mapping[b] = slot (or -1 when seq_lens[b] == 0: nothing is written);
 *   out = kvc_paged_decode over the updated cache.
 *
 * new_key, new_value: [batch, num_kv_heads, head_dim] (device, 16-byte
 * aligned); slot_mapping: int32 [batch] output, may be NULL; every other
 * argument, the workspace rules and the errors are those of kvc_paged_decode.
 * The row of the new token is written by the CTA that then reads it, before it
 * reads it, so no other ordering is needed.  A block_table entry outside
 * [0, num_blocks) sets KVC_FLAG_BLOCK_ID_RANGE and that row is not written.
 */
kvc_status kvc_paged_decode_append(const void* q, const void* new_key, const void* new_value,
                                   void* key_cache, void* value_cache, const int32_t* block_table,
                                   const int32_t* seq_lens, int32_t* slot_mapping, void* out,
                                   int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, int max_blocks_per_seq, int num_blocks,
                                   float scale, kvc_dtype dtype, int num_ctas, void* workspace,
                                   size_t workspace_bytes, uint32_t* err_flag,
                                   kvc_stream_t stream);

/*
 * kvc_varlen_prefill_paged -- packed variable-length causal prefill that
 * writes its own K/V into the paged cache and attends through it.
 * [NOTES] 3.1 (cu_seqlens / seq_offset, per-sequence positions), 3.2 (causal
 * within a sequence only), 3.3 (packed token -> request and offset ->
 * logical block -> physical block); [SKILL] 3.6 (each layer writes its cache,
 * then FA reads it) and Appendix C (sparse_mode 3, causal); [ATB] 4.2 (the
 * cache write).
 *
 *   sequence s owns packed tokens cu_seqlens[s] .. cu_seqlens[s+1]-1; token i
 *   of it sits at position p = context_lens[s] + i.
 *   1. key[t], value[t] are copied to their caches at slot_mapping[t] (as
 *      kvc_reshape_and_cache; slot_mapping as kvc_build_slot_mapping's packed
 *      form with start_pos = context_lens).
 *   2. out[t][h] = sum_{j <= p} softmax_j(scale * q[t][h] . K_s[j][g]) V_s[j][g]
 *      over positions 0..p of sequence s only (the diagonal included),
 *      K_s/V_s read through block_table[s]; g = h / (num_q_heads/num_kv_heads).
 *
 * q, out: [num_tokens, num_q_heads, head_dim]; key, value: [num_tokens,
 * num_kv_heads, head_dim]; cu_seqlens: int32 [num_seqs + 1] (leading 0);
 * context_lens: int32 [num_seqs] cached tokens before this chunk, or NULL for
 * none; slot_mapping: int32 [num_tokens]; block_table: int32 [num_seqs,
 * max_blocks_per_seq]; caches: [num_blocks, block_size, num_kv_heads,
 * head_dim].  max_seqlen_q is informational (the longest chunk).
 * Supported: head_dim 64 or 128; block_size a power of two >= 8.  A sequence
 * whose context_lens + length exceeds max_blocks_per_seq * block_size gets
 * no output and sets KVC_FLAG_LEN_RANGE.
 * With context_lens NULL and an even group size the two steps run in one
 * launch: the attention takes K_s/V_s straight from key/value (the rows step 1
 * copies into the cache, since slot_mapping is the packed form over
 * block_table) while the same kernel writes them at slot_mapping; the cache
 * and the output are those of the two steps in sequence.
 */
kvc_status kvc_varlen_prefill_paged(const void* q, const void* key, const void* value,
                                    const int32_t* cu_seqlens, const int32_t* context_lens,
                                    const int32_t* slot_mapping, const int32_t* block_table,
                                    void* key_cache, void* value_cache, void* out, int num_seqs,
                                    int num_tokens, int max_seqlen_q, int num_q_heads,
                                    int num_kv_heads, int head_dim, int block_size,
                                    int max_blocks_per_seq, int num_blocks, float scale,
                                    kvc_dtype dtype, uint32_t* err_flag, kvc_stream_t stream);

/*
 * kvc_varlen_prefill_paged_window -- kvc_varlen_prefill_paged with band
 * attention: each query sees only the last `window` positions up to its own.
 * [SKILL] Appendix C, sparse_mode 4 (band, for sliding-window models with
 * pre_tokens); ai6s.net KVCache article section 3 item 4 (keep the most recent
 * N tokens).  The band's edges are this library's reading: it ends at the
 * query's own position and holds `window` positions.
 *
 *   token i of sequence s at position p = context_lens[s] + i:
 *   out[t][h] = sum_{max(0, p - window + 1) <= j <= p}
 *                 softmax_j(scale * q[t][h] . K_s[j][g]) V_s[j][g]
 *
 * window >= 1 (else KVC_ERR_INVALID_ARG); window >= p + 1 for every query
 * gives kvc_varlen_prefill_paged's result.  The cache write and every other
 * argument and error are those of kvc_varlen_prefill_paged.  Key tiles that
 * lie wholly before the band of a query tile are not read.
 */
kvc_status kvc_varlen_prefill_paged_window(
    const void* q, const void* key, const void* value, const int32_t* cu_seqlens,
    const int32_t* context_lens, const int32_t* slot_mapping, const int32_t* block_table,
    void* key_cache, void* value_cache, void* out, int num_seqs, int num_tokens,
    int max_seqlen_q, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
    int max_blocks_per_seq, int num_blocks, float scale, int window, kvc_dtype dtype,
    uint32_t* err_flag, kvc_stream_t stream);

/*
 * Bytes of workspace kvc_mla_paged_decode needs with `num_ctas` CTAs (0 = as
 * many CTA pairs as the current device holds resident at once, at most one
 * CTA per SM; an odd count is rounded down to pairs).
 * Returns 0 for an unsupported shape.
 */
size_t kvc_mla_paged_decode_workspace_size(int num_heads, int d_nope, int d_rope, int num_ctas);

/*
 * kvc_mla_paged_decode -- MLA (absorbed) decode over the latent paged cache.
 * [SKILL] Mode 3: the cache stores cache_nope (kv_lora_rank wide) and
 * cache_rope (qk_rope_head_dim wide) per token; FA takes key = value =
 * cache_nope and query_rope / key_rope separately; query_rope and key_rope
 * come together or not at all, rope D must be 64, query D 512.  Paging as in
 * Mode 2.
 *
 *   s_j    = scale * (q_nope[b][h] . nope_j + q_rope[b][h] . rope_j)
 *   out[b][h] = sum_{j < seq_lens[b]} softmax_j(s) nope_j
 *   nope_j = cache_nope[block_table[b][j / block_size]][j % block_size][0]
 *
 * q_nope: [batch, 128, 512]; q_rope: [batch, 128, 64]; cache_nope:
 * [num_blocks, block_size, 1, 512]; cache_rope: [num_blocks, block_size, 1,
 * 64]; out: [batch, 128, 512]; block_table int32 [batch, max_blocks_per_seq];
 * seq_lens int32 [batch].  Supported: num_heads 128, d_nope 512, d_rope 64,
 * block_size a power of two >= 8, batch <= 1024; fp16 or bf16.
 * Runs on CTA pairs (thread-block clusters of 2); long sequences are split
 * over the pairs, and a second kernel on the same stream merges the pieces.
 * workspace: device, >= kvc_mla_paged_decode_workspace_size bytes, needs no
 * initialisation; calls that overlap on the GPU must not share it.
 */
kvc_status kvc_mla_paged_decode(const void* q_nope, const void* q_rope, const void* cache_nope,
                                const void* cache_rope, const int32_t* block_table,
                                const int32_t* seq_lens, void* out, int batch, int num_heads,
                                int d_nope, int d_rope, int block_size, int max_blocks_per_seq,
                                int num_blocks, float scale, kvc_dtype dtype, int num_ctas,
                                void* workspace, size_t workspace_bytes, uint32_t* err_flag,
                                kvc_stream_t stream);

/*
 * kvc_mla_paged_decode_append -- one MLA decode step in one call: the latent
 * row of each sequence's new token is written into the cache, then attended.
 * Identical in effect to kvc_build_slot_mapping (start_pos = seq_lens - 1) +
 * kvc_reshape_and_cache (cache_nope as key, cache_rope as value) +
 * kvc_mla_paged_decode for every sequence with seq_lens[b] >= 1: [SKILL] 3.6
 * and [ATB] 4.2 put the cache write before the attention that reads it;
 * Mode 3 stores the latent as cache_nope + cache_rope.
 *
 *   p = seq_lens[b] - 1;  slot = block_table[b][p / block_size] * block_size
 *                                + p % block_size;
 *   cache_nope row `slot` <- new_nope[b];  cache_rope row `slot` <- new_rope[b];
 *   slot_mapping[b] = slot (or -1 when seq_lens[b] == 0: nothing is written);
 *   out = kvc_mla_paged_decode over the updated caches.
 *
 * new_nope: [batch, 512], new_rope: [batch, 64] (device, 16-byte aligned);
 * slot_mapping: int32 [batch] output, may be NULL; every other argument, the
 * workspace and the errors are those of kvc_mla_paged_decode.  Each CTA
 * writes the columns of the new row that it then reads, before it reads
 * them, so no other ordering is needed.  A block_table entry outside
 * [0, num_blocks) sets KVC_FLAG_BLOCK_ID_RANGE and that row is not written.
 */
kvc_status kvc_mla_paged_decode_append(const void* q_nope, const void* q_rope,
                                       const void* new_nope, const void* new_rope,
                                       void* cache_nope, void* cache_rope,
                                       const int32_t* block_table, const int32_t* seq_lens,
                                       int32_t* slot_mapping, void* out, int batch,
                                       int num_heads, int d_nope, int d_rope, int block_size,
                                       int max_blocks_per_seq, int num_blocks, float scale,
                                       kvc_dtype dtype, int num_ctas, void* workspace,
                                       size_t workspace_bytes, uint32_t* err_flag,
                                       kvc_stream_t stream);

/*
 * kvc_paged_decode_no_alloc -- kvc_paged_decode for callers that cannot
 * allocate device memory.  The source pages have no counterpart to this entry
 * point; it exists for callers such as a host application that gives this
 * library a fixed memory budget and forbids later allocations, a serving loop
 * that has already reserved the whole device for its KV-cache pool, or code
 * that launches kernels from a thread where no device allocator is
 * available.  They cannot provide the split-KV workspace kvc_paged_decode
 * asks for.
 *
 * Arguments and results are those of kvc_paged_decode without `workspace` and
 * `workspace_bytes`.  The scratch is a library-owned device array of
 * KVC_NO_ALLOC_SCRATCH_BYTES (8 MiB) that every GPU which loads the library
 * holds until the process exits; nothing is allocated or freed (no cudaMalloc,
 * no cudaFree, no allocating library call).  If the shape needs more scratch
 * than that (kvc_paged_decode_workspace_size(...) > 8 MiB: too many CTAs or
 * too wide a query group), the call returns KVC_ERR_WORKSPACE and launches
 * nothing.
 *
 * The first call on each device looks up the array's device address once
 * (cudaGetSymbolAddress); make that first call before any stream capture on
 * that device.  Each call first clears, on `stream`, the part of the array it
 * uses (the array keeps the previous call's contents), then runs the decode.
 * All calls on a device share the one array: calls that overlap on the GPU
 * (for example on two streams) race, so the caller must serialise them.
 * Every argument is checked before the clear, so a rejected call enqueues
 * nothing.  The looked-up address belongs to the device's primary context:
 * after cudaDeviceReset on a device this entry point has run on, it must not
 * be called there again in the same process.
 */
#define KVC_NO_ALLOC_SCRATCH_BYTES (8u << 20)
kvc_status kvc_paged_decode_no_alloc(const void* q, const void* key_cache,
                                     const void* value_cache, const int32_t* block_table,
                                     const int32_t* seq_lens, void* out, int batch,
                                     int num_q_heads, int num_kv_heads, int head_dim,
                                     int block_size, int max_blocks_per_seq, int num_blocks,
                                     float scale, kvc_dtype dtype, int num_ctas,
                                     uint32_t* err_flag, kvc_stream_t stream);

/* ---------------------------------------------------------------------------
 * Host block manager: the allocator of the cache pool's physical blocks.
 *
 * What it follows: the hotelren.com notes "Paged KV Cache + Packed Sequence"
 * 2.1 (fixed-size physical blocks taken from a free list, a reference count
 * per block, per sequence its physical blocks in logical order), 2.2 (a decode
 * step allocates a block only when the token it writes opens one; the token's
 * slot is block * block_size + position % block_size) and 5.2 (sequences that
 * share a prefix share its blocks; a block returns to the free list only when
 * its count reaches 0).  Where the notes are silent: appending into a shared,
 * partly filled last block first gives the sequence a private copy of it.
 *
 * Host memory only: no call here touches the GPU.  One manager is used by one
 * thread at a time.  A sequence is an int64 id; its length counts the tokens
 * that have slots.  Blocks are taken from the end of the free list (initially
 * 0 .. num_blocks-1) and returned to its end.  Every call either succeeds or
 * changes nothing.  The tables it produces are the `block_table` / `seq_lens`
 * arguments of the attention calls above (copied to the device by the caller).
 */
typedef struct kvc_block_manager kvc_block_manager;

/* A manager of blocks 0 .. num_blocks-1 holding block_size tokens each; one
 * sequence holds at most max_blocks_per_seq blocks.  *out receives the handle,
 * which the caller owns and releases with kvc_bm_destroy.  KVC_ERR_INVALID_ARG
 * for a non-positive size, num_blocks * block_size above INT32_MAX, or NULL out. */
kvc_status kvc_bm_create(int num_blocks, int block_size, int max_blocks_per_seq,
                         kvc_block_manager** out);
/* Releases the manager (NULL: nothing happens). */
void kvc_bm_destroy(kvc_block_manager* bm);

/* Blocks on the free list (-1 for NULL bm). */
int kvc_bm_num_free(const kvc_block_manager* bm);
/* Reference count of `block` (-1 if it is outside the pool). */
int kvc_bm_ref_count(const kvc_block_manager* bm, int block);
/* Length of sequence seq_id in tokens (-1 if there is no such sequence). */
int kvc_bm_seq_len(const kvc_block_manager* bm, int64_t seq_id);

/* A new sequence of num_tokens (>= 0) tokens, e.g. a prompt: it gets
 * ceil(num_tokens / block_size) blocks with count 1.  slot_mapping (host,
 * num_tokens int32, may be NULL) receives the slots of tokens 0 .. num_tokens-1,
 * for the prompt's cache write.  KVC_ERR_INVALID_ARG: seq_id exists,
 * num_tokens < 0, or more than max_blocks_per_seq blocks would be needed.
 * KVC_ERR_OUT_OF_BLOCKS: fewer free blocks than needed. */
kvc_status kvc_bm_add(kvc_block_manager* bm, int64_t seq_id, int num_tokens,
                      int32_t* slot_mapping);

/* A new sequence `child` sharing every block of `parent` (each count + 1) and
 * its length: a shared prefix, as in beam search or parallel sampling.
 * KVC_ERR_INVALID_ARG: parent unknown, child exists, or parent == child. */
kvc_status kvc_bm_fork(kvc_block_manager* bm, int64_t parent, int64_t child);

/* Room for one more token at position p = the sequence's length, which then
 * grows by one; *slot (required) receives the token's slot.  If p is a
 * multiple of block_size, a free block is appended to the sequence.  Otherwise
 * the token goes into the sequence's last block; if that block is shared
 * (count > 1) a free block replaces it in this sequence first (the shared
 * block loses one count), and *cow_src / *cow_dst receive the shared and the
 * new block: the caller copies rows 0 .. p % block_size - 1 of block cow_src to
 * block cow_dst in each cache before writing the token.  Otherwise both are -1
 * (each may be NULL).  KVC_ERR_INVALID_ARG: unknown sequence, NULL slot, or a
 * new block beyond max_blocks_per_seq.  KVC_ERR_OUT_OF_BLOCKS: no free block. */
kvc_status kvc_bm_append(kvc_block_manager* bm, int64_t seq_id, int32_t* slot,
                         int32_t* cow_src, int32_t* cow_dst);

/* Ends sequence seq_id: each of its blocks loses one count, and a block whose
 * count reaches 0 returns to the free list.  KVC_ERR_INVALID_ARG: unknown id. */
kvc_status kvc_bm_free(kvc_block_manager* bm, int64_t seq_id);

/* Row i of block_table (host int32 [n][max_blocks_per_seq]) receives the blocks
 * of sequence seq_ids[i] in logical order, then `pad` in the unused entries;
 * seq_lens (host int32 [n], may be NULL) receives the lengths.
 * KVC_ERR_INVALID_ARG: an unknown id, n < 0, or a NULL array for n > 0
 * (nothing is written). */
kvc_status kvc_bm_tables(const kvc_block_manager* bm, const int64_t* seq_ids, int n,
                         int32_t pad, int32_t* block_table, int32_t* seq_lens);

/* One decode step of a serving loop in one call: for each of the n distinct
 * sequences seq_ids[i], the effect of kvc_bm_append (slots[i], cow_src[i],
 * cow_dst[i] receive its results; all three arrays are host int32 [n] and
 * required), then, if block_table is not NULL, the effect of kvc_bm_tables
 * on the same ids (block_table [n][max_blocks_per_seq], seq_lens [n] may be
 * NULL; without block_table, seq_lens alone may still be filled).  The step
 * happens for every sequence or for none: KVC_ERR_INVALID_ARG for an unknown
 * or repeated id or a table that would overflow, KVC_ERR_OUT_OF_BLOCKS if the
 * new blocks and copies need more free blocks than there are (counting that a
 * shared block stops needing a copy once its other holders have moved away in
 * the same step). */
kvc_status kvc_bm_step(kvc_block_manager* bm, const int64_t* seq_ids, int n, int32_t pad,
                       int32_t* slots, int32_t* cow_src, int32_t* cow_dst,
                       int32_t* block_table, int32_t* seq_lens);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H */
