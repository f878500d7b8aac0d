// kvc_varlen_prefill_paged: the packed chunk's K/V rows are written into the
// paged cache at slot_mapping (ai6s.net KVCache article 4.2: each layer
// writes its cache, then FA reads it -- "external-cannbot-model-model-infer-
// kvcache" 3.6), then every packed token attends causally to its own
// sequence through the cache (prefill_tc2.cu for an even GQA group size --
// two heads per CTA sharing the K/V stream -- else prefill_tc.cu).  Without
// cached context (context_lens null) and with an even group, both steps run
// in one prefill_tc2.cu launch.
#include <cuda_runtime.h>

#include "kvc_device.cuh"
#include "kvc_host.h"

namespace kvc {

kvc_status launch_varlen_prefill(const PrefillArgs& a) {
  const bool even = (a.num_q_heads / a.num_kv_heads) % 2 == 0;
  // A chunk without cached context attends only to its own rows: the write
  // rides in the attention kernel, which reads the rows from the input.
  if (even && a.context_lens == nullptr && a.num_seqs > 0) return launch_prefill_fused_tc2(a);
  // 1. The chunk's own K/V rows go into the cache (bit-exact row copies).
  kvc_status st = launch_reshape_and_cache(a.key, a.value, a.key_cache, a.value_cache,
                                           a.slot_mapping, a.num_tokens, a.num_kv_heads,
                                           a.head_dim, a.head_dim, a.block_size, a.num_blocks,
                                           a.err_flag, a.stream);
  if (st != KVC_OK) return st;
  // 2. Causal attention of every packed token over its sequence's cache.
  if (even) return launch_prefill_attention_tc2(a);
  return launch_prefill_attention_tc(a);
}

}  // namespace kvc
