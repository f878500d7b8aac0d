// kvc_paged_decode_no_alloc: paged decode whose split-KV scratch lives in a
// fixed, library-owned device array instead of a caller-supplied workspace.
//
// Some callers cannot allocate device memory at the point where they run
// decode attention: a host application that hands this library a fixed
// memory budget and forbids further allocations, a serving loop that has
// reserved the whole device for its KV-cache pool, or code whose allocator
// is not reachable from the thread that launches the kernels.  For them this
// entry point takes no workspace argument and allocates nothing: the scratch
// is the file-scope array below, which every GPU that loads the library holds
// until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/kvc.h"
#include "kvc_host.h"

namespace {

// Upper bound of the scratch this entry point can use (8 MiB).
constexpr size_t kScratchBytes = KVC_NO_ALLOC_SCRATCH_BYTES;

// In host code `g_decode_scratch` is only a host-side stand-in for the device
// array: its device address must be fetched with cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up once
// per device (the first call on each device does this).  The address stays
// valid for the life of the device's primary context: after cudaDeviceReset
// the module is loaded again and this cached address is stale, so the entry
// point must not be used after a reset of a device it has run on.
kvc_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KVC_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
      return KVC_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return KVC_OK;
}

}  // namespace

extern "C" kvc_status kvc_paged_decode_no_alloc(
    const void* q, const void* key_cache, const void* value_cache, const int32_t* block_table,
    const int32_t* seq_lens, void* out, int batch, int num_q_heads, int num_kv_heads,
    int head_dim, int block_size, int max_blocks_per_seq, int num_blocks, float scale,
    kvc_dtype dtype, int num_ctas, uint32_t* err_flag, kvc_stream_t stream) {
  // Every argument is checked before anything is enqueued, so a rejected call
  // leaves nothing on the stream (not even the scratch clear below).
  const kvc::DecodeArgs args = kvc::make_decode_args(
      q, key_cache, value_cache, block_table, seq_lens, out, batch, num_q_heads, num_kv_heads,
      head_dim, block_size, max_blocks_per_seq, num_blocks, scale, dtype, num_ctas, nullptr, 0,
      err_flag, stream);
  bool empty = false;
  const kvc_status checked = kvc::check_decode_args(args, &empty);
  if (checked != KVC_OK || empty) return checked;
  const size_t need = kvc_paged_decode_workspace_size(num_q_heads, num_kv_heads, head_dim,
                                                      num_ctas);
  if (need == 0) return KVC_ERR_CUDA;
  if (need > kScratchBytes) return KVC_ERR_WORKSPACE;  // more CTAs or a wider group than fits
  void* scratch = nullptr;
  const kvc_status st = scratch_address(&scratch);
  if (st != KVC_OK) return st;
  // The array keeps whatever the previous call left; the split-KV arrival
  // counters must start at zero, so clear the part this call uses.
  if (cudaMemsetAsync(scratch, 0, need, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return KVC_ERR_CUDA;
  return kvc_paged_decode(q, key_cache, value_cache, block_table, seq_lens, out, batch,
                          num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                          num_blocks, scale, dtype, num_ctas, scratch, kScratchBytes, err_flag,
                          stream);
}
