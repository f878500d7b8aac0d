// Fused RMSNorm + RoPE + paged cache write, and the RoPE angle table it reads.
//
// What it computes: "external-cannbot-model-model-infer-kvcache" Mode 2 step 3
// and Appendix D name a fused write operator -- RMSNorm, RoPE and the cache
// write in one, driven by slot_mapping -- beside the plain cache write; Mode 3
// stores the MLA latent as a non-positional part (cache_nope) and a positional
// part (cache_rope); 3.5 has kv_len drive the RoPE positions, and the
// hotelren.com notes 3.1 restart packed position ids at 0 for every sequence.
// The pages fix neither the norm's form nor the RoPE convention.  This
// library's reading: a row [norm part (d_norm) | rope part (d_rope)] is split;
// the norm part becomes x / sqrt(mean(x^2) + eps) * gamma and goes to
// cache_norm, the rope part is rotated pairwise -- (x[2i], x[2i+1]) by the
// angle pos * theta_i, theta_i = base^(-2i / d_rope) -- and goes to
// cache_rope, both at the row's slot.
//
// One warp per (token, head) row: 16-byte loads and stores of 8 elements,
// fp32 arithmetic, one rounding to the cache type per element.  The angles
// come from a table of cos / sin built once (fp64 arithmetic, stored fp32).
#include <cuda_runtime.h>

#include <type_traits>

#include "kvc_device.cuh"
#include "kvc_host.h"

namespace kvc {

namespace {

// table[p][i] = cos(p * theta_i), table[p][half + i] = sin(p * theta_i).
__global__ void rope_table_kernel(float* __restrict__ table, int max_position, int rope_dim,
                                  double base) {
  const int half = rope_dim / 2;
  const long long n = static_cast<long long>(max_position) * half;
  for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < n;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int p = static_cast<int>(e / half), i = static_cast<int>(e - static_cast<long long>(p) * half);
    const double theta = pow(base, -2.0 * i / rope_dim);
    double s, c;
    sincos(static_cast<double>(p) * theta, &s, &c);
    table[static_cast<long long>(p) * rope_dim + i] = static_cast<float>(c);
    table[static_cast<long long>(p) * rope_dim + half + i] = static_cast<float>(s);
  }
}

template <typename T>
__device__ __forceinline__ void unpack8(uint4 u, float (&f)[8]) {
  const T* v = reinterpret_cast<const T*>(&u);
#pragma unroll
  for (int e = 0; e < 8; ++e) f[e] = static_cast<float>(v[e]);
}

template <typename T>
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint4 u;
  float a, b;
  u.x = Pack<T>::run(f[0], f[1], a, b);
  u.y = Pack<T>::run(f[2], f[3], a, b);
  u.z = Pack<T>::run(f[4], f[5], a, b);
  u.w = Pack<T>::run(f[6], f[7], a, b);
  return u;
}

template <typename T>
__global__ void rmsnorm_rope_cache_kernel(const T* __restrict__ kv, const T* __restrict__ gamma,
                                          float eps, const float* __restrict__ cos_sin,
                                          int max_position, const int32_t* __restrict__ positions,
                                          const int32_t* __restrict__ slot_mapping,
                                          T* __restrict__ cache_norm, T* __restrict__ cache_rope,
                                          int num_tokens, int num_heads, int d_norm, int d_rope,
                                          long long num_slots, uint32_t* err_flag) {
  const int lane = threadIdx.x & 31;
  const long long w0 = (blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x) >> 5;
  const long long nw = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const long long rows = static_cast<long long>(num_tokens) * num_heads;
  const int width = d_norm + d_rope;
  const int nchunks = d_norm / 8, half = d_rope / 2;
  for (long long r = w0; r < rows; r += nw) {
    const int t = static_cast<int>(r / num_heads);
    const int h = static_cast<int>(r - static_cast<long long>(t) * num_heads);
    const int32_t slot = slot_mapping[t];
    if (slot < 0) continue;
    const int pos = positions[t];
    if (slot >= num_slots || pos < 0 || pos >= max_position) {
      if (lane == 0 && h == 0)
        set_flag(err_flag, slot >= num_slots ? KVC_FLAG_SLOT_RANGE : KVC_FLAG_LEN_RANGE);
      continue;
    }
    const T* src = kv + r * width;
    // Norm part: mean square over d_norm (each lane sums its 8-element chunks),
    // then x * rsqrt * gamma.  The chunks are read twice; the row is in L1.
    float ss = 0.f;
    for (int c = lane; c < nchunks; c += 32) {
      float f[8];
      unpack8<T>(__ldg(reinterpret_cast<const uint4*>(src) + c), f);
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float inv_rms = 1.f / sqrtf(ss / static_cast<float>(d_norm) + eps);
    T* dn = cache_norm + (static_cast<long long>(slot) * num_heads + h) * d_norm;
    for (int c = lane; c < nchunks; c += 32) {
      float f[8], g[8];
      unpack8<T>(__ldg(reinterpret_cast<const uint4*>(src) + c), f);
      unpack8<T>(__ldg(reinterpret_cast<const uint4*>(gamma) + c), g);
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = f[e] * inv_rms * g[e];
      reinterpret_cast<uint4*>(dn)[c] = pack8<T>(f);
    }
    // Rope part: lane i rotates pair i (and i + 32, ...).
    const float* cs = cos_sin + static_cast<long long>(pos) * d_rope;
    T* dr = cache_rope + (static_cast<long long>(slot) * num_heads + h) * d_rope;
    const T* xr = src + d_norm;
    for (int i = lane; i < half; i += 32) {
      const float a = static_cast<float>(xr[2 * i]), b = static_cast<float>(xr[2 * i + 1]);
      const float c = __ldg(cs + i), s = __ldg(cs + half + i);
      float ra, rb;
      *reinterpret_cast<uint32_t*>(dr + 2 * i) = Pack<T>::run(a * c - b * s, a * s + b * c, ra, rb);
    }
  }
}

}  // namespace

kvc_status launch_rope_table(float* cos_sin, int max_position, int rope_dim, float base,
                             cudaStream_t stream) {
  const long long n = static_cast<long long>(max_position) * (rope_dim / 2);
  const int threads = 256;
  const long long want = (n + threads - 1) / threads;
  const int cap = device_sm_count() * 8;
  const int grid = static_cast<int>(want < cap ? want : cap);
  rope_table_kernel<<<grid, threads, 0, stream>>>(cos_sin, max_position, rope_dim,
                                                   static_cast<double>(base));
  return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

kvc_status launch_rmsnorm_rope_cache(const void* kv, const void* gamma, float eps,
                                     const float* cos_sin, int max_position,
                                     const int32_t* positions, const int32_t* slot_mapping,
                                     void* cache_norm, void* cache_rope, int num_tokens,
                                     int num_heads, int d_norm, int d_rope, int block_size,
                                     int num_blocks, kvc_dtype dtype, uint32_t* err_flag,
                                     cudaStream_t stream) {
  if (num_tokens == 0) return KVC_OK;
  const long long rows = static_cast<long long>(num_tokens) * num_heads;
  const int threads = 256;  // 8 rows per CTA pass
  const long long want = (rows * 32 + threads - 1) / threads;
  const int cap = device_sm_count() * 16;
  const int grid = static_cast<int>(want < cap ? want : cap);
  const long long ns = static_cast<long long>(num_blocks) * block_size;
  auto go = [&](auto tag) {
    using T = decltype(tag);
    rmsnorm_rope_cache_kernel<T><<<grid, threads, 0, stream>>>(
        static_cast<const T*>(kv), static_cast<const T*>(gamma), eps, cos_sin, max_position,
        positions, slot_mapping, static_cast<T*>(cache_norm), static_cast<T*>(cache_rope),
        num_tokens, num_heads, d_norm, d_rope, ns, err_flag);
  };
  if (dtype == KVC_BF16) go(__nv_bfloat16());
  else go(__half());
  return cudaGetLastError() == cudaSuccess ? KVC_OK : KVC_ERR_CUDA;
}

}  // namespace kvc
