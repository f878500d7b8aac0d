// Device-side building blocks shared by the kvc kernels (sm_103a).
//
// Thin inline-PTX wrappers for the mbarrier / TMA / ldmatrix / mma.sync
// instructions the kernels use, plus bounded waits: every spin on an
// mbarrier gives up after a wall-clock limit, records KVC_FLAG_WAIT_TIMEOUT
// and lets the kernel return instead of hanging the GPU.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/kvc.h"

namespace kvc {

// Wall-clock limit of one bounded wait (nanoseconds of %globaltimer).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void set_flag(uint32_t* err_flag, uint32_t bit) {
  if (err_flag) atomicOr(err_flag, bit);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.release.cta.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

// Non-blocking probe: true if the phase with the given parity has completed.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false (and
// sets KVC_FLAG_WAIT_TIMEOUT) if it has not completed within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint32_t* err_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      set_flag(err_flag, KVC_FLAG_WAIT_TIMEOUT);
      return false;
    }
  }
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 4-D tiled bulk tensor load global -> shared, completion counted in bytes on
// `bar`.  c0 is the innermost coordinate (elements); c0 * 2 bytes must be a
// multiple of 16 (the kernels only pass 0 or multiples of 64 elements).
__device__ __forceinline__ void tma_load_4d(void* smem_dst, const CUtensorMap* m, uint64_t* bar,
                                            int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(smem_u32(bar))
      : "memory");
}

// 3-D variant of tma_load_4d.
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* m, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// ---------------------------------------------------------------- warp MMA

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <typename T>
struct MmaOp;

template <>
struct MmaOp<__nv_bfloat16> {
  __device__ __forceinline__ static void run(float* d, const uint32_t* a, uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
};

template <>
struct MmaOp<__half> {
  __device__ __forceinline__ static void run(float* d, const uint32_t* a, uint32_t b0,
                                             uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
};

// Pack two fp32 values into one 32-bit register of two 16-bit values (low
// half = first), rounding to nearest even; also return the rounded values.
template <typename T>
struct Pack;

template <>
struct Pack<__nv_bfloat16> {
  __device__ __forceinline__ static uint32_t run(float a, float b, float& ra, float& rb) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    float2 f = __bfloat1622float2(v);
    ra = f.x;
    rb = f.y;
    return *reinterpret_cast<uint32_t*>(&v);
  }
  __device__ __forceinline__ static __nv_bfloat16 cvt(float a) { return __float2bfloat16_rn(a); }
};

template <>
struct Pack<__half> {
  __device__ __forceinline__ static uint32_t run(float a, float b, float& ra, float& rb) {
    __half2 v = __floats2half2_rn(a, b);
    float2 f = __half22float2(v);
    ra = f.x;
    rb = f.y;
    return *reinterpret_cast<uint32_t*>(&v);
  }
  __device__ __forceinline__ static __half cvt(float a) { return __float2half_rn(a); }
};

// 2^x on the SFU (PTX ex2.approx.ftz.f32); ex2(-inf) = +0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Atomic add at GPU scope with acquire-release semantics; returns the old value.
__device__ __forceinline__ int atomic_add_acq_rel(int* addr, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(addr), "r"(v)
               : "memory");
  return old;
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Symmetric INT8 codes of one row spread over kLanes consecutive lanes of a
// warp (32 or 16; an aligned group), E consecutive elements per lane (lane l
// of the group holds elements l*E .. l*E+E-1): amax over the row by
// shuffles, scale = amax / 127, code = rint(x * (127 / amax)) with ties to
// even, clamped to [-127, 127]; the divisions and the product are correctly
// rounded fp32, so the codes do not depend on how the row is spread.
// packed[i]: codes 4i .. 4i+3 of the lane, byte e = element 4i + e.  An
// all-zero row gets scale 0 and codes 0.  Every lane of the warp must call it.
template <int E, int kLanes>
__device__ __forceinline__ void quantize_row_int8(const float (&x)[E],
                                                  uint32_t (&packed)[(E + 3) / 4],
                                                  float& scale) {
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
  for (int off = kLanes / 2; off > 0; off >>= 1)
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float inv = amax > 0.f ? __fdiv_rn(127.f, amax) : 0.f;
  scale = __fdiv_rn(amax, 127.f);
#pragma unroll
  for (int i = 0; i < (E + 3) / 4; ++i) packed[i] = 0;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    int c = __float2int_rn(__fmul_rn(x[e], inv));
    c = c > 127 ? 127 : (c < -127 ? -127 : c);
    packed[e / 4] |= (static_cast<uint32_t>(c) & 0xffu) << (8 * (e % 4));
  }
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` in a tile of
// 128-byte rows written by TMA with CU_TENSOR_MAP_SWIZZLE_128B (the tile base
// is 1024-byte aligned): the chunk index is XORed with row % 8.
__device__ __forceinline__ uint32_t swz128(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

}  // namespace kvc
