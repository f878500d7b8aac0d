// Blackwell (sm_103a) tensor-core and cluster building blocks: tcgen05.mma
// with shared-memory matrix descriptors, tensor-memory (TMEM) allocation and
// loads/stores, and the cluster / distributed-shared-memory operations a CTA
// pair uses to exchange data.  Thin inline-PTX wrappers only.
#pragma once

#include <stdint.h>

#include "kvc_device.cuh"

namespace kvc {

// ----------------------------------------------------------- descriptors

// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile whose
// base is 1024-byte aligned.  K-major operand ([rows][64 elements] regions):
// lbo unused (16), sbo = 1024 (8 rows of 128 B); the start address advances
// by 32 B per 16-element K step inside a region.  MN-major operand ([K rows]
// [64 MN elements] regions): lbo = byte stride between 64-wide MN regions,
// sbo = 1024 (8 K rows); the start advances by 16 rows (2048 B) per K step.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2) << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor of tcgen05.mma.kind::f16: fp32 accumulator, A and B
// both bf16 (bf16 = true) or both fp16, M x N tile, operand majors
// (0 = K-major, 1 = MN-major).
__host__ __device__ constexpr uint32_t umma_idesc_f16(bool bf16, int M, int N, int a_mn,
                                                      int b_mn) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         (static_cast<uint32_t>(a_mn) << 15) | (static_cast<uint32_t>(b_mn) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Descriptor of the same operand `bytes` further on in shared memory (the
// start-address field holds address / 16 and never overflows its 14 bits).
__device__ __forceinline__ uint64_t desc_advance(uint64_t desc, uint32_t bytes) {
  return desc + static_cast<uint64_t>(bytes >> 4);
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Generic-proxy shared-memory writes become visible to the tensor core.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------ warp-convergent issue
//
// The issuing warp runs its loop with all 32 lanes converged and predicates
// each tcgen05.mma / commit on one elected lane.  Descriptors then stay
// warp-uniform, and the issue keeps pace with the tensor core even when the
// other warps on the same scheduler issue arithmetic every cycle (issued from
// a lone diverged lane, the same MMAs slowed down several times over).

// Whole warp: 1 in exactly one lane, 0 in the others.
__device__ __forceinline__ uint32_t elect_one_sync() {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 t;\n\t"
      "elect.sync t|e, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, e;\n\t}"
      : "=r"(r));
  return r;
}

// D (+)= A[smem] * B[smem] from the elected lane; `accumulate` at run time.
__device__ __forceinline__ void umma_ss_e(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate, uint32_t leader) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 e, %5, 0;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(leader)
      : "memory");
}
// The same with A read from tensor memory.
__device__ __forceinline__ void umma_ts_e(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate, uint32_t leader) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t"
      "setp.ne.b32 e, %5, 0;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(leader)
      : "memory");
}
// tcgen05.commit from the elected lane.
__device__ __forceinline__ void umma_commit_e(uint64_t* bar, uint32_t leader) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "setp.ne.b32 e, %1, 0;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar)),
      "r"(leader)
      : "memory");
}
// Two accumulating MMAs (A and B in shared memory) from the elected lane,
// preceded in the same instruction sequence by every lane testing three
// mbarrier phases the next group needs; the predicates are consumed only
// after the MMAs are issued, so the tests' latency hides behind them.
// Returns whether all three phases had completed.
__device__ __forceinline__ bool umma_ss_acc2_test3_e(uint32_t d_tmem, uint64_t a0, uint64_t b0,
                                                     uint64_t a1, uint64_t b1, uint32_t idesc,
                                                     uint64_t* bar0, uint32_t par0, uint64_t* bar1,
                                                     uint32_t par1, uint64_t* bar2, uint32_t par2,
                                                     uint32_t leader) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p, q, r, e;\n\t"
      "setp.ne.b32 e, %13, 0;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%6], %7;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 q, [%8], %9;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 r, [%10], %11;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%1], %2, %3, %12, 1;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%1], %4, %5, %12, 1;\n\t"
      "and.pred p, p, q;\n\t"
      "and.pred p, p, r;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(d_tmem), "l"(a0), "l"(b0), "l"(a1), "l"(b1), "r"(smem_u32(bar0)), "r"(par0),
        "r"(smem_u32(bar1)), "r"(par1), "r"(smem_u32(bar2)), "r"(par2), "r"(idesc), "r"(leader)
      : "memory");
  return ok != 0;
}

// ------------------------------------------------------------------ TMEM

// Whole warp: allocate `ncols` (power of two, 32..512) TMEM columns; the base
// address is written to *slot (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Warp w of a warpgroup reads TMEM lanes 32*(w%4) .. +31 (one row per
// thread), 16 consecutive 32-bit columns starting at taddr's column.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}

__device__ __forceinline__ void tmem_st16_u32(uint32_t taddr, const uint32_t* w) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
      "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// --------------------------------------------------------- paired fp32

// max(a, b, c) in one instruction (sm_100+); exact, like two fmaxf.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Paired fp32 arithmetic (one instruction for two lanes of a float2) and a
// round-to-nearest pack of two floats into 16-bit pairs.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(r)
      : "l"(*reinterpret_cast<const uint64_t*>(&a)), "l"(*reinterpret_cast<const uint64_t*>(&b)),
        "l"(*reinterpret_cast<const uint64_t*>(&c)));
  return *reinterpret_cast<float2*>(&r);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;"
      : "=l"(r)
      : "l"(*reinterpret_cast<const uint64_t*>(&a)), "l"(*reinterpret_cast<const uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&r);
}
template <typename T>
__device__ __forceinline__ uint32_t pack_pair(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack_pair<__nv_bfloat16>(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}
template <>
__device__ __forceinline__ uint32_t pack_pair<__half>(float a, float b) {
  __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}
// acc += the two values of a pair packed by pack_pair (low half into acc.x),
// each widened exactly and added in fp32 with round-to-nearest (the
// mixed-precision add of sm_100 and later, one instruction per value).
template <typename T>
__device__ __forceinline__ void acc_pair(float2& acc, uint32_t w);
template <>
__device__ __forceinline__ void acc_pair<__nv_bfloat16>(float2& acc, uint32_t w) {
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "add.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %1, hi, %1;\n\t}"
      : "+f"(acc.x), "+f"(acc.y)
      : "r"(w));
}
template <>
__device__ __forceinline__ void acc_pair<__half>(float2& acc, uint32_t w) {
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %1, hi, %1;\n\t}"
      : "+f"(acc.x), "+f"(acc.y)
      : "r"(w));
}

// --------------------------------------------------------------- cluster

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// All threads of both CTAs of the cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster_v4(uint32_t caddr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(caddr), "f"(v.x),
               "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}

// Asynchronous 16-byte store into another CTA's shared memory that completes
// 16 bytes of the transaction count of that CTA's mbarrier `cbar` (both
// addresses from map_to_rank).  The receiver's wait on the barrier (acquire,
// cluster scope) makes the data visible; no fence is needed on this side.
__device__ __forceinline__ void st_async_cluster_v4(uint32_t caddr, float4 v, uint32_t cbar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
          caddr),
      "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(cbar)
      : "memory");
}

// Arrive (no memory ordering) on an mbarrier of another CTA of the cluster:
// for "buffer free" signals after reads whose values have been consumed.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t caddr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr)
               : "memory");
}

// Release-arrive on an mbarrier of another CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t caddr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait on a barrier that threads of the other CTA arrive on.
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t* bar, uint32_t parity,
                                                          uint32_t* err_flag) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait_cluster(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      set_flag(err_flag, KVC_FLAG_WAIT_TIMEOUT);
      return false;
    }
  }
}

}  // namespace kvc
