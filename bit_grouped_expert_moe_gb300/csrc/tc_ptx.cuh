// Inline-PTX building blocks for the sm_103a tensor-core path: mbarriers,
// TMA tile loads, cp.async, proxy fences, tensor memory (TMEM) allocation and
// loads, tcgen05.mma with its shared-memory and instruction descriptors.
// Every wait is bounded by a deadline on the global timer; a wait that runs
// out returns false and the caller records MOE_ERR_DEVICE_TIMEOUT.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "common.cuh"

namespace bgmoe {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------ mbarrier ---
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Makes initialised barriers visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// The waiting thread may be suspended (up to the hint, 0.5 ms) until the phase
// completes, instead of spinning on issue slots.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(500000u)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the same condition (no suspension).
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete, sleeping 32 ns
// between polls. Returns false once `*abort` is set or the deadline passes
// (then it sets *abort). A phase that has already completed is seen by the
// non-blocking test, which returns sooner than a potentially blocking wait.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t deadline) {
  if (mbar_test_wait(bar, parity)) return true;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_timer_ns() > deadline) {
      *abort = 1;
      return false;
    }
    __nanosleep(32);  // leave the issue slots to the warps doing work (7 % on the expert GEMMs)
  }
}

// True in exactly one lane of the (converged) warp.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n .reg .b32 r;\n .reg .pred p;\n elect.sync r|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(pred));
  return pred != 0;
}

// ------------------------------------------------------------------ TMA ---
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------- cp.async ---
// 16-byte copy global -> shared; src_bytes = 0 fills the 16 bytes with zeros.
__device__ __forceinline__ void cp_async_16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Arrives on `bar` once every cp.async issued so far by this thread has
// landed; the arrival is counted in the barrier's expected count (noinc).
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy reads (tcgen05.mma operands).
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------- TMEM ---
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 columns of this thread's TMEM lane (32x32b shape:
// thread i of the warp reads lane (taddr.lane + i)).
__device__ __forceinline__ void tmem_ld_32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ------------------------------------------------------------------ MMA ---
// Shared-memory matrix descriptor of a K-major operand tile in the 128-byte
// swizzle layout: rows of 64 fp16 (128 bytes), 8-row atoms of 1024 bytes
// stacked along M/N (stride 1024), tile base 1024-byte aligned. Moving 16
// elements along K inside the atom adds 32 bytes to the start address.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);  // start address
  d |= (uint64_t)1 << 16;                   // leading-dimension byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;         // stride byte offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                   // descriptor version (sm_100 family)
  d |= (uint64_t)2 << 61;                   // layout: 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16 with fp16 A and B, fp32 accumulator,
// both operands K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4)                       // D format: f32
         | (0u << 7) | (0u << 10)        // A, B format: f16
         | ((uint32_t)(N >> 3) << 17)    // N / 8
         | ((uint32_t)(M >> 4) << 24);   // M / 16
}

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives on `bar` once every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// ------------------------------------------------------ 4-bit -> fp16 ---
// One uint32 of 8 codes (code k in bits 4k..4k+3) -> four fp16x2 registers
// W = scale * q + bias, with pairs (q0,q4), (q1,q5), (q2,q6), (q3,q7): the
// operands' K order inside every group of 8 is 0,4,1,5,2,6,3,7, which the
// activations share (a permutation of K applied to both operands leaves the
// product unchanged).
//
// s2 holds scale * 2^14 and b2 the bias (group_scale_bias), and the codes
// come out as q * 2^-14, so that W = fma(q 2^-14, scale 2^14, bias): the
// product is exact and W is rounded once, at its own magnitude. (Taking the
// scale itself to fp16 would round any scale below 2^-14 to a subnormal with
// a fixed step of 2^-24, an error that q, up to 15, then multiplies.)
// 0x2C00 is fp16 2^-4, whose unit in the last place is 2^-14: OR-ing a code
// into its low mantissa bits gives exactly 2^-4 + q 2^-14, and a code 4 bits
// up gives 2^-4 + q 2^-10; (2^-4 + q 2^-14) - 2^-4 and
// (2^-4 + q 2^-10) 2^-4 - 2^-8 are then exactly q 2^-14.
__device__ __forceinline__ void dequant8_f16(uint32_t w, __half2 s2, __half2 b2, uint32_t (&out)[4]) {
  const uint32_t kMagic = 0x2C002C00u;
  uint32_t lo0, hi0, lo1, hi1;
  const uint32_t w8 = w >> 8;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(lo0) : "r"(w), "r"(0x000F000Fu), "r"(kMagic));
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(hi0) : "r"(w), "r"(0x00F000F0u), "r"(kMagic));
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(lo1) : "r"(w8), "r"(0x000F000Fu), "r"(kMagic));
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(hi1) : "r"(w8), "r"(0x00F000F0u), "r"(kMagic));
  const __half2 k4 = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));   // 2^-4
  const __half2 km8 = __halves2half2(__ushort_as_half(0x9C00), __ushort_as_half(0x9C00));  // -2^-8
  const __half2 q04 = __hsub2(*reinterpret_cast<const __half2*>(&lo0), k4);
  const __half2 q15 = __hfma2(*reinterpret_cast<const __half2*>(&hi0), k4, km8);
  const __half2 q26 = __hsub2(*reinterpret_cast<const __half2*>(&lo1), k4);
  const __half2 q37 = __hfma2(*reinterpret_cast<const __half2*>(&hi1), k4, km8);
  const __half2 r0 = __hfma2(q04, s2, b2), r1 = __hfma2(q15, s2, b2);
  const __half2 r2 = __hfma2(q26, s2, b2), r3 = __hfma2(q37, s2, b2);
  out[0] = *reinterpret_cast<const uint32_t*>(&r0);
  out[1] = *reinterpret_cast<const uint32_t*>(&r1);
  out[2] = *reinterpret_cast<const uint32_t*>(&r2);
  out[3] = *reinterpret_cast<const uint32_t*>(&r3);
}

// A group's bf16 scale and bias as the fp16 scale * 2^14 and bias that
// dequant8_f16 takes, packed (scale low, bias high). The scaled scale is
// exact for 2^-28 <= |scale| < 4; smaller scales move a weight by less than
// one fp16 step. Returns false for |scale| >= 4 (scale * 2^14 past fp16),
// which the caller reports as MOE_ERR_RANGE.
__device__ __forceinline__ bool group_scale_bias(float s, float b, uint32_t& packed) {
  const __half2 h = __floats2half2_rn(s * 16384.f, b);
  packed = *reinterpret_cast<const uint32_t*>(&h);
  return fabsf(s) < 4.f;
}

// Position of logical column n inside its group of 8 in the permuted K order
// 0,4,1,5,2,6,3,7 (the inverse of that order).
__host__ __device__ __forceinline__ int perm8_pos(int n) {
  const int r = n & 7;
  return (n & ~7) | (r < 4 ? 2 * r : 2 * (r - 4) + 1);
}

}  // namespace tc
}  // namespace bgmoe
