// Device helpers shared by the kernels of the MoE layer (sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace bgmoe {

constexpr int kGroup = 64;       // weights per scale/bias pair
constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;

// Host-visible launch facts shared between api.cu and the kernel files.
struct Geometry {
  int T, H, I, E, K, BM;
  int shared;       // 1 if a shared expert exists
  int A;            // T * K
  int rows;         // A + (shared ? T : 0): rows of h / o
  int max_tiles;    // block-map capacity
  int route_blocks; // grid of the routing kernel
  int tokens_per_block;
};

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// Monotone map fp32 -> uint32: a > b  <=>  key(a) > key(b) (finite inputs;
// -0 and +0 map to the same key).
__device__ __forceinline__ uint32_t float_order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint64_t ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ float silu_f32(float a) { return a / (1.0f + __expf(-a)); }

// A kernel after the routing kernel does nothing once a device error is set.
__device__ __forceinline__ bool device_failed(const int32_t* status) {
  return *reinterpret_cast<const volatile int32_t*>(status) != 0;
}

// Raises a kernel's dynamic shared-memory limit to `bytes` the first time a
// launch needs it (the value is cached, so launches inside a CUDA-graph
// capture make no attribute call once a first, uncaptured call has run). The
// default limit is 48 KB minus the kernel's static shared memory, so even a
// small request is raised once.
template <typename Kernel>
inline cudaError_t ensure_smem(Kernel k, size_t bytes, int* configured) {
  if (bytes == 0 || (int)bytes <= *configured) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) *configured = (int)bytes;
  return e;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

}  // namespace bgmoe
