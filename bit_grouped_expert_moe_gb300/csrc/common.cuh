// Device helpers shared by the kernels of the MoE layer (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "host_memo.h"
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

// Inverse of float_order_key for the keys it produces from finite values.
__device__ __forceinline__ float order_key_to_float(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

// Top-k of one token by one warp, given the logits: lane l holds
// lv[j] = logit of expert l + 32 j (entries past E ignored) and every lane the
// shared-gate logit. Ties go to the lower expert index, and each pick gets its
// renormalised softmax weight: lane k < K returns pick k in *e_out and its
// weight in *w_out; every lane returns sigmoid(gate_logit) in *gate_out when
// `shared`. Keys are fp32 order keys (0 marks an empty or taken entry: a
// finite logit never maps to 0).
//
// Each lane first sorts its 8 entries once (a 19-comparator network on
// (key, lower j first) packed into 64 bits, no branches). A round then takes
// the warp maximum of the lanes' heads and, among the lanes holding it, the
// lowest expert index; the winning lane pops its head. Every lane runs the
// same instructions, and a round is two warp reductions and a few selects.
__device__ __forceinline__ void warp_topk_select(const float (&lv)[kMaxExperts / 32], float gate_logit,
                                                 const float* bias, int E, int K, bool shared, int lane,
                                                 int* e_out, float* w_out, float* gate_out) {
  constexpr int kN = kMaxExperts / 32;
  static_assert(kN == 8, "the sorting network below sorts 8 entries per lane");
  uint64_t v[kN];
#pragma unroll
  for (int j = 0; j < kN; ++j) {
    const float b = bias ? __ldg(bias + min(lane + 32 * j, E - 1)) : 0.f;
    const uint32_t key = lane + 32 * j < E ? float_order_key(lv[j] + b) : 0u;
    v[j] = ((uint64_t)key << 32) | (uint32_t)(kN - 1 - j);  // equal keys: the lower j sorts first
  }
  auto cx = [&](int a, int b) {  // larger value to position a
    const uint64_t hi = v[a] > v[b] ? v[a] : v[b], lo = v[a] > v[b] ? v[b] : v[a];
    v[a] = hi;
    v[b] = lo;
  };
  cx(0, 2), cx(1, 3), cx(4, 6), cx(5, 7);
  cx(0, 4), cx(1, 5), cx(2, 6), cx(3, 7);
  cx(0, 1), cx(2, 3), cx(4, 5), cx(6, 7);
  cx(2, 4), cx(3, 5);
  cx(1, 4), cx(3, 6);
  cx(1, 2), cx(3, 4), cx(5, 6);
  uint32_t my_key = 0u, top_key = 0u;
  int my_e = 0;
  for (int k = 0; k < K; ++k) {
    const uint32_t hk = (uint32_t)(v[0] >> 32);
    const uint32_t he = (uint32_t)lane + 32u * (uint32_t)(kN - 1 - (int)(v[0] & 0xFFFFFFFFu));
    const uint32_t M = __reduce_max_sync(0xffffffffu, hk);
    const uint32_t ew = __reduce_min_sync(0xffffffffu, hk == M ? he : 0xFFFFFFFFu);
    top_key = k == 0 ? M : top_key;
    my_key = lane == k ? M : my_key;
    my_e = lane == k ? (int)ew : my_e;
    const bool won = lane == (int)(ew & 31u);
#pragma unroll
    for (int j = 0; j < kN - 1; ++j) v[j] = won ? v[j + 1] : v[j];
    v[kN - 1] = won ? 0ull : v[kN - 1];
  }
  // weights: exp(v_k - v_0) / sum over the selected (lanes k < K in parallel)
  const float z = lane < K ? expf(order_key_to_float(my_key) - order_key_to_float(top_key)) : 0.f;
  float sum = z;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  *e_out = my_e;
  *w_out = z / sum;
  *gate_out = shared ? 1.f / (1.f + expf(-gate_logit)) : 0.f;
}

// warp_topk_select over lrow[0..E) (+ bias) read from global memory: every
// logit load is issued before any is used (one L2 round trip).
__device__ __forceinline__ void warp_topk(const float* lrow, const float* bias, int E, int K, bool shared, int lane,
                                          int* e_out, float* w_out, float* gate_out) {
  float lv[kMaxExperts / 32];
#pragma unroll
  for (int j = 0; j < kMaxExperts / 32; ++j) lv[j] = __ldcg(lrow + min(lane + 32 * j, E - 1));
  const float gate_logit = __ldcg(lrow + (shared ? E : 0));
  warp_topk_select(lv, gate_logit, bias, E, K, shared, lane, e_out, w_out, gate_out);
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

// Records MOE_ERR_RANGE in the call's status word, unless a failure is
// already recorded there: a value written as an fp16 operand of the expert
// path (x, h or o) left the range where fp16 holds it to the layer's
// tolerance (see fp16_overflows and kFp16Floor).
__device__ __forceinline__ void flag_range(const int32_t* status) {
  atomicCAS(const_cast<int32_t*>(status), 0, (int32_t)MOE_ERR_RANGE);
}

// A bf16 value that becomes inf in fp16 (|v| >= 65520 rounds past 65504).
__device__ __forceinline__ bool fp16_overflows(float v) { return fabsf(v) >= 65520.f; }

// Below 2^-14 fp16 keeps a fixed absolute step of 2^-24. A slice of h or o
// whose largest magnitude is under 2^-16 is therefore rounded with an error
// above 2^-9 of its largest value: the kernels report such a slice (unless it
// is all zero) as MOE_ERR_RANGE instead of returning a result that has lost
// the precision the rest of the path keeps.
constexpr float kFp16Floor = 1.52587890625e-05f;  // 2^-16

// Debug build (-DBGMOE_BOUNDS_CHECK): an index read from a table that another
// kernel or block wrote is checked against its range before it is used. A
// value outside [lo, hi] is replaced by lo and MOE_ERR_BOUNDS recorded in the
// status word (unless a failure is already there), so the access stays
// inside its buffer and every barrier protocol still runs to the end; the
// result of the call is then not valid. Without the flag the index passes
// through unchanged and the check costs nothing.
__device__ __forceinline__ int checked(int v, int lo, int hi, const int32_t* status) {
#ifdef BGMOE_BOUNDS_CHECK
  if (v < lo || v > hi) {
    atomicCAS(const_cast<int32_t*>(status), 0, (int32_t)MOE_ERR_BOUNDS);
    return lo;
  }
#else
  (void)lo;
  (void)hi;
  (void)status;
#endif
  return v;
}

// A kernel after the routing kernel does nothing once a device error is set.
__device__ __forceinline__ bool device_failed(const int32_t* status) {
  return *reinterpret_cast<const volatile int32_t*>(status) != 0;
}

// device_failed, decided once for the whole block (every thread must call
// it): thread 0 reads the status word and all threads get its answer, so a
// word set meanwhile by another block (a range report) cannot split the
// block into threads that return and threads that wait at a barrier.
__device__ __forceinline__ bool block_failed(const int32_t* status) {
  return __syncthreads_or(threadIdx.x == 0 && device_failed(status)) != 0;
}

// The current device and an identifier of its current CUDA context (0 when
// no context is current or the driver cannot name it). Defined in api.cu.
cudaError_t current_device_context(int* dev, unsigned long long* ctx);

// Raises a kernel's dynamic shared-memory limit to `bytes` the first time a
// launch on this device and context needs it (memoised per device and
// context, so launches inside a CUDA-graph capture make no attribute call
// once a first, uncaptured call has run there). The default limit is 48 KB
// minus the kernel's static shared memory, so even a small request is raised
// once.
template <typename Kernel>
inline cudaError_t ensure_smem(Kernel k, size_t bytes, SmemLimitMemo* memo) {
  int dev = 0;
  unsigned long long ctx = 0;
  cudaError_t e = current_device_context(&dev, &ctx);
  if (e != cudaSuccess) return e;
  return static_cast<cudaError_t>(memo->ensure(dev, ctx, (int)bytes, [&](int b) {
    return static_cast<int>(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, b));
  }));
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

}  // namespace bgmoe
