// Router scores: l[t, e] = x[t, :] . W_r[e, :] for the E routed experts and,
// in column E, the shared-expert gate logit x[t, :] . w_sg.
// [dothoosh.com "Perplexity Lily: 1.35x faster decode for Qwen3.6 on Apple
// silicon", "Model specification": the router scores 256 experts per token.]
//
// One warp owns one weight row (expert e, or the gate row); a block covers
// kRouterTokens tokens whose bf16 rows sit in shared memory, so each 16-byte
// weight load feeds 8 x kRouterTokens FMAs. The blocks also clear the routing
// kernel's look-back words (the routing kernel runs after this one on the same
// stream; the call's status word is cleared in stream order before this
// kernel).
#include "common.cuh"

namespace bgmoe {

constexpr int kRouterWarps = 8;
constexpr int kRouterTokens = 8;

__global__ void __launch_bounds__(kRouterWarps * 32)
router_logits_kernel(const uint16_t* __restrict__ x, const uint16_t* __restrict__ wr,
                     const uint16_t* __restrict__ wsg, float* __restrict__ logits, int T, int H,
                     int E, int ld, unsigned long long* __restrict__ state, int n_state,
                     int32_t* __restrict__ status, uint16_t* __restrict__ x16,
                     unsigned int* __restrict__ bar) {
  extern __shared__ __align__(16) uint16_t xs[];  // [kRouterTokens][H]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.y * kRouterTokens;
  const int nt = min(kRouterTokens, T - t0);

  // Let a kernel launched after this one with programmatic dependent launch
  // start its weight prefetch now; it waits for this grid before reading
  // anything this kernel writes.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // Clear the look-back words and (when given) a grid-barrier counter for
  // this call.
  {
    const int nblocks = gridDim.x * gridDim.y;
    const int b = blockIdx.y * gridDim.x + blockIdx.x;
    for (int i = b * blockDim.x + threadIdx.x; i < n_state; i += nblocks * blockDim.x) state[i] = 0ull;
    if (b == 0 && threadIdx.x == 0 && bar != nullptr) *bar = 0u;
  }

  const int vec_per_row = H / 8;
  const int e = blockIdx.x * kRouterWarps + warp;
  const bool has_gate = wsg != nullptr;
  const bool has_row = e < E || (e == E && has_gate);
  const uint16_t* row = (e < E) ? wr + (size_t)e * H : wsg;

  // The first batch of this warp's weight loads goes out before x is staged
  // (the two do not depend on each other); every batch is issued before any
  // use, so a row of H <= 2048 costs one memory round trip.
  constexpr int kBatch = 8;
  uint4 w4[kBatch];
  auto load_batch = [&](int v0) {
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int v = v0 + 32 * u;
      if (has_row && v < vec_per_row) w4[u] = ldg_nc_v4(row + (size_t)v * 8);
    }
  };
  load_batch(lane);

  // Stage the block's token rows (16-byte copies; H is a multiple of 64).
  for (int i = threadIdx.x; i < nt * vec_per_row; i += blockDim.x) {
    const int j = i / vec_per_row, v = i - j * vec_per_row;
    reinterpret_cast<uint4*>(xs)[j * vec_per_row + v] =
        reinterpret_cast<const uint4*>(x + (size_t)(t0 + j) * H)[v];
  }
  __syncthreads();

  // The tensor-core expert path reads x as fp16 (exact for bf16 values of
  // magnitude >= 2^-14), K-permuted within groups of 8 as 0,4,1,5,2,6,3,7 to
  // match the order in which the 4-bit codes unpack.
  if (x16 != nullptr && blockIdx.x == 0) {
    bool big = false;
    for (int i = threadIdx.x; i < nt * H; i += blockDim.x) {
      const int j = i / H, k = i - j * H;
      const int r = k & 7;
      const int pk = (k & ~7) | (r < 4 ? 2 * r : 2 * (r - 4) + 1);
      const float v = bf16_bits_to_f32(xs[j * H + k]);
      big |= fp16_overflows(v);
      x16[(size_t)(t0 + j) * H + pk] = __half_as_ushort(__float2half_rn(v));
    }
    if (big) flag_range(status);
  }
  if (!has_row) return;

  float acc[kRouterTokens];
#pragma unroll
  for (int j = 0; j < kRouterTokens; ++j) acc[j] = 0.f;

  for (int v0 = lane; v0 < vec_per_row; v0 += 32 * kBatch) {
    if (v0 != lane) load_batch(v0);
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int v = v0 + 32 * u;
      if (v >= vec_per_row) break;
      const uint32_t wv[4] = {w4[u].x, w4[u].y, w4[u].z, w4[u].w};
      float wf[8];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        wf[2 * m] = bf16_bits_to_f32(wv[m] & 0xFFFFu);
        wf[2 * m + 1] = bf16_bits_to_f32(wv[m] >> 16);
      }
#pragma unroll
      for (int j = 0; j < kRouterTokens; ++j) {
        if (j < nt) {
          const uint4 x4 = reinterpret_cast<const uint4*>(xs)[j * vec_per_row + v];
          const uint32_t xv[4] = {x4.x, x4.y, x4.z, x4.w};
          float a = acc[j];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            a = fmaf(wf[2 * m], bf16_bits_to_f32(xv[m] & 0xFFFFu), a);
            a = fmaf(wf[2 * m + 1], bf16_bits_to_f32(xv[m] >> 16), a);
          }
          acc[j] = a;
        }
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kRouterTokens; ++j) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], o);
  }
  if (lane < nt) {
    float mine = acc[0];
#pragma unroll
    for (int j = 1; j < kRouterTokens; ++j)
      if (lane == j) mine = acc[j];
    logits[(size_t)(t0 + lane) * ld + e] = mine;
  }
}

cudaError_t launch_router_logits(const Geometry& g, const void* x, const void* wr, const void* wsg,
                                 float* logits, unsigned long long* state, int n_state,
                                 int32_t* status, uint16_t* x16, cudaStream_t stream, unsigned int* bar) {
  const int rows = g.E + (wsg ? 1 : 0);
  dim3 grid((rows + kRouterWarps - 1) / kRouterWarps, (g.T + kRouterTokens - 1) / kRouterTokens);
  const size_t smem = (size_t)kRouterTokens * g.H * sizeof(uint16_t);
  static SmemLimitMemo smem_memo;
  cudaError_t e = ensure_smem(router_logits_kernel, smem, &smem_memo);
  if (e != cudaSuccess) return e;
  router_logits_kernel<<<grid, kRouterWarps * 32, smem, stream>>>(
      static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(wr), static_cast<const uint16_t*>(wsg),
      logits, g.T, g.H, g.E, g.E + 1, state, n_state, status, x16, bar);
  return cudaGetLastError();
}

}  // namespace bgmoe
