// Gather + weighted combine + shared-expert add:
//   y[t, :] = sum_{k=0..K-1} w[t, k] * o[inv[t*K + k], :] + g[t] * o[A + t, :]
// summed in that fixed order in fp32 (no atomics, so the result is the same
// on every run). [dothoosh.com "Perplexity Lily: 1.35x faster decode for
// Qwen3.6 on Apple silicon", "Model specification": each token's output mixes
// its 8 chosen experts with the shared expert that processes every token.]
#include "kernels.h"

namespace bgmoe {

constexpr int kCombineThreads = 64;

__global__ void __launch_bounds__(kCombineThreads)
combine_kernel(int H, int K, int A, int shared, const __half* __restrict__ o, const int32_t* __restrict__ inv,
               const float* __restrict__ weights, const float* __restrict__ gate,
               const int32_t* __restrict__ status, float* __restrict__ y) {
  if (block_failed(status)) return;
  const int t = blockIdx.x;
  const int c = (blockIdx.y * kCombineThreads + threadIdx.x) * 8;
  const bool active = c < H;  // every thread reaches the block-wide range check
  // Every load of the token goes out before any is used: the K row
  // indices and weights, then the K + 1 rows of o (the shared row last).
  int rows[kMaxTopK + 1];
  float wt[kMaxTopK + 1];
#pragma unroll
  for (int k = 0; k < kMaxTopK; ++k) {
    rows[k] = k < K ? checked(inv[(size_t)t * K + k], 0, A - 1, status) : 0;
    wt[k] = k < K ? weights[(size_t)t * K + k] : 0.f;
  }
  rows[kMaxTopK] = A + t;
  wt[kMaxTopK] = shared ? gate[t] : 0.f;
  uint4 v[kMaxTopK + 1];
#pragma unroll
  for (int k = 0; k <= kMaxTopK; ++k)
    if (active && (k < K || (k == kMaxTopK && shared)))
      v[k] = *reinterpret_cast<const uint4*>(o + (size_t)rows[k] * H + c);
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  // bit k: row k of o has, in this thread's 8 columns, a value >= 2^-16
  // (big) / a nonzero value (nz)
  unsigned big = 0u, nz = 0u;
#pragma unroll
  for (int k = 0; k <= kMaxTopK; ++k) {
    if (!active || !(k < K || (k == kMaxTopK && shared))) continue;
    const __half2* h2 = reinterpret_cast<const __half2*>(&v[k]);
    float mx = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(h2[i]);
      mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
      acc[2 * i] = fmaf(wt[k], f.x, acc[2 * i]);
      acc[2 * i + 1] = fmaf(wt[k], f.y, acc[2 * i + 1]);
    }
    big |= (unsigned)(mx >= kFp16Floor) << k;
    nz |= (unsigned)(mx > 0.f) << k;
  }
  if (active) {
    float4* yo = reinterpret_cast<float4*>(y + (size_t)t * H + c);
    yo[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    yo[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
  // A row of o whose values in this block's columns (up to 512) are all
  // below the fp16 floor, and not all zero.
  __shared__ unsigned red[2][kCombineThreads / 32];
  big = __reduce_or_sync(0xffffffffu, big);
  nz = __reduce_or_sync(0xffffffffu, nz);
  if ((threadIdx.x & 31) == 0) {
    red[0][threadIdx.x >> 5] = big;
    red[1][threadIdx.x >> 5] = nz;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned b = 0u, z = 0u;
#pragma unroll
    for (int w = 0; w < kCombineThreads / 32; ++w) {
      b |= red[0][w];
      z |= red[1][w];
    }
    if (z & ~b) flag_range(status);
  }
}

cudaError_t launch_combine(const Geometry& g, const __half* o, const int32_t* inv, const float* weights,
                           const float* gate, const int32_t* status, float* y, cudaStream_t stream) {
  dim3 grid(g.T, (g.H / 8 + kCombineThreads - 1) / kCombineThreads);
  combine_kernel<<<grid, kCombineThreads, 0, stream>>>(g.H, g.K, g.A, g.shared, o, inv, weights, gate, status, y);
  return cudaGetLastError();
}

}  // namespace bgmoe
