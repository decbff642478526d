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
  if (device_failed(status)) return;
  const int t = blockIdx.x;
  const int c = (blockIdx.y * kCombineThreads + threadIdx.x) * 8;
  if (c >= H) return;
  // Every load of the token goes out before any is used: the K row
  // indices and weights, then the K + 1 rows of o (the shared row last).
  int rows[kMaxTopK + 1];
  float wt[kMaxTopK + 1];
#pragma unroll
  for (int k = 0; k < kMaxTopK; ++k) {
    rows[k] = k < K ? inv[(size_t)t * K + k] : 0;
    wt[k] = k < K ? weights[(size_t)t * K + k] : 0.f;
  }
  rows[kMaxTopK] = A + t;
  wt[kMaxTopK] = shared ? gate[t] : 0.f;
  uint4 v[kMaxTopK + 1];
#pragma unroll
  for (int k = 0; k <= kMaxTopK; ++k)
    if (k < K || (k == kMaxTopK && shared)) v[k] = *reinterpret_cast<const uint4*>(o + (size_t)rows[k] * H + c);
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
  for (int k = 0; k <= kMaxTopK; ++k) {
    if (!(k < K || (k == kMaxTopK && shared))) continue;
    const __half2* h2 = reinterpret_cast<const __half2*>(&v[k]);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(h2[i]);
      acc[2 * i] = fmaf(wt[k], f.x, acc[2 * i]);
      acc[2 * i + 1] = fmaf(wt[k], f.y, acc[2 * i + 1]);
    }
  }
  float4* yo = reinterpret_cast<float4*>(y + (size_t)t * H + c);
  yo[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  yo[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

cudaError_t launch_combine(const Geometry& g, const __half* o, const int32_t* inv, const float* weights,
                           const float* gate, const int32_t* status, float* y, cudaStream_t stream) {
  dim3 grid(g.T, (g.H / 8 + kCombineThreads - 1) / kCombineThreads);
  combine_kernel<<<grid, kCombineThreads, 0, stream>>>(g.H, g.K, g.A, g.shared, o, inv, weights, gate, status, y);
  return cudaGetLastError();
}

}  // namespace bgmoe
