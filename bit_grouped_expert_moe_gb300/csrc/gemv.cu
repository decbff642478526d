// Grouped expert GEMV with fused 4-bit dequantisation, for few tokens per
// expert (decode: T = 1..4), over the block map of the routing kernel.
// [dothoosh.com "Perplexity Lily: 1.35x faster decode for Qwen3.6 on Apple
// silicon", "Prefill optimisations", fused dequantisation: 64 weights share
// one bf16 scale and bias, weights are rebuilt inside the expert product and
// accumulated in FP32; droneth.or.th's Lily article, "Decode is bound by
// bandwidth more than compute": at batch 1 weights are barely reused, so the
// bound is the bytes moved.]
//
// Gate/up: one warp computes one h column n of one tile: it streams the gate
// row n and the up row I+n (16-byte loads per lane, all issued before any
// arithmetic), dequantises in fp32 (W = scale * q + bias, exact in fp32) and
// dots them with up to kTokChunk token rows held in shared memory; a
// warp-shuffle reduction finishes the sums and h = silu(gate) * up is stored as
// fp16. Down: a row of W_down has I/8 words, so lanes split into groups of
// L lanes per output row (the largest power of two <= min(32, I/32)).
//
// Tiles past *num_tiles (the grid is sized by the host-side upper bound, the
// true count lives on the device) return at once, as do all blocks after a
// device error.
#include "kernels.h"

namespace bgmoe {

constexpr int kGemvWarps = 8;
constexpr int kTokChunk = 4;   // token rows per pass over the weights
constexpr int kPad = 36;       // floats per 32-value chunk of a staged row

// Stage token rows (activations) as fp32 chunks of 32 values padded to 36,
// so that lane l reading chunk l with 16-byte loads is bank-conflict free.
__device__ __forceinline__ float to_f32(uint16_t bf16_bits) { return bf16_bits_to_f32(bf16_bits); }
__device__ __forceinline__ float to_f32(__half v) { return __half2float(v); }

template <typename Src>
__device__ __forceinline__ void stage_rows(float* dst, const Src* src, const int* rows_src, int n, int len) {
  const int chunks = len / 32;
  for (int i = threadIdx.x; i < n * len; i += blockDim.x) {
    const int j = i / len, k = i - j * len;
    dst[(j * chunks + (k >> 5)) * kPad + (k & 31)] = to_f32(src[(size_t)rows_src[j] * len + k]);
  }
}

// Lanes per output row of the down projection: the largest power of two
// <= min(32, I/32), so that xor-shuffle reductions stay inside the group.
__host__ __device__ __forceinline__ int down_lanes(int I) {
  const int nvec = I / 32;
  int L = 1;
  while (L * 2 <= nvec && L * 2 <= 32) L *= 2;
  return L;
}

__device__ __forceinline__ void dot32(const uint4 c, float s, float b, const float* xrow, float& acc) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const float4 x0 = *reinterpret_cast<const float4*>(xrow + 8 * m);
    const float4 x1 = *reinterpret_cast<const float4*>(xrow + 8 * m + 4);
    const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
    for (int q = 0; q < 8; ++q) acc = fmaf(fmaf(s, (float)((w[m] >> (4 * q)) & 15u), b), xv[q], acc);
  }
}

template <int kMaxIt>  // 16-byte loads per lane per weight row: ceil(H / 1024)
__global__ void __launch_bounds__(kGemvWarps * 32)
gemv_gate_up_kernel(int H, int I, int E, int K, int A, int rows_total, const uint16_t* __restrict__ x, ExpertArgs w,
                    TileArgs t, __half* __restrict__ h) {
  extern __shared__ __align__(16) float xs[];  // [kTokChunk][H/32][kPad]
  __shared__ int tok_s[kTokChunk];
  const int tile = blockIdx.x;
  if (block_failed(t.status) || tile >= *t.num_tiles) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = A / K;
  const int e = checked(t.tile_expert[tile], 0, E, t.status);
  const int nr = checked(t.tile_rows[tile], 1, rows_total, t.status);  // rows of h: A (+ T with a shared expert)
  const int r0 = checked(t.tile_row0[tile], 0, rows_total - nr, t.status);
  const bool sh = e == E;
  const size_t mat_words = (size_t)2 * I * (H / 8), mat_groups = (size_t)2 * I * (H / kGroup);
  const uint32_t* codes = sh ? w.s_codes : w.codes + (size_t)e * mat_words;
  const uint16_t* scales = sh ? w.s_scales : w.scales + (size_t)e * mat_groups;
  const uint16_t* biases = sh ? w.s_biases : w.biases + (size_t)e * mat_groups;
  const int n = blockIdx.y * kGemvWarps + warp;
  const int nvec = H / 32, chunks = H / 32;
  const int gpr = H / kGroup;

  // Issue this warp's weight loads first (2 rows x H/2 bytes).
  uint4 cg[kMaxIt], cu[kMaxIt];
  float sg[kMaxIt], bg[kMaxIt], su[kMaxIt], bu[kMaxIt];
#pragma unroll
  for (int it = 0; it < kMaxIt; ++it) {
    const int v = lane + 32 * it;
    if (v < nvec) {
      cg[it] = ldg_nc_v4(codes + (size_t)n * (H / 8) + 4 * v);
      cu[it] = ldg_nc_v4(codes + (size_t)(I + n) * (H / 8) + 4 * v);
      sg[it] = bf16_bits_to_f32(__ldg(scales + (size_t)n * gpr + v / 2));
      bg[it] = bf16_bits_to_f32(__ldg(biases + (size_t)n * gpr + v / 2));
      su[it] = bf16_bits_to_f32(__ldg(scales + (size_t)(I + n) * gpr + v / 2));
      bu[it] = bf16_bits_to_f32(__ldg(biases + (size_t)(I + n) * gpr + v / 2));
    }
  }

  for (int c0 = 0; c0 < nr; c0 += kTokChunk) {
    const int nc = min(kTokChunk, nr - c0);
    __syncthreads();
    if (threadIdx.x < nc) {
      const int r = r0 + c0 + threadIdx.x;
      tok_s[threadIdx.x] = checked(r < A ? t.sorted[r] / K : r - A, 0, T - 1, t.status);
    }
    __syncthreads();
    stage_rows(xs, x, tok_s, nc, H);
    __syncthreads();
    float ag[kTokChunk] = {0.f, 0.f, 0.f, 0.f}, au[kTokChunk] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int it = 0; it < kMaxIt; ++it) {
      const int v = lane + 32 * it;
      if (v < nvec) {
#pragma unroll
        for (int j = 0; j < kTokChunk; ++j) {
          if (j < nc) {
            const float* xr = xs + (j * chunks + v) * kPad;
            dot32(cg[it], sg[it], bg[it], xr, ag[j]);
            dot32(cu[it], su[it], bu[it], xr, au[j]);
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kTokChunk; ++j) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        ag[j] += __shfl_xor_sync(0xffffffffu, ag[j], o);
        au[j] += __shfl_xor_sync(0xffffffffu, au[j], o);
      }
    }
    bool big = false, nz = false;
    if (lane < nc) {
      float g = ag[0], u = au[0];
#pragma unroll
      for (int j = 1; j < kTokChunk; ++j)
        if (lane == j) { g = ag[j]; u = au[j]; }
      const float hf = silu_f32(g) * u;
      if (fabsf(hf) >= 65520.f) flag_range(t.status);  // inf in fp16
      big = fabsf(hf) >= kFp16Floor;
      nz = hf != 0.f;
      h[(size_t)(r0 + c0 + lane) * I + n] = __float2half_rn(hf);
    }
    // The block's kGemvWarps columns of h for these tokens, all below the
    // fp16 floor (o is checked row by row where it is combined).
    const int any_big = __syncthreads_or(big), any_nz = __syncthreads_or(nz);
    if (threadIdx.x == 0 && any_nz && !any_big) flag_range(t.status);
  }
}

// Down projection: o[r][m] = sum_n h[r][n] * W_down[m][n].
__global__ void __launch_bounds__(kGemvWarps * 32)
gemv_down_kernel(int H, int I, int E, int rows_total, int rows_per_block, const __half* __restrict__ hbuf, ExpertArgs w,
                 TileArgs t, __half* __restrict__ o) {
  extern __shared__ __align__(16) float hs[];  // [kTokChunk][I/32][kPad]
  __shared__ int row_s[kTokChunk];
  const int tile = blockIdx.x;
  if (block_failed(t.status) || tile >= *t.num_tiles) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = checked(t.tile_expert[tile], 0, E, t.status);
  const int nr = checked(t.tile_rows[tile], 1, rows_total, t.status);  // rows of h and o: A (+ T)
  const int r0 = checked(t.tile_row0[tile], 0, rows_total - nr, t.status);
  const bool sh = e == E;
  const size_t mat_words = (size_t)H * (I / 8), mat_groups = (size_t)H * (I / kGroup);
  const uint32_t* codes = sh ? w.s_codes : w.codes + (size_t)e * mat_words;
  const uint16_t* scales = sh ? w.s_scales : w.scales + (size_t)e * mat_groups;
  const uint16_t* biases = sh ? w.s_biases : w.biases + (size_t)e * mat_groups;
  const int nvec = I / 32, chunks = I / 32, gpr = I / kGroup;
  const int L = down_lanes(I);           // lanes per output row
  const int R = 32 / L;                  // output rows per warp per pass
  const int sub = lane % L, rw = lane / L;
  const int its = (nvec + L - 1) / L;    // 16-byte loads per lane per row
  const int m_first = blockIdx.y * rows_per_block;

  for (int c0 = 0; c0 < nr; c0 += kTokChunk) {
    const int nc = min(kTokChunk, nr - c0);
    __syncthreads();
    if (threadIdx.x < nc) row_s[threadIdx.x] = r0 + c0 + threadIdx.x;
    __syncthreads();
    stage_rows(hs, hbuf, row_s, nc, I);
    __syncthreads();
    for (int mb = warp * R; mb < rows_per_block; mb += kGemvWarps * R) {
      const int m = m_first + mb + rw;
      float acc[kTokChunk] = {0.f, 0.f, 0.f, 0.f};
      if (m < H) {
        constexpr int kMaxIt = 4;  // I <= 4096
        uint4 c[kMaxIt];
        float s[kMaxIt], b[kMaxIt];
#pragma unroll
        for (int it = 0; it < kMaxIt; ++it) {
          if (it < its && sub + L * it < nvec) {
            const int v = sub + L * it;
            c[it] = ldg_nc_v4(codes + (size_t)m * (I / 8) + 4 * v);
            s[it] = bf16_bits_to_f32(__ldg(scales + (size_t)m * gpr + v / 2));
            b[it] = bf16_bits_to_f32(__ldg(biases + (size_t)m * gpr + v / 2));
          }
        }
#pragma unroll
        for (int it = 0; it < kMaxIt; ++it) {
          if (it < its && sub + L * it < nvec) {
            const int v = sub + L * it;
#pragma unroll
            for (int j = 0; j < kTokChunk; ++j)
              if (j < nc) dot32(c[it], s[it], b[it], hs + (j * chunks + v) * kPad, acc[j]);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kTokChunk; ++j) {
        for (int off = L >> 1; off > 0; off >>= 1) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], off);
      }
      if (m < H) {
#pragma unroll
        for (int j = 0; j < kTokChunk; ++j)
          if (j < nc && (j % L) == sub) {
            if (fabsf(acc[j]) >= 65520.f) flag_range(t.status);  // inf in fp16
            o[(size_t)(r0 + c0 + j) * H + m] = __float2half_rn(acc[j]);
          }
      }
    }
  }
}

template <int kIt>
static cudaError_t launch_gate_up_it(const Geometry& g, const uint16_t* x, const ExpertArgs& w, const TileArgs& t,
                                     __half* h, size_t smem, cudaStream_t stream) {
  static SmemLimitMemo smem_memo;
  cudaError_t e = ensure_smem(gemv_gate_up_kernel<kIt>, smem, &smem_memo);
  if (e != cudaSuccess) return e;
  dim3 grid(g.max_tiles, g.I / kGemvWarps);
  gemv_gate_up_kernel<kIt><<<grid, kGemvWarps * 32, smem, stream>>>(g.H, g.I, g.E, g.K, g.A, g.rows, x, w, t, h);
  return cudaGetLastError();
}

cudaError_t launch_gemv_gate_up(const Geometry& g, const uint16_t* x, const ExpertArgs& w, const TileArgs& t,
                                __half* h, cudaStream_t stream) {
  const size_t smem = (size_t)kTokChunk * g.H * kPad / 32 * sizeof(float);
  const int its = (g.H / 32 + 31) / 32;
  if (its <= 1) return launch_gate_up_it<1>(g, x, w, t, h, smem, stream);
  if (its <= 2) return launch_gate_up_it<2>(g, x, w, t, h, smem, stream);
  if (its <= 4) return launch_gate_up_it<4>(g, x, w, t, h, smem, stream);
  return launch_gate_up_it<8>(g, x, w, t, h, smem, stream);
}

cudaError_t launch_gemv_down(const Geometry& g, const __half* h, const ExpertArgs& w, const TileArgs& t,
                             __half* o, cudaStream_t stream) {
  const int L = down_lanes(g.I);
  const int R = 32 / L;
  const int rows_per_block = (kGemvWarps * R > 64) ? kGemvWarps * R : 64;
  const size_t smem = (size_t)kTokChunk * g.I * kPad / 32 * sizeof(float);
  static SmemLimitMemo smem_memo;
  cudaError_t e = ensure_smem(gemv_down_kernel, smem, &smem_memo);
  if (e != cudaSuccess) return e;
  dim3 grid(g.max_tiles, (g.H + rows_per_block - 1) / rows_per_block);
  gemv_down_kernel<<<grid, kGemvWarps * 32, smem, stream>>>(g.H, g.I, g.E, g.rows, rows_per_block, h, w, t, o);
  return cudaGetLastError();
}

}  // namespace bgmoe
