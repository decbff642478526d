// Fused decode MoE layer (T <= 4 tokens): router, top-k, routing tables,
// gate/up with fused dequantisation and SiLU, down projection and the
// weighted combine in one kernel, after a one-block prelude.
// [droneth.or.th Lily article, "Decode is bound by bandwidth more than
// compute": at batch 1 weights are barely reused, so the bound is the bytes
// moved; dothoosh.com "Perplexity Lily: 1.35x faster decode for Qwen3.6 on
// Apple silicon", "Decode optimisations", kernel fusion: chains of kernels
// fused so intermediates stay on chip.]
//
// Work split. An item is (expert slot s, 32 h columns n0..n0+31). The block
// that computes those h columns also computes their share of the down
// projection, W_down[:, n0..n0+31] h[n0..n0+31] for every output row, so h
// never leaves the block; each warp keeps its output rows' sums in registers
// across the block's items, and the blocks' sums meet once, at the end, in a
// fixed-order reduction. Slot 0 is the shared expert (every token; it needs
// no routing), slots 1.. the distinct routed experts in increasing index;
// item i goes to block i mod G, so blocks 0..I/32-1 start with a shared item.
//
// Phases of one block:
//   0  (before the programmatic-dependent-launch wait: weights only) the
//      warps load their router rows into registers; a block whose first item
//      is a shared one issues that item's weight copies;
//   R  the layer input is staged (fp32 for the router, fp16 in the permuted
//      K order for the MMAs; with the pre-norm join it is RMSNorm of the
//      residual row, never rounded to bf16); the router rows b + G*w give
//      logits, stored straight to global memory; a block with a shared item
//      computes the shared gate;
//   1  blocks with routed items poll the T logit rows until no entry holds
//      the sentinel the prelude wrote (no grid barrier: the wait is on the
//      data itself), select the top-k and build the slot table;
//   2  items: gate/up (the 16 warps split K), one block barrier, four warps
//      add the partial sums in a fixed order and form h = w silu(gate) up in
//      shared memory (the routing weight, or the shared gate, folded in),
//      another barrier, then every warp adds its W_down rows times h into its
//      register sums;
//   3  every block stores its sums and arrives on one counter; blocks owning
//      16 output rows wait for every arrival and add the blocks' sums in
//      block order: y (fp32), and the next residual row bf16(r + y) when
//      asked for.
//
// Weights reach shared memory by cp.async, each warp loading exactly the
// bytes it will use into a two-slot ring of its own (an item's gate/up part
// and its down part), so copies of the next part overlap the current part's
// arithmetic and no warp waits on another warp's copies.
//
// Products on mma.sync.m16n8k16 (fp16 operands, fp32 accumulation): 16
// weight rows x 8 token columns per instruction. Gate/up: the 16 MMA rows are
// 8 gate rows then the matching 8 up rows, so the lane holding gate(n, t)
// also holds up(n, t). Each lane dequantises whole code words into A
// fragments; one word unpacks as the pairs (k0,k4), (k1,k5), (k2,k6), (k3,k7),
// so x and h are kept in that K order inside every group of 8
// (0,4,1,5,2,6,3,7) and a B fragment is one 16-byte shared-memory load.
#include <atomic>

#include "kernels.h"
#include "tc_ptx.cuh"

namespace bgmoe {

constexpr int kDecWarps = 16;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kDecMaxA = kDecodeMaxTokens * kMaxTopK;
constexpr int kDecMaxSlots = kDecMaxA + 1;
constexpr int kItemCols = 32;                   // h columns per item
constexpr int kUnits = kItemCols / 8;           // MMA units of 8 h columns (8 gate + 8 up rows)
constexpr int kGuTaskBytes = 16 * 64 + 16 * 8;  // 16 code rows x 128 K, and their scale and bias pairs
constexpr int kDnTileBytes = 16 * 16 + 16 * 8;  // 16 W_down rows x 32 K, and their scale and bias pairs
constexpr int kMaxDnTiles = 8;                  // W_down tiles of 16 rows per warp (H <= 2048)
constexpr int kDnTilesPerTask = 4;              // W_down tiles per down task (two down tasks per item)
constexpr int kTaskBytes = kDnTilesPerTask * kDnTileBytes;  // one ring slot (>= kGuTaskBytes)
constexpr int kSlots = 6;                       // ring slots per warp: a whole item at H = 2048
static_assert(kGuTaskBytes <= kTaskBytes, "a gate/up task must fit a ring slot");
constexpr int kDecMaxH = kDecWarps * 16 * kMaxDnTiles;
constexpr int kGateWarp = kDecWarps - 1;        // computes the shared gate in blocks with a shared item
// The prelude fills the logits with this pattern; fp32 arithmetic never
// produces it (a NaN result is 0x7FFFFFFF), so a reader that sees any other
// value sees the router's output.
constexpr uint32_t kLogitSentinel = 0xFFFFFFFFu;

struct DecodeSmall {
  int ids[kDecMaxA];
  float w[kDecMaxA];
  float g[kDecodeMaxTokens];                   // shared gate per token
  float inv_rms[kDecodeMaxTokens];             // 1 / rms of each token's residual row (pre-norm join)
  int pos[kDecMaxA];                           // expert-sorted position of assignment a
  int slot_e[kDecMaxSlots];                    // expert of each slot (slot 0 = shared when present)
  int slot_n[kDecMaxSlots];                    // rows (tokens) of the slot
  int slot_row[kDecMaxSlots][kDecodeMaxTokens];
  float slot_wt[kDecMaxSlots][kDecodeMaxTokens];  // weight of token t in the slot (0: not routed there)
  const uint8_t* slot_src[kDecMaxSlots][6];    // gate/up codes, scales, biases; down codes, scales, biases
  int nslots;
  int failed;        // a logit poll or the final wait ran out
  int range;         // an fp16 operand (x or h) left the fp16 range
  unsigned nb;       // blocks holding down-projection sums
};

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ uint32_t ld_relaxed_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_f32(float* p, float v) {
  asm volatile("st.relaxed.gpu.global.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// Arrival on a counter: release orders the block's earlier writes (made
// visible to this thread by the preceding block barrier) before the add.
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}

// d += A * B with A 16x16 (row), B 16x8 (col), fp16 in, fp32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ __half2 bf16_h2(uint16_t bits16) {
  const __half h = __float2half_rn(bf16_bits_to_f32(bits16));
  return __halves2half2(h, h);
}

// The 32 K of one lane's 16-byte code chunk for its two rows (fragment rows g
// and g+8) against the matching B fragments xb[w] (permuted activations,
// 8 K per 16-byte word): 8 MMAs. With g = lane / 4 and c = lane % 4, MMA k
// slots 2c, 2c+1, 2c+8, 2c+9 of word w hold K offsets 8w + {0,4}, {1,5} (first
// MMA) and 8w + {2,6}, {3,7} (second), on A and B alike.
__device__ __forceinline__ void mma_chunk(float (&d)[4], const uint4& r0, const uint4& r1, __half2 s0, __half2 b0,
                                          __half2 s1, __half2 b1, const uint4 (&xb)[4]) {
  const uint32_t w0[4] = {r0.x, r0.y, r0.z, r0.w}, w1[4] = {r1.x, r1.y, r1.z, r1.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t p0[4], p1[4];
    tc::dequant8_f16(w0[w], s0, b0, p0);
    tc::dequant8_f16(w1[w], s1, b1, p1);
    mma_16816(d, p0[0], p1[0], p0[1], p1[1], xb[w].x, xb[w].y);
    mma_16816(d, p0[2], p1[2], p0[3], p1[3], xb[w].z, xb[w].w);
  }
}

// x[t] . row for the router: lane l holds bf16 elements 8 (l + 32 q) .. +7 of
// the row in w4[q]; the activations are fp32 in shared memory; fp32 sums in
// lane order, then a butterfly over the warp (every lane gets the result).
__device__ __forceinline__ float row_dot(const uint4 (&w4)[8], const float* xrow, int rvec, int lane) {
  float acc = 0.f;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int v = lane + 32 * q;
    if (v < rvec) {
      const uint32_t ww[4] = {w4[q].x, w4[q].y, w4[q].z, w4[q].w};
      const float4 xa = *reinterpret_cast<const float4*>(xrow + (size_t)v * 8);
      const float4 xc = *reinterpret_cast<const float4*>(xrow + (size_t)v * 8 + 4);
      const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xc.x, xc.y, xc.z, xc.w};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        acc = fmaf(bf16_bits_to_f32(ww[m] & 0xFFFFu), xv[2 * m], acc);
        acc = fmaf(bf16_bits_to_f32(ww[m] >> 16), xv[2 * m + 1], acc);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  return acc;
}

__device__ __forceinline__ void load_row(uint4 (&w4)[8], const uint16_t* row, int rvec, int lane) {
#pragma unroll
  for (int q = 0; q < 8; ++q)
    if (lane + 32 * q < rvec) w4[q] = ldg_nc_v4(row + (size_t)(lane + 32 * q) * 8);
}

__global__ void __launch_bounds__(kDecThreads, 1) decode_layer_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t dsm_raw[];
  __shared__ DecodeSmall S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g8 = lane >> 2, c4 = lane & 3;  // fragment coordinates
  const int T = a.T, H = a.H, I = a.I, E = a.E, K = a.K;
  const int A = T * K;
  const int sh = a.shared ? 1 : 0;
  const int G = gridDim.x, b = blockIdx.x;
  const int gpr = H / kGroup, igpr = I / kGroup;
  const int cpi = I / kItemCols;     // items per slot
  const int nkb = H / 128;           // gate/up K blocks of 128
  const int mtiles = H / 16;         // W_down tiles of 16 output rows
  const size_t slot_bytes = (size_t)a.slot_bytes;
  uint8_t* ring = dsm_raw + (size_t)warp * slot_bytes;              // this warp's ring of kSlots tasks
  __half* x16 = reinterpret_cast<__half*>(dsm_raw + a.x16_offset);   // [T][H] fp16, K-permuted
  float* xf = reinterpret_cast<float*>(dsm_raw + a.xf_offset);      // [T][H] fp32 layer input
  float* part = reinterpret_cast<float*>(dsm_raw + a.part_offset);   // [16 warps][4][32]
  __half* hs = reinterpret_cast<__half*>(dsm_raw + a.hs_offset);     // [8 tokens][32 columns]
  const uint64_t deadline = global_timer_ns() + (uint64_t)a.timeout_ns;

  if (tid == 0) {
    S.failed = 0;
    S.range = 0;
    S.nslots = sh;
    if (sh) {
      S.slot_e[0] = E;
      S.slot_n[0] = T;
      S.slot_src[0][0] = reinterpret_cast<const uint8_t*>(a.gu.s_codes);
      S.slot_src[0][1] = reinterpret_cast<const uint8_t*>(a.gu.s_scales);
      S.slot_src[0][2] = reinterpret_cast<const uint8_t*>(a.gu.s_biases);
      S.slot_src[0][3] = reinterpret_cast<const uint8_t*>(a.dn.s_codes);
      S.slot_src[0][4] = reinterpret_cast<const uint8_t*>(a.dn.s_scales);
      S.slot_src[0][5] = reinterpret_cast<const uint8_t*>(a.dn.s_biases);
    }
  }
  for (int i = tid; i < kDecMaxSlots * kDecodeMaxTokens; i += kDecThreads) (&S.slot_wt[0][0])[i] = 0.f;
  for (int i = tid; i < 8 * kItemCols / 2; i += kDecThreads) reinterpret_cast<uint32_t*>(hs)[i] = 0u;
  __syncthreads();

  // ---- this warp's tasks, in order: for each of the block's items, its
  // gate/up tasks (unit u = warp % 4, i.e. h columns n0 + 8u .. +7 as gate
  // rows and up rows, one K block kb = warp / 4 + 4 jj each), then two down
  // tasks (W_down tiles 16 (warp + 16 i) .. +15, i = 4 d .. 4 d + 3, columns
  // n0 .. n0 + 31). Each task's bytes are one cp.async group in one slot of
  // the warp's ring, so a task is computed as soon as its own bytes land.
  const int ngu = (warp >> 2) < nkb ? (nkb - (warp >> 2) + 3) / 4 : 0;  // gate/up tasks per item
  const int tpi = ngu + 2;                                                 // tasks per item
  auto issue_gu = [&](int item, int jj, uint8_t* td) {
    const int s = item / cpi, n0 = (item - s * cpi) * kItemCols;
    const uint8_t* codes = S.slot_src[s][0];
    const uint16_t* sc = reinterpret_cast<const uint16_t*>(S.slot_src[s][1]);
    const uint16_t* bi = reinterpret_cast<const uint16_t*>(S.slot_src[s][2]);
    const int u = warp & 3, kb = (warp >> 2) + 4 * jj;
#pragma unroll
    for (int q0 = 0; q0 < 64; q0 += 32) {  // 16 rows x 4 pieces of 16 bytes
      const int q = q0 + lane, r = q >> 2, piece = q & 3;
      const int row = r < 8 ? n0 + 8 * u + r : I + n0 + 8 * u + r - 8;
      cp_async16(td + r * 64 + piece * 16, codes + (size_t)row * (H / 2) + kb * 64 + piece * 16);
    }
    {  // scale and bias pairs of groups 2kb, 2kb+1 of the 16 rows
      const int r = lane >> 1, kind = lane & 1;
      const int row = r < 8 ? n0 + 8 * u + r : I + n0 + 8 * u + r - 8;
      cp_async4(td + 1024 + r * 8 + kind * 4, (kind ? bi : sc) + (size_t)row * gpr + 2 * kb);
    }
  };
  auto issue_dn = [&](int item, int dt, uint8_t* td) {
    const int s = item / cpi, c = item - s * cpi;
    const uint8_t* codes = S.slot_src[s][3];
    const uint16_t* sc = reinterpret_cast<const uint16_t*>(S.slot_src[s][4]);
    const uint16_t* bi = reinterpret_cast<const uint16_t*>(S.slot_src[s][5]);
    const int gp = (c >> 1) & ~1;  // the aligned pair of groups holding this item's group
#pragma unroll
    for (int q0 = 0; q0 < 16 * kDnTilesPerTask; q0 += 32) {  // 16 bytes of codes per row
      const int q = q0 + lane, i = q >> 4, r = q & 15, tile = warp + 16 * (kDnTilesPerTask * dt + i);
      if (tile < mtiles) cp_async16(td + i * kDnTileBytes + r * 16, codes + (size_t)(16 * tile + r) * (I / 2) + c * 16);
    }
#pragma unroll
    for (int q0 = 0; q0 < 32 * kDnTilesPerTask; q0 += 32) {  // scale and bias pairs
      const int q = q0 + lane, i = q >> 5, r = (q & 31) >> 1, kind = q & 1;
      const int tile = warp + 16 * (kDnTilesPerTask * dt + i);
      if (tile < mtiles)
        cp_async4(td + i * kDnTileBytes + 256 + r * 8 + kind * 4, (kind ? bi : sc) + (size_t)(16 * tile + r) * igpr + gp);
    }
  };
  int issued = 0;  // tasks issued by this warp (one cp.async group each)
  auto issue_task = [&](int k) {
    const int j = k / tpi, t = k - j * tpi;
    uint8_t* td = ring + (size_t)(k % kSlots) * kTaskBytes;
    if (t < ngu) issue_gu(b + G * j, t, td);
    else issue_dn(b + G * j, t - ngu, td);
    tc::cp_async_commit();
  };
  // Task k's bytes have landed (every later group may still be in flight),
  // and every lane of the warp sees them.
  auto wait_task = [&](int k) {
    switch (issued - k - 1) {
      case 0: tc::cp_async_wait<0>(); break;
      case 1: tc::cp_async_wait<1>(); break;
      case 2: tc::cp_async_wait<2>(); break;
      case 3: tc::cp_async_wait<3>(); break;
      case 4: tc::cp_async_wait<4>(); break;
      default: tc::cp_async_wait<kSlots - 1>(); break;
    }
    __syncwarp();
  };

  // ---- phase 0: weights only (they do not depend on the previous kernel).
  // Blocks with a shared item start its copies; the router rows go to the
  // other blocks (their x arrives without queueing behind those copies).
  const bool shared_first = sh && b < cpi;
  if (shared_first)
    for (; issued < tpi && issued < kSlots; ++issued) issue_task(issued);
  const int sfb = sh ? (cpi < G ? cpi : 0) : 0;  // blocks with a shared item (none hold router rows)
  const int RG = G - sfb;                        // router blocks
  const int rrows = E + sh, rvec = H / 8;
  const int rrow = b - sfb + RG * warp;
  const bool router_warp = b >= sfb && rrow < rrows && warp != kGateWarp;
  uint4 w4[8];
  if (router_warp) load_row(w4, rrow < E ? a.wr + (size_t)rrow * H : a.wsg, rvec, lane);
  if (shared_first && warp == kGateWarp) load_row(w4, a.wsg, rvec, lane);

  // x (and this call's workspace) may be the previous kernel's output: wait
  // for the prelude, which itself waits for the previous layer's kernels.
  grid_dep_wait();
  // x as fp32 (exact from bf16); with the pre-norm join, the sum of squares
  // of each token's residual row as well (fixed order: per thread, then the
  // warp butterfly, then the warps in order)
  float ss[kDecodeMaxTokens] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int t = 0; t < kDecodeMaxTokens; ++t)
    if (t < T)
      for (int v = tid; v < H / 8; v += kDecThreads) {
        const uint4 u = ldg_nc_v4(a.x + (size_t)t * H + (size_t)v * 8);
        const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
        float f[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          f[2 * q] = bf16_bits_to_f32(wv[q] & 0xFFFFu);
          f[2 * q + 1] = bf16_bits_to_f32(wv[q] >> 16);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) ss[t] = fmaf(f[q], f[q], ss[t]);
        float4* dst = reinterpret_cast<float4*>(xf + (size_t)t * H + (size_t)v * 8);
        dst[0] = make_float4(f[0], f[1], f[2], f[3]);
        dst[1] = make_float4(f[4], f[5], f[6], f[7]);
      }
  if (a.norm) {
#pragma unroll
    for (int t = 0; t < kDecodeMaxTokens; ++t) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss[t] += __shfl_xor_sync(0xffffffffu, ss[t], o);
      if (lane == 0) part[warp * kDecodeMaxTokens + t] = ss[t];
    }
  }
  __syncthreads();
  if (a.norm && tid < T) {
    float tot = 0.f;
    for (int w = 0; w < kDecWarps; ++w) tot += part[w * kDecodeMaxTokens + tid];
    S.inv_rms[tid] = 1.f / sqrtf(tot / (float)H + a.norm_eps);
  }
  __syncthreads();
  // the layer input: x (or RMSNorm(r) = r / rms(r) * gain, kept in fp32 for
  // the router), and its fp16 copy in the permuted K order for the MMAs
  for (int i = tid; i < T * H / 8; i += kDecThreads) {
    const int t = i / (H / 8);
    float4* src = reinterpret_cast<float4*>(xf + (size_t)i * 8);
    float f[8];
    const float4 fa = src[0], fc = src[1];
    f[0] = fa.x, f[1] = fa.y, f[2] = fa.z, f[3] = fa.w, f[4] = fc.x, f[5] = fc.y, f[6] = fc.z, f[7] = fc.w;
    if (a.norm) {
      const float s = S.inv_rms[t];
      uint4 gw = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);  // bf16 1.0 pairs
      if (a.norm_w) gw = ldg_nc_v4(a.norm_w + (size_t)(i - t * (H / 8)) * 8);
      const uint32_t gv[4] = {gw.x, gw.y, gw.z, gw.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        f[2 * q] = f[2 * q] * s * bf16_bits_to_f32(gv[q] & 0xFFFFu);
        f[2 * q + 1] = f[2 * q + 1] * s * bf16_bits_to_f32(gv[q] >> 16);
      }
      src[0] = make_float4(f[0], f[1], f[2], f[3]);
      src[1] = make_float4(f[4], f[5], f[6], f[7]);
    }
    bool big = false;
#pragma unroll
    for (int q = 0; q < 8; ++q) big |= fabsf(f[q]) >= 65520.f;  // becomes inf in fp16
    if (big) S.range = 1;
    const __half2 p0 = __floats2half2_rn(f[0], f[4]), p1 = __floats2half2_rn(f[1], f[5]);
    const __half2 p2 = __floats2half2_rn(f[2], f[6]), p3 = __floats2half2_rn(f[3], f[7]);
    uint4 o;
    o.x = *reinterpret_cast<const uint32_t*>(&p0);
    o.y = *reinterpret_cast<const uint32_t*>(&p1);
    o.z = *reinterpret_cast<const uint32_t*>(&p2);
    o.w = *reinterpret_cast<const uint32_t*>(&p3);
    reinterpret_cast<uint4*>(x16)[i] = o;
  }
  __syncthreads();

  // ---- phase R: router logits l[t][r] (r = E: the shared gate row), stored
  // for the other blocks; the shared gate itself where a shared item is here
  if (router_warp)
    for (int t = 0; t < T; ++t) {
      const float l = row_dot(w4, xf + (size_t)t * H, rvec, lane);
      if (lane == 0) st_relaxed_f32(a.logits + (size_t)t * (E + 1) + rrow, l);
    }
  if (shared_first && warp == kGateWarp)
    for (int t = 0; t < T; ++t) {
      const float l = row_dot(w4, xf + (size_t)t * H, rvec, lane);
      if (lane == 0) {
        S.g[t] = 1.f / (1.f + expf(-l));
        S.slot_wt[0][t] = S.g[t];
      }
    }
  // The next call's prelude may launch now: it waits for this grid to finish.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // ---- phase 1: top-k and slots, where this block may hold routed items.
  // A block whose only item is its shared one skips it (every item index
  // past its first is beyond the largest possible item count).
  const int max_items = ((A < E ? A : E) + sh) * cpi;
  const bool need_topk = !(shared_first && b + G >= max_items && b != G - 1);
  if (need_topk) {
    if (warp < T) {
      const float* lrow = a.logits + (size_t)warp * (E + 1);
      float lv[kMaxExperts / 32];
      float gl = 0.f;
      bool ok = false;
      while (true) {
#pragma unroll
        for (int j = 0; j < kMaxExperts / 32; ++j)
          lv[j] = __uint_as_float(ld_relaxed_u32(lrow + min(lane + 32 * j, E - 1)));
        gl = __uint_as_float(ld_relaxed_u32(lrow + (sh ? E : 0)));
        bool mine = __float_as_uint(gl) != kLogitSentinel;
#pragma unroll
        for (int j = 0; j < kMaxExperts / 32; ++j) mine &= __float_as_uint(lv[j]) != kLogitSentinel;
        if (__all_sync(0xffffffffu, mine)) {
          ok = true;
          break;
        }
        if (global_timer_ns() > deadline) break;
        __nanosleep(32);
      }
      if (ok) {
        int e;
        float w, g;
        warp_topk_select(lv, gl, a.bias, E, K, a.shared, lane, &e, &w, &g);
        if (lane < K) {
          S.ids[warp * K + lane] = e;
          S.w[warp * K + lane] = w;
        }
        if (lane == 0 && !shared_first) S.g[warp] = g;  // a shared-item block keeps its own (same bits)
      } else if (lane == 0) {
        S.failed = 1;
      }
    }
    __syncthreads();
    if (!S.failed && warp == 0) {
      // expert-sorted positions and slots (one lane per assignment)
      const bool live = lane < A;
      const int e = live ? S.ids[lane] : kMaxExperts + 1;
      const unsigned same = __match_any_sync(0xffffffffu, e) & __ballot_sync(0xffffffffu, live);
      const int before = __popc(same & lanemask_lt());  // earlier assignments of the same expert
      const bool first = live && before == 0;
      int lt = 0, dlt = 0;  // assignments / distinct experts with a lower index
      for (int q = 0; q < A; ++q) {
        const int vq = __shfl_sync(0xffffffffu, 2 * e + (first ? 1 : 0), q);
        const int lower = (vq >> 1) < e;
        lt += lower;
        dlt += lower & vq;
      }
      if (live) {
        const int slot = dlt + sh, tok = lane / K;
        S.pos[lane] = lt + before;
        S.slot_row[slot][before] = lt + before;
        S.slot_wt[slot][tok] = S.w[lane];
        if (first) {
          S.slot_e[slot] = e;
          S.slot_n[slot] = __popc(same);
        }
      }
      const int d = __popc(__ballot_sync(0xffffffffu, first));
      if (lane == 0) S.nslots = d + sh;
      if (sh && lane < T) {
        S.slot_row[0][lane] = A + lane;
        if (!shared_first) S.slot_wt[0][lane] = S.g[lane];
      }
      __syncwarp();
      for (int q = lane + sh; q < d + sh; q += 32) {  // weight addresses of the routed slots
        const int ex = S.slot_e[q];
        S.slot_src[q][0] = reinterpret_cast<const uint8_t*>(a.gu.codes + (size_t)ex * 2 * I * (H / 8));
        S.slot_src[q][1] = reinterpret_cast<const uint8_t*>(a.gu.scales + (size_t)ex * 2 * I * gpr);
        S.slot_src[q][2] = reinterpret_cast<const uint8_t*>(a.gu.biases + (size_t)ex * 2 * I * gpr);
        S.slot_src[q][3] = reinterpret_cast<const uint8_t*>(a.dn.codes + (size_t)ex * H * (I / 8));
        S.slot_src[q][4] = reinterpret_cast<const uint8_t*>(a.dn.scales + (size_t)ex * H * igpr);
        S.slot_src[q][5] = reinterpret_cast<const uint8_t*>(a.dn.biases + (size_t)ex * H * igpr);
      }
    }
    __syncthreads();
    if (S.failed && tid == 0) atomicExch(a.status, (int32_t)MOE_ERR_DEVICE_TIMEOUT);
  }
  const int items = S.failed ? 0 : S.nslots * cpi;
  const int nitems = b < items ? (items - b + G - 1) / G : 0;

  // The routing outputs (same definitions as moe_route), written by the last
  // block, which holds no item at T = 1.
  if (b == G - 1 && !S.failed) {
    for (int i = tid; i < A; i += kDecThreads) {
      a.ids[i] = S.ids[i];
      a.weights[i] = S.w[i];
      a.sorted[S.pos[i]] = i;
      a.inv[i] = S.pos[i];
    }
    if (a.shared)
      for (int t = tid; t < T; t += kDecThreads) a.gate[t] = S.g[t];
    for (int e = tid; e <= E + 1; e += kDecThreads) {
      int lt = 0, eq = 0;
      for (int q = 0; q < A; ++q) {
        lt += S.ids[q] < e;
        eq += S.ids[q] == e;
      }
      if (e <= E) a.counts[e] = e < E ? eq : (a.shared ? T : 0);
      a.offsets[e] = e <= E ? lt : A + (a.shared ? T : 0);
    }
    // one tile per expert in use (counts <= T <= 4 < block_m), then the shared tile
    const int d = S.nslots - sh;
    for (int s = tid; s < d; s += kDecThreads) {
      a.tile_expert[s] = S.slot_e[s + sh];
      a.tile_row0[s] = S.slot_row[s + sh][0];
      a.tile_rows[s] = S.slot_n[s + sh];
    }
    if (tid == 0) {
      if (a.shared) {
        a.tile_expert[d] = E;
        a.tile_row0[d] = A;
        a.tile_rows[d] = T;
      }
      *a.num_tiles = S.nslots;
    }
  }

  // ---- phase 2: this block's items b, b + G, ..., task by task
  float acc[kMaxDnTiles][4];
#pragma unroll
  for (int i = 0; i < kMaxDnTiles; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  const int ntasks = nitems * tpi;
  for (; issued < ntasks && issued < kSlots; ++issued) issue_task(issued);
  int k = 0;  // next task of this warp
  for (int j = 0; j < nitems; ++j) {
    const int item = b + G * j;
    const int s = item / cpi;
    float d[4] = {0.f, 0.f, 0.f, 0.f};
    for (int jj = 0; jj < ngu; ++jj, ++k) {
      wait_task(k);
      const uint8_t* t = ring + (size_t)(k % kSlots) * kTaskBytes;
      const int kb = (warp >> 2) + 4 * jj;
      uint4 xb[4];
      const __half* xrow = x16 + (size_t)(g8 < T ? g8 : 0) * H + kb * 128 + 32 * c4;
#pragma unroll
      for (int w = 0; w < 4; ++w)
        xb[w] = g8 < T ? *reinterpret_cast<const uint4*>(xrow + 8 * w) : make_uint4(0u, 0u, 0u, 0u);
      const uint4 cg = *reinterpret_cast<const uint4*>(t + g8 * 64 + c4 * 16);
      const uint4 cu = *reinterpret_cast<const uint4*>(t + (8 + g8) * 64 + c4 * 16);
      const uint16_t* sb = reinterpret_cast<const uint16_t*>(t + 1024);  // per row: scale pair, bias pair
      const int gs = c4 >> 1;  // this lane's 32 K lie in group 2kb + gs
      mma_chunk(d, cg, cu, bf16_h2(sb[g8 * 4 + gs]), bf16_h2(sb[g8 * 4 + 2 + gs]), bf16_h2(sb[(8 + g8) * 4 + gs]),
                bf16_h2(sb[(8 + g8) * 4 + 2 + gs]), xb);
      __syncwarp();  // the slot is read: refill it
      if (issued < ntasks) issue_task(issued++);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) part[(warp * 4 + r) * 32 + lane] = d[r];
    __syncthreads();
    if (warp < kUnits) {
      // unit u = warp: warps u, u+4, u+8, u+12 hold its partial sums (fixed
      // order). d0, d1: gate(column 8u + g, tokens 2c, 2c+1); d2, d3: up.
      float v[4];
#pragma unroll
      for (int r = 0; r < 4; ++r)
        v[r] = ((part[(warp * 4 + r) * 32 + lane] + part[((warp + 4) * 4 + r) * 32 + lane]) +
                part[((warp + 8) * 4 + r) * 32 + lane]) +
               part[((warp + 12) * 4 + r) * 32 + lane];
      const int pc = tc::perm8_pos(8 * warp + g8);
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int t = 2 * c4 + jj;
        if (t < T) {
          const __half hv = __float2half_rn(silu_f32(v[jj]) * v[2 + jj] * S.slot_wt[s][t]);
          if (__hisinf(hv)) S.range = 1;
          hs[t * kItemCols + pc] = hv;
        }
      }
    }
    __syncthreads();
    const uint4 hb = *reinterpret_cast<const uint4*>(hs + g8 * kItemCols + 8 * c4);  // token g (zero if >= T)
    const int gs = ((item - s * cpi) >> 1) & 1;  // this item's group within the loaded pair
#pragma unroll
    for (int dt = 0; dt < kMaxDnTiles / kDnTilesPerTask; ++dt, ++k) {
      wait_task(k);
      const uint8_t* td = ring + (size_t)(k % kSlots) * kTaskBytes;
#pragma unroll
      for (int i = 0; i < kDnTilesPerTask; ++i)
        if (warp + 16 * (kDnTilesPerTask * dt + i) < mtiles) {
          const uint8_t* t = td + i * kDnTileBytes;
          const uint32_t c0 = *reinterpret_cast<const uint32_t*>(t + g8 * 16 + c4 * 4);
          const uint32_t c1 = *reinterpret_cast<const uint32_t*>(t + (8 + g8) * 16 + c4 * 4);
          const uint16_t* sb = reinterpret_cast<const uint16_t*>(t + 256);
          uint32_t p0[4], p1[4];
          tc::dequant8_f16(c0, bf16_h2(sb[g8 * 4 + gs]), bf16_h2(sb[g8 * 4 + 2 + gs]), p0);
          tc::dequant8_f16(c1, bf16_h2(sb[(8 + g8) * 4 + gs]), bf16_h2(sb[(8 + g8) * 4 + 2 + gs]), p1);
          float (&ac)[4] = acc[kDnTilesPerTask * dt + i];
          mma_16816(ac, p0[0], p1[0], p0[1], p1[1], hb.x, hb.y);
          mma_16816(ac, p0[2], p1[2], p0[3], p1[3], hb.z, hb.w);
        }
      __syncwarp();
      if (issued < ntasks) issue_task(issued++);
    }
  }
  tc::cp_async_wait_all();  // no copy into this block's shared memory outlives it

  // ---- phase 3: this block's sums, one arrival, the fixed-order reduction
  if (nitems > 0) {
    float* P = a.partial + (size_t)b * T * H;
#pragma unroll
    for (int i = 0; i < kMaxDnTiles; ++i) {
      const int tile = warp + 16 * i;
      if (tile < mtiles) {
        const int m0 = 16 * tile + g8, t0 = 2 * c4;
        if (t0 < T) {
          P[(size_t)t0 * H + m0] = acc[i][0];
          P[(size_t)t0 * H + m0 + 8] = acc[i][2];
        }
        if (t0 + 1 < T) {
          P[(size_t)(t0 + 1) * H + m0] = acc[i][1];
          P[(size_t)(t0 + 1) * H + m0 + 8] = acc[i][3];
        }
      }
    }
  }
  // Each warp arrives once its own sums are stored (warp 0 also counts the
  // block among those holding sums); no block barrier on this path.
  __syncwarp();
  if (lane == 0 && b != a.stall_block)
    red_release_add(a.bar, 1u + (warp == 0 && nitems > 0 ? (1u << 16) : 0u));
  __syncthreads();
  if (tid == 0 && S.range) atomicCAS(a.status, 0, (int32_t)MOE_ERR_RANGE);
  if (b >= mtiles) return;  // no output rows here
  if (tid == 0) {
    unsigned v = 0;
    while (((v = ld_acquire_u32(a.bar)) & 0xFFFFu) < (unsigned)(G * kDecWarps)) {
      if (global_timer_ns() > deadline) {
        S.failed = 1;
        break;
      }
      __nanosleep(32);
    }
    S.nb = v >> 16;
    if (S.failed) atomicExch(a.status, (int32_t)MOE_ERR_DEVICE_TIMEOUT);
  }
  __syncthreads();
  if (S.failed) return;
  const int nb = (int)S.nb;
  float* red = reinterpret_cast<float*>(dsm_raw);  // [32][T][16] (the ring is no longer in use)
  const int ml = tid & 15, bl = tid >> 4;
  for (int slice = b; slice < mtiles; slice += G) {
    const int m = 16 * slice + ml;
    float v[kDecodeMaxTokens] = {0.f, 0.f, 0.f, 0.f};
    constexpr int kMaxPer = (kMaxDecodeBlocks + 31) / 32;
    float pv[kMaxPer][kDecodeMaxTokens];
#pragma unroll
    for (int k = 0; k < kMaxPer; ++k)  // every load before any use
#pragma unroll
      for (int t = 0; t < kDecodeMaxTokens; ++t)
        pv[k][t] = (bl + 32 * k < nb && t < T) ? __ldcg(a.partial + ((size_t)(bl + 32 * k) * T + t) * H + m) : 0.f;
#pragma unroll
    for (int k = 0; k < kMaxPer; ++k)
#pragma unroll
      for (int t = 0; t < kDecodeMaxTokens; ++t) v[t] += pv[k][t];
#pragma unroll
    for (int t = 0; t < kDecodeMaxTokens; ++t)
      if (t < T) red[(bl * T + t) * 16 + ml] = v[t];
    __syncthreads();
    if (tid < 16 * T) {
      const int t = tid >> 4;
      float y = 0.f;
      for (int q = 0; q < 32; ++q) y += red[(q * T + t) * 16 + ml];  // fixed order
      a.y[(size_t)t * H + m] = y;
      if (a.x_next) {
        const float xv = bf16_bits_to_f32(a.x[(size_t)t * H + m]);
        a.x_next[(size_t)t * H + m] = __bfloat16_as_ushort(__float2bfloat16_rn(xv + y));
      }
    }
    __syncthreads();
  }
}

namespace {
int sm_count(int dev) {
  static std::atomic<int> sms[kMaxDevices];
  if (dev < 0 || dev >= kMaxDevices) return 0;
  int v = sms[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    sms[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

constexpr size_t kDecDynamicLimit = 220 * 1024;  // 227 KB per block minus the static part

// Dynamic shared memory: 16 warps x kSlots task slots, x16 fp16 and x fp32
// [T][H], the partial sums of the gate/up reduction, h of one item.
struct DecodeLayout {
  size_t slot_bytes, x16_offset, xf_offset, part_offset, hs_offset, total;
};

DecodeLayout decode_layout(const Geometry& g) {
  DecodeLayout L{};
  L.slot_bytes = (size_t)kSlots * kTaskBytes;  // one warp's ring
  const size_t xb = ((size_t)g.T * g.H * 2 + 127) & ~size_t(127);
  L.x16_offset = (size_t)kDecWarps * L.slot_bytes;
  L.xf_offset = L.x16_offset + xb;
  L.part_offset = L.xf_offset + 2 * xb;
  L.hs_offset = L.part_offset + (size_t)kDecWarps * 4 * 32 * 4;
  L.total = L.hs_offset + 8 * kItemCols * 2;
  const size_t red = (size_t)32 * kDecodeMaxTokens * 16 * 4;  // the final reduction reuses the ring
  if (L.total < red) L.total = red;
  return L;
}
}  // namespace

// One block per SM, every block resident (blocks wait for each other's
// logits and sums); K of gate/up in whole 128-wide blocks, H at most 2048
// (each warp keeps at most 8 tiles of output sums in registers), I in whole
// 128-wide blocks, enough router warps (15 per block without a shared item)
// for the E (+ 1) router rows.
bool decode_supported(const Geometry& g) {
  int dev = 0;
  if (g.T < 1 || g.T > kDecodeMaxTokens || g.H % 128 || g.H > kDecMaxH || g.I % 128 ||
      cudaGetDevice(&dev) != cudaSuccess)
    return false;
  const int sms = sm_count(dev);
  if (sms <= 0 || sms > kMaxDecodeBlocks) return false;
  // router rows live on the blocks without a shared item, 15 warps each
  const int cpi = g.I / kItemCols, sfb = g.shared ? (cpi < sms ? cpi : 0) : 0;
  if (g.E + g.shared > (sms - sfb) * (kDecWarps - 1)) return false;
  return decode_layout(g).total <= kDecDynamicLimit;
}

// Fills the call's logits with the sentinel and clears the arrival counter
// and the status word. Launched with programmatic dependent launch, it starts
// while the previous kernel on the stream (often the previous layer's decode
// kernel) is finishing, lets the decode kernel start at once, and waits for
// the previous kernel to complete before it writes; the decode kernel waits
// for this grid before it reads x, the logits or the counter.
__global__ void decode_prelude_kernel(float* logits, int n_logits, unsigned int* bar, int32_t* status) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  for (int i = threadIdx.x; i < n_logits; i += blockDim.x) reinterpret_cast<uint32_t*>(logits)[i] = kLogitSentinel;
  if (threadIdx.x == 0) {
    bar[0] = 0u;
    *status = 0;
  }
}

cudaError_t launch_decode(const DecodeArgs& args_in, const Geometry& g, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int grid = sm_count(dev);
  if (grid <= 0 || grid > kMaxDecodeBlocks) return cudaErrorInvalidDevice;
  const DecodeLayout L = decode_layout(g);
  static SmemLimitMemo smem_memo;
  e = ensure_smem(decode_layer_kernel, L.total, &smem_memo);
  if (e != cudaSuccess) return e;
  // Every block must be resident at once: one block per SM must fit.
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_layer_kernel, kDecThreads, L.total);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
  {
    cudaLaunchConfig_t pc{};
    pc.gridDim = dim3(1);
    pc.blockDim = dim3(256);
    pc.stream = stream;
    cudaLaunchAttribute pa[1];
    pa[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pa[0].val.programmaticStreamSerializationAllowed = 1;
    pc.attrs = pa;
    pc.numAttrs = 1;
    e = cudaLaunchKernelEx(&pc, decode_prelude_kernel, args_in.logits, g.T * (g.E + 1), args_in.bar, args_in.status);
    if (e != cudaSuccess) return e;
  }
  DecodeArgs args = args_in;
  args.slot_bytes = (long long)L.slot_bytes;
  args.x16_offset = (long long)L.x16_offset;
  args.xf_offset = (long long)L.xf_offset;
  args.part_offset = (long long)L.part_offset;
  args.hs_offset = (long long)L.hs_offset;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_layer_kernel, args);
}

}  // namespace bgmoe
