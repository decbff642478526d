// Fused decode MoE layer (T <= 4 tokens): router, top-k, routing tables,
// gate/up with fused dequantisation and SiLU, down projection and the
// weighted combine in one kernel, after a one-block prelude.
// [droneth.or.th Lily article, "Decode is bound by bandwidth more than
// compute": at batch 1 weights are barely reused, so the bound is the bytes
// moved; dothoosh.com "Perplexity Lily: 1.35x faster decode for Qwen3.6 on
// Apple silicon", "Decode optimisations", kernel fusion: chains of kernels
// fused so intermediates stay on chip.]
//
// Work split. Slot 0 is the shared expert (every token; it needs no
// routing), slots 1.. the distinct routed experts in increasing index.
//   gate/up: an item is (slot s, 32 h columns n0..n0+31); item i goes to
//     block i mod G, so blocks 0..I/32-1 start with a shared item. The block
//     forms h = w silu(gate) up for its columns (the routing weight, or the
//     shared gate, folded in) and stores it to the workspace.
//   down: block b owns output rows 16b..16b+15 (W_down rows of every slot:
//     4 KB of codes per slot, contiguous). It reads the h of the slots,
//     polling each 16-byte piece until it no longer holds the sentinel the
//     prelude wrote, and adds the products into per-warp sums; the 16 warps'
//     sums are added in a fixed order into y, so results are bit-identical
//     run to run.
// No grid-wide barrier and no counters: the router's logits and h are both
// exchanged through sentinels the prelude writes (a reader polls the data
// itself, one L2 round trip once the data is there).
//
// Tasks. Every unit of work is 16 weight rows x 128 K: a gate/up task (8
// gate rows and the matching 8 up rows of one 8-column unit, one K block)
// or a down task (16 W_down rows, one 128-wide block of h columns). Each
// warp streams its tasks through a ring of kSlots shared-memory slots, one
// cp.async group per task, and computes a task as soon as its bytes land;
// the copies of the next tasks overlap the arithmetic. The shared expert's
// down tasks are copied into a buffer of their own before the kernel waits
// for its predecessor (their weights need no routing).
//
// Phases of one block:
//   0  (before the programmatic-dependent-launch wait: weights only) router
//      rows into registers on the blocks without a shared item; the shared
//      item's gate/up tasks and the shared down tasks go out;
//   R  the layer input is staged (fp32 for the router, fp16 in the permuted
//      K order for the MMAs; with the pre-norm join it is RMSNorm of the
//      residual row, never rounded to bf16); logits are written to L2 by
//      atomic exchange; a block with a shared item computes the shared gate
//      and its shared item;
//   1  blocks with routed work poll the T logit rows until no entry holds
//      the sentinel, select the top-k and build the slot table;
//   2  routed gate/up items;
//   3  down: the slots' h polled into shared memory in batches, then the
//      fixed-order sum into y and the next residual row bf16(r + y) when
//      asked for.
//
// Products on mma.sync.m16n8k16 (fp16 operands, fp32 accumulation): 16
// weight rows x 8 token columns per instruction. Each lane dequantises whole
// code words into A fragments; one word unpacks as the pairs (k0,k4),
// (k1,k5), (k2,k6), (k3,k7), so x and h are kept in that K order inside every
// group of 8 (0,4,1,5,2,6,3,7) and a B fragment is one 16-byte load.
#include <atomic>

#include "kernels.h"
#include "tc_ptx.cuh"

namespace bgmoe {

constexpr int kDecWarps = 16;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kDecMaxA = kDecodeMaxTokens * kMaxTopK;
constexpr int kItemCols = 32;                 // h columns per gate/up item
constexpr int kUnits = kItemCols / 8;         // MMA units of 8 h columns (8 gate + 8 up rows)
constexpr int kTaskBytes = 16 * 64 + 16 * 8;  // 16 code rows x 128 K, their scale and bias pairs
constexpr int kSlots = 6;                     // ring slots per warp
constexpr int kDecMaxI = 1024;                // shared down tasks: one per warp at most (I / 128 <= 8)
constexpr int kGateWarp = kDecWarps - 1;      // computes the shared gate in blocks with a shared item
// The prelude fills the logits with this pattern; fp32 arithmetic never
// produces it (a NaN result is 0x7FFFFFFF), so a reader that sees any other
// value sees the router's output.
constexpr uint32_t kLogitSentinel = 0xFFFFFFFFu;
// The prelude fills the h of every slot a call can use with this fp16
// pattern (a NaN that float-to-half conversion never produces; a computed
// value with these bits is stored as another NaN and reported), so a reader
// that finds no sentinel in a piece of h reads the producer's values.
constexpr uint16_t kHSentinel = 0xFFFFu;
static_assert(kDecodeMaxSlots >= kDecMaxA + 1, "slot table");

struct DecodeSmall {
  int ids[kDecMaxA];
  float w[kDecMaxA];
  float g[kDecodeMaxTokens];                   // shared gate per token
  int pos[kDecMaxA];                           // expert-sorted position of assignment a
  int slot_e[kDecodeMaxSlots];                 // expert of each slot (slot 0 = shared when present)
  int slot_n[kDecodeMaxSlots];                 // rows (tokens) of the slot
  int slot_row[kDecodeMaxSlots][kDecodeMaxTokens];
  float slot_wt[kDecodeMaxSlots][kDecodeMaxTokens];  // weight of token t in the slot (0: not routed there)
  const uint8_t* slot_src[kDecodeMaxSlots][6];  // gate/up codes, scales, biases; down codes, scales, biases
  int nslots;
  int failed;        // a logit poll or an h poll ran out
  int range;         // an fp16 operand (x or h) left the fp16 range
};

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint32_t ld_relaxed_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// 16 bytes of h read past L1 (at the GPU scope, fresh on every call).
__device__ __forceinline__ uint4 ld_relaxed_v4(const void* p) {
  uint4 v;
  asm volatile("ld.relaxed.gpu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

// Whether any of the 8 halves of a piece of h still holds the sentinel.
__device__ __forceinline__ bool has_h_sentinel(const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  bool any = false;
#pragma unroll
  for (int i = 0; i < 4; ++i) any |= (w[i] & 0xFFFFu) == kHSentinel || (w[i] >> 16) == kHSentinel;
  return any;
}

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}

// Waits until at most n of this thread's most recent cp.async groups are
// pending (every older group has landed).
__device__ __forceinline__ void cp_async_wait_dyn(int n) {
  switch (n <= 0 ? 0 : n) {
    case 0: tc::cp_async_wait<0>(); break;
    case 1: tc::cp_async_wait<1>(); break;
    case 2: tc::cp_async_wait<2>(); break;
    case 3: tc::cp_async_wait<3>(); break;
    case 4: tc::cp_async_wait<4>(); break;
    case 5: tc::cp_async_wait<5>(); break;
    default: tc::cp_async_wait<6>(); break;
  }
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

// One task's products: this lane's 32 K of fragment rows g and g+8 (16-byte
// code chunks at c * 16 of rows g and g + 8 of the slot; the task's two
// groups' scales at sb[row * rs + 0, 1] and biases at sb[row * rs + bo + 0, 1],
// in bf16) against the B fragments xb[w]
// (permuted activations, 8 K per 16-byte word): 8 MMAs. With g = lane / 4
// and c = lane % 4, MMA k slots 2c, 2c+1, 2c+8, 2c+9 of word w hold K
// offsets 8w + {0,4}, {1,5} (first MMA, into d0) and 8w + {2,6}, {3,7}
// (second, into d1), on A and B alike: two accumulator chains, since one
// warp's dependent MMAs are what this phase waits on. Returns false when a
// scale of 4 or more (scale * 2^14 past fp16) was met.
__device__ __forceinline__ bool task_mma(float (&d0)[4], float (&d1)[4], const uint8_t* t, const uint16_t* sb,
                                         int rs, int bo, int g8, int c4, const uint4 (&xb)[4]) {
  const uint4 r0 = *reinterpret_cast<const uint4*>(t + g8 * 64 + c4 * 16);
  const uint4 r1 = *reinterpret_cast<const uint4*>(t + (8 + g8) * 64 + c4 * 16);
  const int gs = c4 >> 1;  // this lane's 32 K lie in the second group of the pair when c >= 2
  // scale * 2^14 and bias per row (tc::dequant8_f16)
  const __half2 s0 = __float2half2_rn(bf16_bits_to_f32(sb[g8 * rs + gs]) * 16384.f);
  const __half2 b0 = __float2half2_rn(bf16_bits_to_f32(sb[g8 * rs + bo + gs]));
  const __half2 s1 = __float2half2_rn(bf16_bits_to_f32(sb[(8 + g8) * rs + gs]) * 16384.f);
  const __half2 b1 = __float2half2_rn(bf16_bits_to_f32(sb[(8 + g8) * rs + bo + gs]));
  const uint32_t w0[4] = {r0.x, r0.y, r0.z, r0.w}, w1[4] = {r1.x, r1.y, r1.z, r1.w};
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    uint32_t p0[4], p1[4];
    tc::dequant8_f16(w0[w], s0, b0, p0);
    tc::dequant8_f16(w1[w], s1, b1, p1);
    mma_16816(d0, p0[0], p1[0], p0[1], p1[1], xb[w].x, xb[w].y);
    mma_16816(d1, p0[2], p1[2], p0[3], p1[3], xb[w].z, xb[w].w);
  }
  return !(__hisinf(__low2half(s0)) | __hisinf(__low2half(s1)));
}

// Copies of one task: 16 rows of a packed matrix (rows lo .. lo + 7, then
// hi .. hi + 7), K block kb (64 bytes of codes per row), and the scale and
// bias pairs of groups 2kb, 2kb+1 of each row.
__device__ __forceinline__ void task_copy(uint8_t* td, const uint8_t* codes, const uint16_t* sc, const uint16_t* bi,
                                          int lo, int hi, int row_bytes, int gpr, int kb, int lane) {
#pragma unroll
  for (int q0 = 0; q0 < 64; q0 += 32) {  // 16 rows x 4 pieces of 16 bytes
    const int q = q0 + lane, r = q >> 2, piece = q & 3;
    const int row = (r < 8 ? lo : hi) + (r & 7);
    cp_async16(td + r * 64 + piece * 16, codes + (size_t)row * row_bytes + kb * 64 + piece * 16);
  }
  const int r = lane >> 1, kind = lane & 1;
  const int row = (r < 8 ? lo : hi) + (r & 7);
  cp_async4(td + 1024 + r * 8 + kind * 4, (kind ? bi : sc) + (size_t)row * gpr + 2 * kb);
}

// x[t] . row for the router: lane l holds bf16 elements 8 (l + 32 q) .. +7
// of the row in w4[q]; the activations are fp32 in shared memory, elements
// 8v..8v+3 at xrow[4v] and 8v+4..8v+7 at xrow[H/2 + 4v] (consecutive lanes
// read consecutive 16-byte words). Four fp32 sums per lane (element pairs
// 0-1, 2-3, 4-5, 6-7 of each vector, in q order), added as (0+1)+(2+3),
// then a butterfly over the warp (every lane gets the result): one warp's
// dependent chain is what this step waits on, so it is kept short.
__device__ __forceinline__ float row_dot(const uint4 (&w4)[8], const float* xrow, int H, int rvec, int lane) {
  float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const int v = lane + 32 * q;
    if (v < rvec) {
      const float4 xa = reinterpret_cast<const float4*>(xrow)[v];
      const float4 xc = reinterpret_cast<const float4*>(xrow + H / 2)[v];
      const float xv[8] = {xa.x, xa.y, xa.z, xa.w, xc.x, xc.y, xc.z, xc.w};
      const uint32_t ww[4] = {w4[q].x, w4[q].y, w4[q].z, w4[q].w};
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        a[m] = fmaf(bf16_bits_to_f32(ww[m] & 0xFFFFu), xv[2 * m], a[m]);
        a[m] = fmaf(__uint_as_float(ww[m] & 0xFFFF0000u), xv[2 * m + 1], a[m]);
      }
    }
  }
  float acc = (a[0] + a[1]) + (a[2] + a[3]);
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
  const int cpi = I / kItemCols;     // gate/up items per slot
  const int nkb = H / 128;           // gate/up K blocks of 128 (4 per item and warp at H = 2048)
  const int dkb = I / 128;           // down K blocks of 128 per slot
  const int tpw = nkb / 4;           // gate/up tasks per item and warp (H % 512 == 0)
  const bool has_rows = b < H / 16;  // this block owns output rows 16b .. 16b + 15
  uint8_t* ring = dsm_raw + (size_t)warp * kSlots * kTaskBytes;        // this warp's ring
  uint8_t* sdn = dsm_raw + a.sdn_offset;                                // shared down tasks [dkb][kTaskBytes]
  __half* x16 = reinterpret_cast<__half*>(dsm_raw + a.x16_offset);     // [T][H] fp16, K-permuted
  float* xf = reinterpret_cast<float*>(dsm_raw + a.xf_offset);         // [T][H] fp32 layer input
  __half* hst = reinterpret_cast<__half*>(dsm_raw + a.x16_offset);     // down phase: h of a batch of slots
  float* part = reinterpret_cast<float*>(dsm_raw + a.part_offset);     // [16 warps][4][32]
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
  for (int i = tid; i < kDecodeMaxSlots * kDecodeMaxTokens; i += kDecThreads) (&S.slot_wt[0][0])[i] = 0.f;
  __syncthreads();

  // ---- this warp's ring of tasks, in order: for each of the block's gate/up
  // items, its tasks (unit u = warp % 4: gate rows n0 + 8u .. +7 and the up
  // rows I + n0 + 8u .. +7; K blocks kb = (warp / 4) tpw + jj), then its
  // routed down tasks (slot s >= sh, K block kc, task number
  // q = (s - sh) dkb + kc taken by warp q % 16).
  int n_items = 0, n_dn = 0;  // set once the slots are known
  auto issue_task = [&](int k) {
    uint8_t* td = ring + (size_t)(k % kSlots) * kTaskBytes;
    if (k < n_items * tpw) {
      const int j = k / tpw, jj = k - j * tpw;
      const int item = b + G * j, s = item / cpi, n0 = (item - s * cpi) * kItemCols;
      const int u = warp & 3, kb = (warp >> 2) * tpw + jj;
      task_copy(td, S.slot_src[s][0], reinterpret_cast<const uint16_t*>(S.slot_src[s][1]),
                reinterpret_cast<const uint16_t*>(S.slot_src[s][2]), n0 + 8 * u, I + n0 + 8 * u, H / 2, gpr, kb,
                lane);
    } else {
      const int q = warp + kDecWarps * (k - n_items * tpw);
      const int s = sh + q / dkb, kc = q - (s - sh) * dkb;
      task_copy(td, S.slot_src[s][3], reinterpret_cast<const uint16_t*>(S.slot_src[s][4]),
                reinterpret_cast<const uint16_t*>(S.slot_src[s][5]), 16 * b, 16 * b + 8, I / 2, igpr, kc, lane);
    }
    tc::cp_async_commit();
  };
  int issued = 0;  // tasks issued by this warp (one cp.async group each)
  auto wait_task = [&](int k) {  // task k's bytes have landed, for every lane
    cp_async_wait_dyn(issued - k - 1);
    __syncwarp();
  };

  // ---- phase 0: weights only (they do not depend on the previous kernel)
  const bool shared_first = sh && b < cpi;
  if (sh && has_rows && warp < dkb) {  // the shared down task of K block `warp`
    task_copy(sdn + (size_t)warp * kTaskBytes, S.slot_src[0][3], reinterpret_cast<const uint16_t*>(S.slot_src[0][4]),
              reinterpret_cast<const uint16_t*>(S.slot_src[0][5]), 16 * b, 16 * b + 8, I / 2, igpr, warp, lane);
    tc::cp_async_commit();
  }
  if (shared_first) {
    n_items = 1;  // the shared item (more items, if any, are counted after routing)
    for (; issued < tpw && issued < kSlots; ++issued) issue_task(issued);
  }
  // router rows on the blocks without a shared item (their x loads then do
  // not queue behind those copies)
  const int sfb = sh ? (cpi < G ? cpi : 0) : 0;
  const int RG = G - sfb;
  const int rrows = E + sh, rvec = H / 8;
  const int rrow = b - sfb + RG * warp;
  const bool router_warp = b >= sfb && rrow < rrows && warp != kGateWarp;
  uint4 w4[8];
  if (router_warp) load_row(w4, rrow < E ? a.wr + (size_t)rrow * H : a.wsg, rvec, lane);
  if (shared_first && warp == kGateWarp) load_row(w4, a.wsg, rvec, lane);

  // the gain row (a weight too): vector v = tid of it (H / 8 <= 256 vectors)
  uint4 gw = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);  // bf16 1.0 pairs
  if (a.norm && a.norm_w && tid < H / 8) gw = ldg_nc_v4(a.norm_w + (size_t)tid * 8);

  // x (and this call's workspace) may be the previous kernel's output: wait
  // for the prelude, which itself waits for the previous layer's kernels.
  grid_dep_wait();
  // The layer input x, or with the pre-norm join x = RMSNorm(r) = r / rms(r)
  // * gain, in two parts. First every thread turns its vectors of the input
  // row into fp32 (exact from bf16), times the gain, into xf in the router's
  // layout (elements 8v..8v+3 at [4v], 8v+4..8v+7 at [H/2 + 4v]), with each
  // token's sum of squares of r (per thread, the warp butterfly, then a tree
  // over the warps: inv_rms below). The router rows are dotted with r * gain
  // and scaled by 1 / rms(r) at the end, so the second part (the normalised
  // fp16 copy for the MMAs and its range check) is left to the warps that
  // have no top-k to run and is needed only once the routing is known.
  float ss[kDecodeMaxTokens] = {0.f, 0.f, 0.f, 0.f};
  {
    const uint32_t gv[4] = {gw.x, gw.y, gw.z, gw.w};
#pragma unroll
    for (int t = 0; t < kDecodeMaxTokens; ++t)
      if (t < T && tid < H / 8) {
        const int v = tid;
        const uint4 u = ldg_nc_v4(a.x + (size_t)t * H + (size_t)v * 8);
        const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
        float f[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          f[2 * q] = bf16_bits_to_f32(wv[q] & 0xFFFFu);
          f[2 * q + 1] = bf16_bits_to_f32(wv[q] >> 16);
        }
        float s0 = 0.f, s1 = 0.f;  // two chains, then added: shorter dependences
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          s0 = fmaf(f[q], f[q], s0);
          s1 = fmaf(f[4 + q], f[4 + q], s1);
        }
        ss[t] = s0 + s1;
        if (a.norm)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            f[2 * q] *= bf16_bits_to_f32(gv[q] & 0xFFFFu);
            f[2 * q + 1] *= bf16_bits_to_f32(gv[q] >> 16);
          }
        reinterpret_cast<float4*>(xf + (size_t)t * H)[v] = make_float4(f[0], f[1], f[2], f[3]);
        reinterpret_cast<float4*>(xf + (size_t)t * H + H / 2)[v] = make_float4(f[4], f[5], f[6], f[7]);
      }
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
  // 1 / rms(r) of token t from the 16 warps' partials (a tree: 4 sums of 4,
  // then pairs), or 1 without the join
  auto inv_rms = [&](int t) -> float {
    if (!a.norm) return 1.f;
    float q4[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      q4[j] = (part[(4 * j) * kDecodeMaxTokens + t] + part[(4 * j + 1) * kDecodeMaxTokens + t]) +
              (part[(4 * j + 2) * kDecodeMaxTokens + t] + part[(4 * j + 3) * kDecodeMaxTokens + t]);
    const float tot = (q4[0] + q4[1]) + (q4[2] + q4[3]);
    return 1.f / sqrtf(tot / (float)H + a.norm_eps);
  };

  // ---- phase R: router logits l[t][r] (r = E: the shared gate row), stored
  // for the other blocks; the shared gate itself where a shared item is here
  if (router_warp)
    for (int t = 0; t < T; ++t) {
      const float l = row_dot(w4, xf + (size_t)t * H, H, rvec, lane) * inv_rms(t);
      // an atomic exchange is performed at L2, where the polling blocks read
      // (a plain store could sit in this SM's L1 for microseconds)
      if (lane == 0) atomicExch(a.logits + (size_t)t * (E + 1) + rrow, l);
    }
  if (shared_first && warp == kGateWarp)
    for (int t = 0; t < T; ++t) {
      const float l = row_dot(w4, xf + (size_t)t * H, H, rvec, lane) * inv_rms(t);
      if (lane == 0) {
        S.g[t] = 1.f / (1.f + expf(-l));
        S.slot_wt[0][t] = S.g[t];
      }
    }
  // The normalised input in fp16, in the permuted K order, for the MMAs, by
  // warps T..15 (warps below T run the top-k next); fp16 keeps |x| < 65520.
  if (warp >= T)
    for (int i = tid - 32 * T; i < T * H / 8; i += kDecThreads - 32 * T) {
      const int t = i / (H / 8), v = i - t * (H / 8);
      const float4 fa = reinterpret_cast<const float4*>(xf + (size_t)t * H)[v];
      const float4 fc = reinterpret_cast<const float4*>(xf + (size_t)t * H + H / 2)[v];
      const float sc = inv_rms(t);
      float f[8] = {fa.x, fa.y, fa.z, fa.w, fc.x, fc.y, fc.z, fc.w};
      bool big = false;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        f[q] *= sc;
        big |= fabsf(f[q]) >= 65520.f;  // becomes inf in fp16
      }
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
  // The next call's prelude may launch now: it waits for this grid to finish.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // One gate/up item: tasks k0 .. k0 + tpw - 1 of this warp's ring; then h
  // to the workspace.
  auto run_item = [&](int j, int k0) {
    const int item = b + G * j, s = item / cpi, n0 = (item - s * cpi) * kItemCols;
    float d[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
    for (int jj = 0; jj < tpw; ++jj) {
      const int k = k0 + jj;
      wait_task(k);
      const int kb = (warp >> 2) * tpw + jj;
      uint4 xb[4];
      const __half* xrow = x16 + (size_t)(g8 < T ? g8 : 0) * H + kb * 128 + 32 * c4;
#pragma unroll
      for (int w = 0; w < 4; ++w)
        xb[w] = g8 < T ? *reinterpret_cast<const uint4*>(xrow + 8 * w) : make_uint4(0u, 0u, 0u, 0u);
      const uint8_t* td = ring + (size_t)(k % kSlots) * kTaskBytes;
      if (!task_mma(d, d1, td, reinterpret_cast<const uint16_t*>(td + 1024), 4, 2, g8, c4, xb)) S.range = 1;
      __syncwarp();  // the slot is read: refill it
      if (issued < n_items * tpw + n_dn) issue_task(issued++);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) part[(warp * 4 + r) * 32 + lane] = d[r] + d1[r];
    __syncthreads();
    if (warp < kUnits) {
      // unit u = warp: warps u, u+4, u+8, u+12 hold its partial sums (fixed
      // order). d0, d1: gate(column 8u + g, tokens 2c, 2c+1); d2, d3: up.
      float v[4];
#pragma unroll
      for (int r = 0; r < 4; ++r)
        v[r] = (part[(warp * 4 + r) * 32 + lane] + part[((warp + 4) * 4 + r) * 32 + lane]) +
               (part[((warp + 8) * 4 + r) * 32 + lane] + part[((warp + 12) * 4 + r) * 32 + lane]);
      const int pc = tc::perm8_pos(n0 + 8 * warp + g8);
      bool big = false, nz = false;
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int t = 2 * c4 + jj;
        if (t < T) {
          // The floor is checked on h itself: the stored value also carries
          // the routing weight, which may be tiny when the expert adds
          // next to nothing to y.
          const float hu = silu_f32(v[jj]) * v[2 + jj], hw = hu * S.slot_wt[s][t];
          __half hv = __float2half_rn(hw);
          if (!(fabsf(hw) < 65520.f)) S.range = 1;  // inf in fp16, or NaN
          if (__half_as_ushort(hv) == kHSentinel) hv = __ushort_as_half((unsigned short)0x7FFFu);
          big |= fabsf(hu) >= kFp16Floor;
          nz |= hu != 0.f;
          if (b != a.stall_block) a.h[((size_t)s * T + t) * I + pc] = hv;
        }
      }
      // the unit's 8 columns of h for every token, all below the fp16 floor
      if (__any_sync(0xffffffffu, nz) && !__any_sync(0xffffffffu, big)) S.range = 1;
      // no fence: every half of h is written once and readers poll each half
      // for the sentinel at L2, so nothing is ordered after these stores; a
      // fence here waited for this warp's copies still in flight as well
      // (decode-t1 14.85 -> 14.53 us per layer without it)
    }
    __syncthreads();  // the partial sums are read before the next item writes them
  };

  int k = 0;  // next task of this warp's ring
  if (shared_first) {
    __syncthreads();  // x16 is complete
    run_item(0, 0);
    k = tpw;
  }

  // ---- phase 1: top-k and slots, where this block has routed work: routed
  // items (past its shared one) or output rows. A block with neither skips
  // it, except the last block, which writes the routing outputs.
  const int max_items = ((A < E ? A : E) + sh) * cpi;
  const bool routed_items = b + (shared_first ? G : 0) < max_items;
  const bool need_topk = routed_items || has_rows || b == G - 1;
  if (need_topk) {
    if (warp < T) {
      const float* lrow = a.logits + (size_t)warp * (E + 1);
      float lv[kMaxExperts / 32];
      float gl = 0.f;
      bool ok = false;
      // Measured on GB300: the selection's eight rounds took about 5000
      // cycles when they followed this poll directly and about 780 when a
      // warp reduction ran in every poll round just before the exit test
      // (the reductions themselves cost 28 cycles each).
      uint32_t warm = (uint32_t)lane;
      while (true) {
#pragma unroll
        for (int j = 0; j < kMaxExperts / 32; ++j)
          lv[j] = __uint_as_float(ld_relaxed_u32(lrow + min(lane + 32 * j, E - 1)));
        gl = __uint_as_float(ld_relaxed_u32(lrow + (sh ? E : 0)));
        bool mine = __float_as_uint(gl) != kLogitSentinel;
#pragma unroll
        for (int j = 0; j < kMaxExperts / 32; ++j) mine &= __float_as_uint(lv[j]) != kLogitSentinel;
        warm = __reduce_max_sync(0xffffffffu, warm + (uint32_t)lane);
        if (__all_sync(0xffffffffu, mine)) {
          ok = true;
          break;
        }
        if (global_timer_ns() > deadline) break;
        __nanosleep(32);
      }
      if (warm == 0xFFFFFFFFu) S.range = 1;  // keeps the reduction (never true: warm grows by at most 62 a round)
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
        const int ex = checked(S.slot_e[q], 0, E - 1, a.status);
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
  const bool routed = need_topk && !S.failed;
  const int nslots = routed ? S.nslots : sh;
  const int items = nslots * cpi;
  n_items = b < items ? (items - b + G - 1) / G : 0;
  // routed down tasks of this warp: q = warp, warp + 16, ... < (nslots - sh) dkb
  const int nq = has_rows && routed ? (nslots - sh) * dkb : 0;
  n_dn = nq > warp ? (nq - warp + kDecWarps - 1) / kDecWarps : 0;

  // The routing outputs (same definitions as moe_route), written by the last
  // block.
  if (b == G - 1 && routed) {
    for (int i = tid; i < A; i += kDecThreads) {
      a.ids[i] = S.ids[i];
      a.weights[i] = S.w[i];
      const int pos = checked(S.pos[i], 0, A - 1, a.status);
      a.sorted[pos] = i;
      a.inv[i] = pos;
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

  // ---- phase 2: the routed gate/up items
  const int ntasks = n_items * tpw + n_dn;
  for (; issued < ntasks && issued - k < kSlots; ++issued) issue_task(issued);
  for (int j = shared_first ? 1 : 0; j < n_items; ++j) {
    run_item(j, k);
    k += tpw;
  }

  // ---- phase 3: down, for the blocks with output rows
  if (has_rows && routed) {
    // rows g, g+8 x tokens 2c, 2c+1, over this warp's down tasks (two chains)
    float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
    const int hb_bytes = T * I * 2;
    const int batch = (int)(a.hst_bytes / hb_bytes);  // slots whose h fits in shared memory at once
    for (int s0 = 0; s0 < nslots; s0 += batch) {
      const int s1 = min(nslots, s0 + batch);
      // h of the batch (fp16 [slot][T][I], K-permuted): each 16-byte piece is
      // read past L1 until none of its halves holds the prelude's sentinel
      // (every half is written once per call), up to 4 pieces per thread in
      // flight at a time
      {
        const int nch = (s1 - s0) * hb_bytes / 16;
        const uint4* hsrc = reinterpret_cast<const uint4*>(a.h + (size_t)s0 * T * I);
        for (int i0 = tid; i0 < nch; i0 += 4 * kDecThreads) {
          uint4 v[4];
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (i0 + j * kDecThreads < nch) v[j] = ld_relaxed_v4(hsrc + i0 + j * kDecThreads);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int i = i0 + j * kDecThreads;
            if (i >= nch) continue;
            while (has_h_sentinel(v[j])) {
              if (global_timer_ns() > deadline) {
                S.failed = 1;
                break;
              }
              __nanosleep(128);  // fewer polls of L2 while the weights stream in
              v[j] = ld_relaxed_v4(hsrc + i);
            }
            reinterpret_cast<uint4*>(hst)[i] = v[j];
          }
        }
      }
      __syncthreads();
      if (S.failed) break;
      // this batch's tasks in order through one copy of the product code: the
      // shared slot's task first (from its own buffer, in the first batch),
      // then the routed slots' ring tasks
      bool own = s0 == 0 && sh && warp < dkb;
      for (;;) {
        const uint8_t* td;
        int s, kc;
        if (own) {
          cp_async_wait_dyn(issued);  // the oldest group: the shared down task
          td = sdn + (size_t)warp * kTaskBytes;
          s = 0;
          kc = warp;
        } else {
          if (k >= ntasks) break;
          const int q = warp + kDecWarps * (k - n_items * tpw);
          s = sh + q / dkb;
          kc = q - (s - sh) * dkb;
          if (s >= s1) break;
          cp_async_wait_dyn(issued - k - 1);
          td = ring + (size_t)(k % kSlots) * kTaskBytes;
        }
        __syncwarp();
        uint4 xb[4];
        const __half* hrow = hst + ((size_t)(s - s0) * T + (g8 < T ? g8 : 0)) * I + kc * 128 + 32 * c4;
#pragma unroll
        for (int w = 0; w < 4; ++w)
          xb[w] = g8 < T ? *reinterpret_cast<const uint4*>(hrow + 8 * w) : make_uint4(0u, 0u, 0u, 0u);
        if (!task_mma(acc, acc1, td, reinterpret_cast<const uint16_t*>(td + 1024), 4, 2, g8, c4, xb)) S.range = 1;
        __syncwarp();
        if (own) {
          own = false;
        } else {
          ++k;
          if (issued < ntasks) issue_task(issued++);
        }
      }
      __syncthreads();  // the batch's h is read
    }
    // the 16 warps' sums in a fixed order: y and the next residual row
#pragma unroll
    for (int r = 0; r < 4; ++r) part[(warp * 4 + r) * 32 + lane] = acc[r] + acc1[r];
    __syncthreads();
    if (!S.failed && tid < 16 * T) {
      const int t = tid >> 4, row = tid & 15;
      const int ln = (row & 7) * 4 + (t >> 1), r = (t & 1) + ((row >> 3) << 1);
      float q4[4];  // the 16 warps' sums as a tree: 4 sums of 4, then pairs
#pragma unroll
      for (int j = 0; j < 4; ++j)
        q4[j] = (part[((4 * j) * 4 + r) * 32 + ln] + part[((4 * j + 1) * 4 + r) * 32 + ln]) +
                (part[((4 * j + 2) * 4 + r) * 32 + ln] + part[((4 * j + 3) * 4 + r) * 32 + ln]);
      const float y = (q4[0] + q4[1]) + (q4[2] + q4[3]);
      const int m = 16 * b + row;
      a.y[(size_t)t * H + m] = y;
      if (a.x_next) {
        const float xv = bf16_bits_to_f32(a.x[(size_t)t * H + m]);
        a.x_next[(size_t)t * H + m] = __bfloat16_as_ushort(__float2bfloat16_rn(xv + y));
      }
    }
  }
  tc::cp_async_wait_all();  // no copy into this block's shared memory outlives it
  __syncthreads();
  if (tid == 0) {
    if (S.failed) atomicExch(a.status, (int32_t)MOE_ERR_DEVICE_TIMEOUT);
    else if (S.range) atomicCAS(a.status, 0, (int32_t)MOE_ERR_RANGE);
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

// Dynamic shared memory: 16 warps x kSlots task slots, the shared down
// tasks, x16 fp16 and x fp32 [T][H] (in the down phase: h of a batch of
// slots), the partial sums of the gate/up reduction and of the final sum.
struct DecodeLayout {
  size_t sdn_offset, x16_offset, xf_offset, part_offset, hst_bytes, total;
};

DecodeLayout decode_layout(const Geometry& g) {
  DecodeLayout L{};
  L.sdn_offset = (size_t)kDecWarps * kSlots * kTaskBytes;
  L.x16_offset = L.sdn_offset + (size_t)(g.I / 128) * kTaskBytes;
  const size_t xb = ((size_t)g.T * g.H * 2 + 127) & ~size_t(127);
  L.xf_offset = L.x16_offset + xb;
  L.part_offset = L.xf_offset + 2 * xb;
  L.hst_bytes = 3 * xb;  // x16 and xf, reused for h
  L.total = L.part_offset + (size_t)kDecWarps * 4 * 32 * 4;
  return L;
}
}  // namespace

// One block per SM, every block resident (blocks wait for each other's
// logits and h); H a multiple of 512 up to 2048 (each warp takes a quarter of
// K in whole 128-wide blocks; 16-row output tiles on at most the SM count),
// I a multiple of 128 up to 1024, enough router warps (15 per block without a
// shared item) for the E (+ 1) router rows, h of a slot within the staging
// area.
bool decode_supported(const Geometry& g) {
  int dev = 0;
  if (g.T < 1 || g.T > kDecodeMaxTokens || g.H % 512 || g.H > 2048 || g.I % 128 || g.I > kDecMaxI ||
      cudaGetDevice(&dev) != cudaSuccess)
    return false;
  const int sms = sm_count(dev);
  if (sms <= 0 || g.H / 16 > sms) return false;
  const int cpi = g.I / kItemCols, sfb = g.shared ? (cpi < sms ? cpi : 0) : 0;
  if (g.E + g.shared > (sms - sfb) * (kDecWarps - 1)) return false;
  const DecodeLayout L = decode_layout(g);
  return L.total <= kDecDynamicLimit && L.hst_bytes >= (size_t)g.T * g.I * 2;
}

// Fills the call's logits and the h of every slot it can use with their
// sentinels and clears the status word. Launched with programmatic dependent
// launch, it starts while the previous kernel on the stream (often the
// previous layer's decode kernel, the last reader of h) is finishing, lets
// the decode kernel start at once, and waits for the previous kernel to
// complete before it writes; the decode kernel waits for this grid before it
// reads x, the logits or h.
__global__ void decode_prelude_kernel(float* logits, int n_logits, uint4* h, int h_pieces, int32_t* status) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < n_logits; i += blockDim.x) reinterpret_cast<uint32_t*>(logits)[i] = kLogitSentinel;
    if (threadIdx.x == 0) *status = 0;
  }
  const uint32_t s2 = ((uint32_t)kHSentinel << 16) | kHSentinel;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < h_pieces; i += gridDim.x * blockDim.x)
    h[i] = make_uint4(s2, s2, s2, s2);
}

cudaError_t launch_decode(const DecodeArgs& args_in, const Geometry& g, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int grid = sm_count(dev);
  if (grid <= 0) return cudaErrorInvalidDevice;
  const DecodeLayout L = decode_layout(g);
  static SmemLimitMemo smem_memo;
  e = ensure_smem(decode_layer_kernel, L.total, &smem_memo);
  if (e != cudaSuccess) return e;
  // Every block must be resident at once: one block per SM must fit.
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_layer_kernel, kDecThreads, L.total);
  if (e != cudaSuccess) return e;
  if (!all_blocks_resident(per_sm, grid, grid)) return cudaErrorCooperativeLaunchTooLarge;
  {
    // the h of every slot this call can use: T K routed + 1 shared, T rows each
    const int h_pieces = (g.T * g.K + 1) * g.T * g.I * 2 / 16;
    cudaLaunchConfig_t pc{};
    pc.gridDim = dim3((h_pieces + 255) / 256);  // one 16-byte store per thread
    pc.blockDim = dim3(256);
    pc.stream = stream;
    cudaLaunchAttribute pa[1];
    pa[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pa[0].val.programmaticStreamSerializationAllowed = 1;
    pc.attrs = pa;
    pc.numAttrs = 1;
    e = cudaLaunchKernelEx(&pc, decode_prelude_kernel, args_in.logits, g.T * (g.E + 1),
                           reinterpret_cast<uint4*>(args_in.h), h_pieces, args_in.status);
    if (e != cudaSuccess) return e;
  }
  DecodeArgs args = args_in;
  args.sdn_offset = (long long)L.sdn_offset;
  args.x16_offset = (long long)L.x16_offset;
  args.xf_offset = (long long)L.xf_offset;
  args.part_offset = (long long)L.part_offset;
  args.hst_bytes = (long long)L.hst_bytes;
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
