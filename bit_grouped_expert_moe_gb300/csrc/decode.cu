// Fused decode MoE layer (T <= 4 tokens): top-k, routing tables, gate/up with
// fused dequantisation and SiLU, down projection and the weighted combine in
// one kernel that follows the router kernel.
// [droneth.or.th Lily article, "Decode is bound by bandwidth more than
// compute": at batch 1 weights are barely reused, so the bound is the bytes
// moved; dothoosh.com "Perplexity Lily: 1.35x faster decode for Qwen3.6 on
// Apple silicon", "Decode optimisations", kernel fusion: chains of kernels
// fused so intermediates stay on chip.]
//
// Weights stream through a ring of shared-memory stages filled by bulk async
// copies (cp.async.bulk, completion counted on an mbarrier), so a block keeps
// up to `stages` tiles in flight whatever the compute between them does. One
// ring item is either
//   a gate/up item: expert slot s, h columns n0..n0+15 -> gate rows
//     n0..n0+15 and up rows I+n0..I+n0+15 with their scales and biases
//     (18H bytes; two MMA units of 8 columns), or
//   a down item: rows m0..m0+15 of W_down for up to `per_item` slots.
// The products run on mma.sync.m16n8k16 (fp16 operands, fp32 accumulation):
// 16 weight rows x 8 token columns per instruction. In a gate/up unit the 16
// MMA rows are 8 gate rows then the matching 8 up rows, so the lane that
// holds gate(n, j) also holds up(n, j). Each lane dequantises whole code words into
// A fragments; one word unpacks as the pairs (k0,k4), (k1,k5), (k2,k6),
// (k3,k7), so the activations are kept in that K order inside every group of
// 8 (0,4,1,5,2,6,3,7) and a B fragment is one 16-byte shared-memory load.
//
// One block per SM, every block resident: 16 consumer warps and one producer
// warp whose lane 0 issues the bulk copies (kept out of the consumer warps: a
// lane issuing while its warp-mates wait on an mbarrier is held up by them).
// A one-block prelude kernel clears the two grid-barrier counters and the
// status word. Both kernels use programmatic dependent launch: the prelude
// starts while the previous layer's kernel finishes (after that kernel's
// barrier B) and waits for it before clearing; this kernel starts at once,
// loads weights, and waits for the prelude before it reads x. Phases:
//   0  the router's first weight loads and, in a block whose first item
//      belongs to the shared expert (which every token uses), that item's
//      copies go out; after the wait x is staged (fp16 in the permuted K
//      order for the experts, bf16 for the router);
//   R  router logits: block b, warp w computes rows b + G*w, G*16 apart, and
//      writes l[t][r] to global memory; grid barrier A;
//   1  every block selects the top-k experts of the T tokens itself (reading
//      the logits through L2) and derives the expert slots; from here the
//      producer fills the ring as the consumers release stages (one "empty"
//      mbarrier per stage);
//   2  gate/up items: the 16 warps split K, the partial sums of each 8-column
//      unit are added in a fixed order by one warp while the others go on,
//      and h = w * silu(gate) * up (the token's routing weight, or the shared
//      gate, folded in) goes to global memory as fp16;
//   3  grid barrier B;
//   4  block b owns output rows 16b..16b+15: with the weights folded into h,
//      y[t][m] = sum over slots of W_down[m] . h_slot,t, so every warp keeps one
//      accumulator over its (slot, K block) tasks and the 16 accumulators are
//      added in a fixed order at the end. The last block writes the routing
//      tables.
// Reading, right after a programmatic-dependent-launch wait, values another
// kernel wrote just before it finished proved slow (about 2.8 us for the
// logits row on GB300, against 1.5 us for a DRAM miss of unrelated data),
// which is why the router runs inside this kernel.
#include "kernels.h"
#include "tc_ptx.cuh"

namespace bgmoe {

constexpr int kDecWarps = 16;                        // consumer warps
constexpr int kDecConsumers = kDecWarps * 32;
constexpr int kDecThreads = kDecConsumers + 32;      // + the producer warp
constexpr int kDecMaxA = kDecodeMaxTokens * kMaxTopK;
constexpr int kDecMaxSlots = kDecMaxA + 1;

struct DecodeSmall {
  int ids[kDecMaxA];
  float w[kDecMaxA];
  float g[kDecodeMaxTokens];
  int pos[kDecMaxA];                             // expert-sorted position of assignment a
  int slot_e[kDecMaxSlots];                      // expert of each slot (slot 0 = shared when present)
  int slot_n[kDecMaxSlots];                      // rows (tokens) of the slot
  int slot_row[kDecMaxSlots][kDecodeMaxTokens];
  int slot_tok[kDecMaxSlots][kDecodeMaxTokens];
  float slot_w[kDecMaxSlots][kDecodeMaxTokens];  // routing weight (shared slot: gate) of each slot row
  int tok_row[kDecMaxSlots][kDecodeMaxTokens];   // h row of (slot, token), -1 if the token skips it
  const uint8_t* slot_src[kDecMaxSlots][6];     // gate/up codes, scales, biases; down codes, scales, biases
  int nslots;
  int failed;    // consumer abort flag (a stage or grid-barrier wait ran out)
  int pfail;     // producer abort flag (kept apart: consumers branch on `failed` only)
  uint64_t full[kDecodeMaxStages];               // stage filled (bulk-copy bytes landed)
  uint64_t empty[kDecodeMaxStages];              // stage released by all consumer warps
  float part[2][2][kDecWarps][4][32];            // per-warp MMA partials: [item parity][sub-unit][warp][reg][lane]
};


__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bulk async copy global -> this CTA's shared memory, completion counted in
// bytes on `bar` (both addresses and the size multiples of 16 bytes).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   tc::smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(tc::smem_u32(bar))
               : "memory");
}

// Waits for the mbarrier phase with the given parity, sleeping between polls
// (up to 256 ns) so that waiting warps leave the issue slots to the warps
// doing work. Returns false once *abort is set or the deadline passes (then
// it sets *abort).
__device__ __forceinline__ bool ring_wait(uint64_t* bar, uint32_t parity, volatile int* abort, uint64_t deadline) {
  unsigned ns = 32;
  while (!tc::mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (global_timer_ns() > deadline) {
      *abort = 1;
      return false;
    }
    __nanosleep(ns);
    ns = ns < 256 ? 2 * ns : 256;
  }
  return true;
}

// Arrival on a grid barrier: release orders the block's earlier writes (made
// visible to this thread by the preceding block barrier) before the add.
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
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

__device__ __forceinline__ void load_b(uint4 (&xb)[4], const __half* row, bool live) {
#pragma unroll
  for (int w = 0; w < 4; ++w)
    xb[w] = live ? *reinterpret_cast<const uint4*>(row + 8 * w) : make_uint4(0u, 0u, 0u, 0u);
}


// Named barrier of the 16 consumer warps (the producer warp never joins it).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kDecConsumers) : "memory");
}

__global__ void __launch_bounds__(kDecThreads, 1) decode_layer_kernel(const DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t dsm_raw[];
  __shared__ DecodeSmall S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool producer = warp == kDecWarps;
  const int g8 = lane >> 2, c4 = lane & 3;  // fragment coordinates
  const int T = a.T, H = a.H, I = a.I, E = a.E, K = a.K;
  const int A = T * K;
  const int G = gridDim.x, b = blockIdx.x;
  const int gpr = H / kGroup, igpr = I / kGroup;
  const int NST = a.stages;
  const int cpb = I / 16;            // gate/up items per slot (16 h columns each)
  const int mblocks = H / 16;        // blocks with output rows
  const int m0 = b * 16;
  const int kbs = I / 128, nkb = H / 128;
  const int per_item = a.per_item;   // down slots per ring item
  const size_t stage_bytes = (size_t)a.stage_bytes;
  __half* xs = reinterpret_cast<__half*>(dsm_raw);  // phases 0-2: x16 [T][H]; phase 4: h [R][I]
  uint16_t* xraw = reinterpret_cast<uint16_t*>(xs + (size_t)T * H);  // phases 0-R: x bf16 [T][H]
  uint8_t* ring = dsm_raw + a.ring_offset;
  const uint64_t deadline0 = global_timer_ns() + (uint64_t)a.timeout_ns;

  // ---- ring producer (the producer warp): item i -> stage i % NST. Every
  // part of an item is one bulk copy, each posted by its own lane in a single
  // instruction; the producer shares its scheduler with busy consumer warps,
  // so it keeps its own instruction count per item small.
  int n2 = 0;  // gate/up items of this block (known after routing); down items follow them
  const uint32_t gcb = 16u * (H / 2), gsb = 16u * gpr * 2;     // gate/up item: 16 code rows / scale rows
  const uint32_t dcb = 16u * (I / 2), dsb = 16u * igpr * 2;    // down item, per slot: 16 code rows / scale rows
  auto issue = [&](int i, int nslots) {  // called by all 32 lanes of the producer warp
    const int st = i % NST;
    uint8_t* dst = ring + (size_t)st * stage_bytes;
    uint64_t* bar = &S.full[st];
    if (nslots < 0 || i < n2) {  // gate/up item (nslots < 0: the shared item issued before routing)
      const int u = b + i * G;
      const int s = u / cpb, n0 = (u - s * cpb) * 16;
      if (lane == 0) tc::mbar_arrive_expect_tx(bar, 2 * gcb + 4 * gsb);
      __syncwarp();
      if (lane < 6) {
        // lane: 0 gate codes, 1 up codes, 2 gate scales, 3 up scales, 4 gate biases, 5 up biases
        const int kind = lane >> 1, up = lane & 1;
        const uint8_t* base = nslots >= 0 ? S.slot_src[s][kind]
                              : reinterpret_cast<const uint8_t*>(kind == 0 ? (const void*)a.gu.s_codes
                                                                 : kind == 1 ? (const void*)a.gu.s_scales
                                                                             : (const void*)a.gu.s_biases);
        const size_t row = up ? (size_t)(I + n0) : (size_t)n0;
        const uint32_t rb = kind == 0 ? (uint32_t)(H / 2) : (uint32_t)gpr * 2;
        const uint32_t off = kind == 0 ? up * gcb : 2 * gcb + (uint32_t)(lane - 2) * gsb;
        bulk_g2s(dst + off, base + row * rb, kind == 0 ? gcb : gsb, bar);
      }
    } else {  // down item: rows m0..m0+15 of slots p0..p0+np-1
      const int p0 = (i - n2) * per_item;
      const int np = min(per_item, nslots - p0);
      if (lane == 0) tc::mbar_arrive_expect_tx(bar, (uint32_t)np * (dcb + 2 * dsb));
      __syncwarp();
      for (int c = lane; c < 3 * np; c += 32) {  // lane: slot c / 3, part c % 3 (codes, scales, biases)
        const int p = c / 3, kind = c - 3 * p;
        const uint32_t rb = kind == 0 ? (uint32_t)(I / 2) : (uint32_t)igpr * 2;
        const uint32_t off = (uint32_t)p * (dcb + 2 * dsb) + (kind == 0 ? 0u : dcb + (uint32_t)(kind - 1) * dsb);
        bulk_g2s(dst + off, S.slot_src[p0 + p][3 + kind] + (size_t)m0 * rb, kind == 0 ? dcb : dsb, bar);
      }
    }
  };
  int issued = 0;  // items issued so far (producer warp)
  // Waits (bounded) until the last copy of every stage has landed, so the
  // block never exits with copies into its shared memory in flight.
  auto drain = [&]() {
    for (int i = issued > NST ? issued - NST : 0; i < issued; ++i) {
      const uint64_t dl = global_timer_ns() + (uint64_t)a.timeout_ns;
      while (!tc::mbar_try_wait(&S.full[i % NST], (uint32_t)((i / NST) & 1)))
        if (global_timer_ns() > dl) break;
    }
  };

  // ---- phase 0: barriers, x as fp16 in the permuted K order, the shared unit
  if (producer) {
    if (lane == 0) {
      for (int st = 0; st < NST; ++st) {
        tc::mbar_init(&S.full[st], 1);
        tc::mbar_init(&S.empty[st], kDecWarps);
      }
      tc::fence_barrier_init();
      S.failed = 0;
      S.pfail = 0;
    }
    __syncwarp();
    if (a.shared && b < cpb) {  // this block's first unit belongs to the shared expert
      issue(0, -1);
      issued = 1;
    }
  }
  for (int i = tid; i < kDecMaxSlots * kDecodeMaxTokens; i += kDecThreads) (&S.tok_row[0][0])[i] = -1;
  // The router warps' first weight loads go out before x is staged (they do
  // not depend on it).
  const int rrows = E + (a.shared ? 1 : 0), rvec = H / 8;
  const int r0 = b + G * warp;
  const bool router_warp = warp < kDecWarps && r0 < rrows;
  uint4 w4[8];
  if (router_warp) {
    const uint16_t* wrow = r0 < E ? a.wr + (size_t)r0 * H : a.wsg;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (lane + 32 * q < rvec) w4[q] = ldg_nc_v4(wrow + (size_t)(lane + 32 * q) * 8);
  }
  // Everything above reads only weights. x (and this call's workspace) may be
  // the previous kernel's output: wait for the prelude, which itself waits
  // for the previous layer's kernels to finish.
  grid_dep_wait();
  for (int i = tid; i < T * H / 8; i += kDecThreads) {
    const uint4 v = ldg_nc_v4(a.x + (size_t)i * 8);
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
    float f[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      f[2 * q] = bf16_bits_to_f32(wv[q] & 0xFFFFu);
      f[2 * q + 1] = bf16_bits_to_f32(wv[q] >> 16);
    }
    const __half2 p0 = __floats2half2_rn(f[0], f[4]), p1 = __floats2half2_rn(f[1], f[5]);
    const __half2 p2 = __floats2half2_rn(f[2], f[6]), p3 = __floats2half2_rn(f[3], f[7]);
    uint4 o;
    o.x = *reinterpret_cast<const uint32_t*>(&p0);
    o.y = *reinterpret_cast<const uint32_t*>(&p1);
    o.z = *reinterpret_cast<const uint32_t*>(&p2);
    o.w = *reinterpret_cast<const uint32_t*>(&p3);
    reinterpret_cast<uint4*>(xs)[i] = o;
    reinterpret_cast<uint4*>(xraw)[i] = v;  // bf16 as given, for the router
  }
  __syncthreads();

  // ---- phase R: router logits l[t][r] = x[t] . W_r[r] (r = E: the shared
  // expert's gate row), fp32, rows r = b + G * warp (+ G * 16 ...)
  for (int r = r0; router_warp && r < rrows; r += G * kDecWarps) {
    const uint16_t* wrow = r < E ? a.wr + (size_t)r * H : a.wsg;
    float acc[kDecodeMaxTokens] = {0.f, 0.f, 0.f, 0.f};
    for (int v0 = lane; v0 < rvec; v0 += 32 * 8) {
      if (r != r0 || v0 != lane) {  // the first batch was loaded before the x staging
#pragma unroll
        for (int q = 0; q < 8; ++q)  // every load of the batch before any use
          if (v0 + 32 * q < rvec) w4[q] = ldg_nc_v4(wrow + (size_t)(v0 + 32 * q) * 8);
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int v = v0 + 32 * q;
        if (v < rvec) {
          const uint32_t ww[4] = {w4[q].x, w4[q].y, w4[q].z, w4[q].w};
#pragma unroll
          for (int t = 0; t < kDecodeMaxTokens; ++t)
            if (t < T) {
              const uint4 x4 = *reinterpret_cast<const uint4*>(xraw + (size_t)t * H + (size_t)v * 8);
              const uint32_t xv[4] = {x4.x, x4.y, x4.z, x4.w};
              float sacc = acc[t];
#pragma unroll
              for (int m = 0; m < 4; ++m) {
                sacc = fmaf(bf16_bits_to_f32(ww[m] & 0xFFFFu), bf16_bits_to_f32(xv[m] & 0xFFFFu), sacc);
                sacc = fmaf(bf16_bits_to_f32(ww[m] >> 16), bf16_bits_to_f32(xv[m] >> 16), sacc);
              }
              acc[t] = sacc;
            }
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kDecodeMaxTokens; ++t) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
      if (lane == 0 && t < T) a.logits[(size_t)t * (E + 1) + r] = acc[t];
    }
  }

  // ---- grid barrier A: every logit written (the prelude kernel cleared the
  // counters before this grid's wait returned)
  __syncthreads();
  if (tid == 0) {
    red_release_add(a.bar, 1u);
    while (ld_acquire_u32(a.bar) < (unsigned)G) {
      if (global_timer_ns() > deadline0) {
        S.failed = 1;
        atomicExch(a.status, (int32_t)MOE_ERR_DEVICE_TIMEOUT);
        break;
      }
      __nanosleep(20);
    }
  }
  __syncthreads();

  // ---- phase 1a: top-k, renormalised weights, shared gate (warp per token)
  if (warp < T) {
    int e;
    float w, g;
    warp_topk(a.logits + (size_t)warp * (E + 1), a.bias, E, K, a.shared, lane, &e, &w, &g);
    if (lane < K) {
      S.ids[warp * K + lane] = e;
      S.w[warp * K + lane] = w;
    }
    if (lane == 0) S.g[warp] = g;
  }
  __syncthreads();
  if (S.failed) {  // grid barrier A ran out
    if (producer && lane == 0) drain();
    return;
  }

  // ---- phase 1b: expert-sorted positions and slots (one lane per assignment)
  if (warp == 0) {
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
    const int sh = a.shared ? 1 : 0;
    if (live) {
      const int slot = dlt + sh, tok = lane / K;
      S.pos[lane] = lt + before;
      S.slot_row[slot][before] = lt + before;
      S.slot_tok[slot][before] = tok;
      S.slot_w[slot][before] = S.w[lane];
      S.tok_row[slot][tok] = lt + before;
      if (first) {
        S.slot_e[slot] = e;
        S.slot_n[slot] = __popc(same);
      }
    }
    const int d = __popc(__ballot_sync(0xffffffffu, first));
    if (lane == 0) {
      S.nslots = d + sh;
      if (sh) {
        S.slot_e[0] = E;
        S.slot_n[0] = T;
      }
    }
    if (sh && lane < T) {
      S.slot_row[0][lane] = A + lane;
      S.slot_tok[0][lane] = lane;
      S.slot_w[0][lane] = S.g[lane];
      S.tok_row[0][lane] = A + lane;
    }
    __syncwarp();
    // weight addresses of every slot, for the producer
    const int ns = d + sh;
    for (int q = lane; q < ns; q += 32) {
      const int ex = S.slot_e[q];
      const bool shq = ex == E;
      S.slot_src[q][0] = reinterpret_cast<const uint8_t*>(shq ? a.gu.s_codes : a.gu.codes + (size_t)ex * 2 * I * (H / 8));
      S.slot_src[q][1] = reinterpret_cast<const uint8_t*>(shq ? a.gu.s_scales : a.gu.scales + (size_t)ex * 2 * I * gpr);
      S.slot_src[q][2] = reinterpret_cast<const uint8_t*>(shq ? a.gu.s_biases : a.gu.biases + (size_t)ex * 2 * I * gpr);
      S.slot_src[q][3] = reinterpret_cast<const uint8_t*>(shq ? a.dn.s_codes : a.dn.codes + (size_t)ex * H * (I / 8));
      S.slot_src[q][4] = reinterpret_cast<const uint8_t*>(shq ? a.dn.s_scales : a.dn.scales + (size_t)ex * H * igpr);
      S.slot_src[q][5] = reinterpret_cast<const uint8_t*>(shq ? a.dn.s_biases : a.dn.biases + (size_t)ex * H * igpr);
    }
  }
  __syncthreads();  // the last block-wide barrier: from here on the producer runs on its own
  const int nslots = S.nslots;
  const int units = nslots * cpb;
  n2 = units > b ? (units - b + G - 1) / G : 0;
  const int n4 = b < mblocks ? (nslots + per_item - 1) / per_item : 0;
  const int items = n2 + n4;

  if (producer) {
    for (int i = issued; i < items; ++i) {
      // stage i % NST is free once every consumer warp released item i - NST
      if (i >= NST && !ring_wait(&S.empty[i % NST], (uint32_t)((i / NST - 1) & 1), &S.pfail, deadline0))
        break;
      issue(i, nslots);
      issued = i + 1;
    }
    if (lane == 0) drain();
    return;
  }

  // ---- phase 2: gate/up items (consumer warps). An item is two 8-column
  // units: unit q takes gate rows 8q..8q+7 and up rows 8q..8q+7 of the stage
  // as its 16 MMA rows.
  const int R = A + (a.shared ? T : 0);
  for (int i = 0; i < n2; ++i) {
    // On a timeout every consumer still runs every iteration (skipping the
    // math), so all of them pass the same named barriers.
    const int st = i % NST;
    const uint8_t* sp = ring + (size_t)st * stage_bytes;
    const bool ok = ring_wait(&S.full[st], (uint32_t)((i / NST) & 1), &S.failed, deadline0);
    const int u = b + i * G;
    const int s = u / cpb, n0 = (u - s * cpb) * 16;
    const int nr = S.slot_n[s];
    float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
    if (ok) {
      const bool col_live = g8 < nr;
      const __half* xrow = xs + (size_t)(col_live ? S.slot_tok[s][g8] : 0) * H;
      const uint16_t* s16 = reinterpret_cast<const uint16_t*>(sp + 2 * gcb);  // gate sc, up sc, gate bi, up bi
      const int q16 = gsb / 2;  // uint16 entries per run
      for (int kb = warp; kb < nkb; kb += kDecWarps) {
        const int koff = kb * 64 + 16 * c4;  // byte offset of this lane's 32 K inside a code row
        const int gi = g8 * gpr + 2 * kb + (c4 >> 1), gi8 = gi + 8 * gpr;
        uint4 xb[4];
        load_b(xb, xrow + kb * 128 + 32 * c4, col_live);
        const uint4 cg0 = *reinterpret_cast<const uint4*>(sp + g8 * (H / 2) + koff);
        const uint4 cu0 = *reinterpret_cast<const uint4*>(sp + gcb + g8 * (H / 2) + koff);
        const uint4 cg1 = *reinterpret_cast<const uint4*>(sp + (g8 + 8) * (H / 2) + koff);
        const uint4 cu1 = *reinterpret_cast<const uint4*>(sp + gcb + (g8 + 8) * (H / 2) + koff);
        mma_chunk(d0, cg0, cu0, bf16_h2(s16[gi]), bf16_h2(s16[2 * q16 + gi]), bf16_h2(s16[q16 + gi]),
                  bf16_h2(s16[3 * q16 + gi]), xb);
        mma_chunk(d1, cg1, cu1, bf16_h2(s16[gi8]), bf16_h2(s16[2 * q16 + gi8]), bf16_h2(s16[q16 + gi8]),
                  bf16_h2(s16[3 * q16 + gi8]), xb);
      }
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&S.empty[st]);  // this warp is done with the stage
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      S.part[i & 1][0][warp][r][lane] = d0[r];
      S.part[i & 1][1][warp][r][lane] = d1[r];
    }
    consumer_sync();
#pragma unroll
    for (int q = 0; q < 2; ++q)
      if (ok && warp == (2 * i + q) % kDecWarps) {
        // d0, d1: gate(n0+8q+g, slot rows 2c, 2c+1); d2, d3: up of the same
        float v[4] = {0.f, 0.f, 0.f, 0.f};
        for (int w = 0; w < kDecWarps; ++w)  // fixed order: the same bits on every run
#pragma unroll
          for (int r = 0; r < 4; ++r) v[r] += S.part[i & 1][q][w][r][lane];
        const int pn = tc::perm8_pos(n0 + 8 * q + g8);
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
          const int j = 2 * c4 + jj;
          if (j < nr)
            a.h[(size_t)S.slot_row[s][j] * I + pn] = __float2half_rn(silu_f32(v[jj]) * v[2 + jj] * S.slot_w[s][j]);
        }
      }
  }

  // ---- phase 3: grid barrier (every block resident; bounded wait)
  consumer_sync();
  if (tid == 0) {
    if (!S.failed) {
      if (b != a.stall_block) red_release_add(a.bar + 1, 1u);
      while (ld_acquire_u32(a.bar + 1) < (unsigned)G) {
        if (global_timer_ns() > deadline0) {
          S.failed = 1;
          break;
        }
        __nanosleep(20);
      }
    }
    if (S.failed) atomicExch(a.status, (int32_t)MOE_ERR_DEVICE_TIMEOUT);
  }
  consumer_sync();
  // The next call's prelude may now be scheduled; it waits for this grid to
  // finish before it clears the counters.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (S.failed) return;  // the producer drains the copies in flight

  // The routing outputs (same definitions as moe_route), written by the last
  // block: it has no output rows when H / 16 < gridDim.x, so this costs the
  // layer nothing.
  if (b == G - 1) {
    for (int i = tid; i < A; i += kDecConsumers) {
      a.ids[i] = S.ids[i];
      a.weights[i] = S.w[i];
      a.sorted[S.pos[i]] = i;
      a.inv[i] = S.pos[i];
    }
    if (a.shared)
      for (int t = tid; t < T; t += kDecConsumers) a.gate[t] = S.g[t];
    for (int e = tid; e <= E + 1; e += kDecConsumers) {
      int lt = 0, eq = 0;
      for (int q = 0; q < A; ++q) {
        lt += S.ids[q] < e;
        eq += S.ids[q] == e;
      }
      if (e <= E) a.counts[e] = e < E ? eq : (a.shared ? T : 0);
      a.offsets[e] = e <= E ? lt : A + (a.shared ? T : 0);
    }
    // one tile per expert in use (counts <= T <= 4 < block_m), then the shared tile
    const int d = nslots - (a.shared ? 1 : 0);
    for (int s = tid; s < d; s += kDecConsumers) {
      const int slot = s + (a.shared ? 1 : 0);
      a.tile_expert[s] = S.slot_e[slot];
      a.tile_row0[s] = S.slot_row[slot][0];
      a.tile_rows[s] = S.slot_n[slot];
    }
    if (tid == 0) {
      if (a.shared) {
        a.tile_expert[d] = E;
        a.tile_row0[d] = A;
        a.tile_rows[d] = T;
      }
      *a.num_tiles = nslots;
    }
  }
  if (n4 == 0) return;

  // ---- phase 4: W_down rows m0..m0+15 of every slot against the weighted h
  __half* hs = xs;  // [R][I] (x is no longer needed)
  for (int i = tid; i < R * I / 8; i += kDecConsumers)
    reinterpret_cast<uint4*>(hs)[i] = __ldcg(reinterpret_cast<const uint4*>(a.h) + i);
  consumer_sync();
  float acc[4] = {0.f, 0.f, 0.f, 0.f};  // rows g, g+8 x tokens 2c, 2c+1 over this warp's tasks
  for (int i = n2; i < items; ++i) {
    const int st = i % NST;
    const uint8_t* sp = ring + (size_t)st * stage_bytes;
    if (ring_wait(&S.full[st], (uint32_t)((i / NST) & 1), &S.failed, deadline0)) {
      const int p0 = (i - n2) * per_item;
      const int np = min(per_item, nslots - p0);
      for (int task = warp; task < np * kbs; task += kDecWarps) {
        const int p = task / kbs, kb = task - p * kbs;
        const int s = p0 + p;
        const uint8_t* dp = sp + (size_t)p * (dcb + 2 * dsb);
        const int koff = kb * 64 + 16 * c4;
        const int gi = g8 * igpr + 2 * kb + (c4 >> 1), gi8 = gi + 8 * igpr;
        const uint4 c0 = *reinterpret_cast<const uint4*>(dp + g8 * (I / 2) + koff);
        const uint4 c1 = *reinterpret_cast<const uint4*>(dp + (g8 + 8) * (I / 2) + koff);
        const uint16_t* s16 = reinterpret_cast<const uint16_t*>(dp + dcb);  // scales, then biases
        const __half2 s0 = bf16_h2(s16[gi]), s1 = bf16_h2(s16[gi8]);
        const __half2 b0 = bf16_h2(s16[dsb / 2 + gi]), b1 = bf16_h2(s16[dsb / 2 + gi8]);
        const int row = g8 < T ? S.tok_row[s][g8] : -1;  // B column = token
        uint4 xb[4];
        load_b(xb, hs + (size_t)(row < 0 ? 0 : row) * I + kb * 128 + 32 * c4, row >= 0);
        mma_chunk(acc, c0, c1, s0, b0, s1, b1, xb);
      }
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&S.empty[st]);
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) S.part[0][0][warp][r][lane] = acc[r];
  consumer_sync();
  if (S.failed) {
    if (tid == 0) atomicExch(a.status, (int32_t)MOE_ERR_DEVICE_TIMEOUT);
    return;
  }
  for (int i = tid; i < T * 16; i += kDecConsumers) {
    const int t = i >> 4, row = i & 15;
    const int ln = (row & 7) * 4 + (t >> 1), r = (t & 1) + ((row >> 3) << 1);
    float v = 0.f;
    for (int w = 0; w < kDecWarps; ++w) v += S.part[0][0][w][r][ln];  // fixed order
    a.y[(size_t)t * H + m0 + row] = v;
  }
}

namespace {
int sm_count(int dev) {
  static int sms[64] = {0};
  if (dev < 0 || dev >= 64) return 0;
  if (sms[dev] == 0 && cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms[dev] = 0;
  return sms[dev];
}

constexpr size_t kDecDynamicLimit = 186 * 1024;  // 227 KB per block minus the static part (about 38 KB)

// Dynamic shared memory: x16 [T][H] and x bf16 [T][H] (phases 0-2) / h [R][I]
// (phase 4), then
// the ring. A stage holds one gate/up item (18H bytes: 32 code rows of H/2,
// 32 scale rows and 32 bias rows of H/32) or W_down rows of `per_item` slots
// (9I bytes each).
struct DecodeLayout {
  size_t ring_offset, stage_bytes, total;
  int stages, per_item;
};

DecodeLayout decode_layout(const Geometry& g) {
  DecodeLayout L{};
  const int R = g.A + (g.shared ? g.T : 0);
  const size_t xs = 2 * (size_t)g.T * g.H * 2, hs = (size_t)R * g.I * 2;  // x16 + x bf16, or h
  L.ring_offset = ((xs > hs ? xs : hs) + 127) & ~size_t(127);
  const int big = g.H > g.I ? g.H : g.I;
  L.stage_bytes = 18 * (size_t)big;
  L.per_item = 2 * big / g.I;
  const size_t room = kDecDynamicLimit > L.ring_offset ? kDecDynamicLimit - L.ring_offset : 0;
  const size_t fit = room / L.stage_bytes;
  L.stages = (int)(fit < (size_t)kDecodeMaxStages ? fit : kDecodeMaxStages);
  L.total = L.ring_offset + (size_t)L.stages * L.stage_bytes;
  return L;
}
}  // namespace

// One block per SM, all resident (the grid barrier needs that); 16 output
// rows per block; K in whole 128-wide blocks on both projections; at least
// two ring stages.
bool decode_supported(const Geometry& g) {
  int dev = 0;
  if (g.T < 1 || g.T > kDecodeMaxTokens || g.H % 128 || g.I % 128 || cudaGetDevice(&dev) != cudaSuccess)
    return false;
  const int sms = sm_count(dev);
  return sms > 0 && g.H / 16 <= sms && decode_layout(g).stages >= 2;
}

// Clears the decode kernel's two grid-barrier counters and the call's status
// word. Launched with programmatic dependent launch, it starts while the
// previous kernel on the stream (often the previous layer's decode kernel) is
// finishing, lets the decode kernel start at once, and waits for the previous
// kernel to complete before it touches the counters; the decode kernel waits
// for this grid before it reads x or the counters.
__global__ void decode_prelude_kernel(unsigned int* bar, int32_t* status) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) {
    bar[0] = 0u;
    bar[1] = 0u;
    *status = 0;
  }
}

cudaError_t launch_decode(const DecodeArgs& args_in, const Geometry& g, cudaStream_t stream) {
  {
    cudaLaunchConfig_t pc{};
    pc.gridDim = dim3(1);
    pc.blockDim = dim3(32);
    pc.stream = stream;
    cudaLaunchAttribute pa[1];
    pa[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pa[0].val.programmaticStreamSerializationAllowed = 1;
    pc.attrs = pa;
    pc.numAttrs = 1;
    const cudaError_t pe = cudaLaunchKernelEx(&pc, decode_prelude_kernel, args_in.bar, args_in.status);
    if (pe != cudaSuccess) return pe;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int grid = sm_count(dev);
  if (grid <= 0) return cudaErrorInvalidDevice;
  const DecodeLayout L = decode_layout(g);
  DecodeArgs args = args_in;
  args.stages = L.stages;
  args.per_item = L.per_item;
  args.stage_bytes = (long long)L.stage_bytes;
  args.ring_offset = (long long)L.ring_offset;
  static SmemLimitMemo smem_memo;
  e = ensure_smem(decode_layer_kernel, L.total, &smem_memo);
  if (e != cudaSuccess) return e;
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
