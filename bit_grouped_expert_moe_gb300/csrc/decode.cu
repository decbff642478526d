// Fused decode MoE layer (T <= 4 tokens): top-k, routing tables, gate/up with
// fused dequantisation and SiLU, down projection and the weighted combine in
// one kernel that follows the router kernel.
// [droneth.or.th Lily article, "Decode is bound by bandwidth more than
// compute": at batch 1 weights are barely reused, so the bound is the bytes
// moved; dothoosh.com "Perplexity Lily: 1.35x faster decode for Qwen3.6 on
// Apple silicon", "Decode optimisations", kernel fusion: chains of kernels
// fused so intermediates stay on chip.]
//
// One block per SM, every block resident. Phases:
//   0  before the router finishes (programmatic dependent launch): warps
//      that will compute a column of the shared expert issue its weight loads
//      (the shared expert does not depend on routing);
//   1  every block selects the top-k experts of the T tokens itself (T * 257
//      logits); block 0 also writes the routing tables. Each block prefetches
//      into L2 the down-projection rows it will need in phase 3, then warps
//      compute gate/up units (one expert, one h column: two weight rows) for
//      the shared expert and every distinct routed expert: h fp32 [A+T][I];
//   2  one grid barrier (counter cleared by the router kernel, bounded wait);
//   3  each block owns a slice of output columns m: for every expert in use
//      it dots W_down[m] with that expert's h rows, then forms
//      y[t][m] = sum_k w[t,k] o[t,k][m] + g[t] o_shared[t][m] in that fixed
//      order, so o never leaves the SM.
#include "kernels.h"

namespace bgmoe {

constexpr int kDecThreads = 512;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kDecMaxA = kDecodeMaxTokens * kMaxTopK;
constexpr int kDecMaxSlots = kDecMaxA + 1;
constexpr int kDecPad = 36;                 // floats per staged 32-value chunk

struct DecodeSmall {
  int ids[kDecMaxA];
  float w[kDecMaxA];
  float g[kDecodeMaxTokens];
  int pos[kDecMaxA];                        // expert-sorted position of assignment a
  int first[kDecMaxA];
  int slot_e[kDecMaxSlots];                 // expert of each slot (slot 0 = shared when present)
  int slot_n[kDecMaxSlots];                 // rows of the slot
  int slot_row[kDecMaxSlots][kDecodeMaxTokens];
  int slot_tok[kDecMaxSlots][kDecodeMaxTokens];
  int nslots;
  int failed;
};

__device__ __forceinline__ float dec_key_to_float(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// 32 weights of one 16-byte code chunk against a staged fp32 activation chunk
__device__ __forceinline__ float dot32_f(const uint4 c, float s, float b, const float* xr, float acc) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const float4 x0 = *reinterpret_cast<const float4*>(xr + 8 * m);
    const float4 x1 = *reinterpret_cast<const float4*>(xr + 8 * m + 4);
    const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
    for (int q = 0; q < 8; ++q) acc = fmaf(fmaf(s, (float)((w[m] >> (4 * q)) & 15u), b), xv[q], acc);
  }
  return acc;
}

template <int kDecMaxIt>  // 16-byte loads per lane per gate/up row: ceil(H / 1024)
__global__ void __launch_bounds__(kDecThreads, 1) decode_layer_kernel(const DecodeArgs a) {
  extern __shared__ __align__(16) float dsm[];
  __shared__ DecodeSmall S;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = a.T, H = a.H, I = a.I, E = a.E, K = a.K;
  const int A = T * K;
  const int G = gridDim.x;
  const int gw = blockIdx.x * kDecWarps + warp, nw = G * kDecWarps;
  const int nvec = H / 32, gpr = H / kGroup;
  const int shared_units = a.shared ? I : 0;

  // ---- phase 0: the shared expert's weight rows of this warp's first unit
  uint4 pc_g[kDecMaxIt], pc_u[kDecMaxIt];
  float ps_g[kDecMaxIt], pb_g[kDecMaxIt], ps_u[kDecMaxIt], pb_u[kDecMaxIt];
  const bool pre = gw < shared_units;
  if (pre) {
    const int n = gw;
#pragma unroll
    for (int it = 0; it < kDecMaxIt; ++it) {
      const int v = lane + 32 * it;
      if (v < nvec) {
        pc_g[it] = ldg_nc_v4(a.gu.s_codes + (size_t)n * (H / 8) + 4 * v);
        pc_u[it] = ldg_nc_v4(a.gu.s_codes + (size_t)(I + n) * (H / 8) + 4 * v);
        ps_g[it] = bf16_bits_to_f32(__ldg(a.gu.s_scales + (size_t)n * gpr + v / 2));
        pb_g[it] = bf16_bits_to_f32(__ldg(a.gu.s_biases + (size_t)n * gpr + v / 2));
        ps_u[it] = bf16_bits_to_f32(__ldg(a.gu.s_scales + (size_t)(I + n) * gpr + v / 2));
        pb_u[it] = bf16_bits_to_f32(__ldg(a.gu.s_biases + (size_t)(I + n) * gpr + v / 2));
      }
    }
  }
  grid_dep_wait();  // the router kernel (logits, cleared barrier) is complete
  if (device_failed(a.status)) return;

  // ---- phase 1a: stage x (fp32, padded chunks) and select the top-k
  float* xs = dsm;  // [T][H/32][kDecPad]
  {
    const int xvec = T * H / 8;  // 16-byte chunks of x; all loads of a batch before any store
    for (int i0 = tid; i0 < xvec; i0 += 2 * kDecThreads) {
      uint4 v[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int i = i0 + u * kDecThreads;
        if (i < xvec) v[u] = ldg_nc_v4(a.x + (size_t)i * 8);
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int i = i0 + u * kDecThreads;
        if (i < xvec) {
          const int t = (i * 8) / H, k = i * 8 - t * H;
          float* d = xs + (t * nvec + (k >> 5)) * kDecPad + (k & 31);
          const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
          *reinterpret_cast<float4*>(d) = make_float4(bf16_bits_to_f32(w[0] & 0xFFFFu), bf16_bits_to_f32(w[0] >> 16),
                                                      bf16_bits_to_f32(w[1] & 0xFFFFu), bf16_bits_to_f32(w[1] >> 16));
          *reinterpret_cast<float4*>(d + 4) = make_float4(bf16_bits_to_f32(w[2] & 0xFFFFu),
                                                          bf16_bits_to_f32(w[2] >> 16),
                                                          bf16_bits_to_f32(w[3] & 0xFFFFu), bf16_bits_to_f32(w[3] >> 16));
        }
      }
    }
  }
  if (tid == 0) S.failed = 0;
  if (warp < T) {
    const int t = warp;
    const float* lrow = a.logits + (size_t)t * (E + 1);
    unsigned long long key[kMaxExperts / 32];
#pragma unroll
    for (int j = 0; j < kMaxExperts / 32; ++j) {
      const int e = lane + 32 * j;
      key[j] = 0ull;
      if (e < E) {
        const float v = lrow[e] + (a.bias ? a.bias[e] : 0.f);
        key[j] = ((unsigned long long)float_order_key(v) << 32) | (0xFFFFFFFFu - (uint32_t)e);
      }
    }
    float sel_v[kMaxTopK];
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k) {
      if (k < K) {
        unsigned long long best = key[0];
#pragma unroll
        for (int j = 1; j < kMaxExperts / 32; ++j) best = key[j] > best ? key[j] : best;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
          best = other > best ? other : best;
        }
        const int e = (int)(0xFFFFFFFFu - (uint32_t)best);
        sel_v[k] = dec_key_to_float((uint32_t)(best >> 32));
        if (lane == 0) S.ids[t * K + k] = e;
#pragma unroll
        for (int j = 0; j < kMaxExperts / 32; ++j)
          if (lane == (e & 31) && j == (e >> 5)) key[j] = 0ull;
      }
    }
    if (lane == 0) {
      float z[kMaxTopK], sum = 0.f;
#pragma unroll
      for (int k = 0; k < kMaxTopK; ++k)
        if (k < K) {
          z[k] = expf(sel_v[k] - sel_v[0]);
          sum += z[k];
        }
#pragma unroll
      for (int k = 0; k < kMaxTopK; ++k)
        if (k < K) S.w[t * K + k] = z[k] / sum;
      S.g[t] = a.shared ? 1.f / (1.f + expf(-lrow[E])) : 0.f;
    }
  }
  __syncthreads();

  // ---- phase 1b: expert-sorted positions and the slots (distinct experts)
  if (tid < A) {
    const int e = S.ids[tid];
    int fst = 1;
    for (int b = 0; b < tid; ++b) fst &= (S.ids[b] != e);
    S.first[tid] = fst;
  }
  __syncthreads();
  if (tid < A) {
    const int e = S.ids[tid];
    int lt = 0, before = 0, dlt = 0;
    for (int b = 0; b < A; ++b) {
      const int eb = S.ids[b];
      lt += eb < e;
      before += (b < tid) & (eb == e);
      dlt += (eb < e) & S.first[b];
    }
    S.pos[tid] = lt + before;
    const int slot = dlt + (a.shared ? 1 : 0);
    S.slot_row[slot][before] = lt + before;
    S.slot_tok[slot][before] = tid / K;
    if (S.first[tid]) S.slot_e[slot] = e;
    if (S.first[tid]) {
      int n = 0;
      for (int b = 0; b < A; ++b) n += S.ids[b] == e;
      S.slot_n[slot] = n;
    }
  }
  if (tid == 0) {
    int d = 0;
    for (int b = 0; b < A; ++b) d += S.first[b];
    S.nslots = d + (a.shared ? 1 : 0);
    if (a.shared) {
      S.slot_e[0] = E;
      S.slot_n[0] = T;
      for (int t = 0; t < T; ++t) {
        S.slot_row[0][t] = A + t;
        S.slot_tok[0][t] = t;
      }
    }
  }
  __syncthreads();
  const int nslots = S.nslots;

  // block 0 publishes the routing outputs (same definitions as moe_route)
  if (blockIdx.x == 0) {
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
      for (int b = 0; b < A; ++b) {
        lt += S.ids[b] < e;
        eq += S.ids[b] == e;
      }
      if (e <= E) a.counts[e] = e < E ? eq : (a.shared ? T : 0);
      a.offsets[e] = e <= E ? lt : A + (a.shared ? T : 0);
    }
    // one tile per expert in use (counts <= T <= 4 < block_m), then the shared tile
    const int d = nslots - (a.shared ? 1 : 0);
    for (int s = tid; s < d; s += kDecThreads) {
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

  // prefetch into L2 the down rows this block reads in phase 3
  const int rows_per_blk = (H + G - 1) / G;
  const int m0 = blockIdx.x * rows_per_blk, m1 = min(H, m0 + rows_per_blk);
  {
    const int mrows = max(0, m1 - m0);
    const int row_bytes = I / 2;
    const int lines_per_row = (row_bytes + 127) / 128;
    const int total = nslots * mrows * lines_per_row;
    for (int i = tid; i < total; i += kDecThreads) {
      const int s = i / (mrows * lines_per_row), r = i - s * mrows * lines_per_row;
      const int m = m0 + r / lines_per_row, l = r % lines_per_row;
      const int e = S.slot_e[s];
      const uint32_t* codes = e == E ? a.dn.s_codes : a.dn.codes + (size_t)e * H * (I / 8);
      prefetch_l2(codes + (size_t)m * (I / 8) + l * 32);
      if (l == 0) {
        const uint16_t* sc = e == E ? a.dn.s_scales : a.dn.scales + (size_t)e * H * (I / kGroup);
        const uint16_t* bi = e == E ? a.dn.s_biases : a.dn.biases + (size_t)e * H * (I / kGroup);
        prefetch_l2(sc + (size_t)m * (I / kGroup));
        prefetch_l2(bi + (size_t)m * (I / kGroup));
      }
    }
  }

  // ---- phase 1c: gate/up units (slot, h column n), shared slot first. A warp
  // takes two units at a time and issues both units' loads before any math.
  const int units = nslots * I;
  for (int u0 = gw; u0 < units; u0 += 2 * nw) {
    uint4 cg[2][kDecMaxIt], cu[2][kDecMaxIt];
    float sg[2][kDecMaxIt], bg[2][kDecMaxIt], su[2][kDecMaxIt], bu[2][kDecMaxIt];
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const int u = u0 + b * nw;
      if (u >= units) break;
      const int s = u / I, n = u - s * I;
      const int e = S.slot_e[s];
      const bool sh = e == E;
      const uint32_t* codes = sh ? a.gu.s_codes : a.gu.codes + (size_t)e * 2 * I * (H / 8);
      const uint16_t* sc = sh ? a.gu.s_scales : a.gu.scales + (size_t)e * 2 * I * gpr;
      const uint16_t* bi = sh ? a.gu.s_biases : a.gu.biases + (size_t)e * 2 * I * gpr;
      const bool reuse = pre && u == gw;  // the shared unit loaded in phase 0
#pragma unroll
      for (int it = 0; it < kDecMaxIt; ++it) {
        const int v = lane + 32 * it;
        if (v < nvec) {
          if (reuse) {
            cg[b][it] = pc_g[it];
            cu[b][it] = pc_u[it];
            sg[b][it] = ps_g[it];
            bg[b][it] = pb_g[it];
            su[b][it] = ps_u[it];
            bu[b][it] = pb_u[it];
          } else {
            cg[b][it] = ldg_nc_v4(codes + (size_t)n * (H / 8) + 4 * v);
            cu[b][it] = ldg_nc_v4(codes + (size_t)(I + n) * (H / 8) + 4 * v);
            sg[b][it] = bf16_bits_to_f32(__ldg(sc + (size_t)n * gpr + v / 2));
            bg[b][it] = bf16_bits_to_f32(__ldg(bi + (size_t)n * gpr + v / 2));
            su[b][it] = bf16_bits_to_f32(__ldg(sc + (size_t)(I + n) * gpr + v / 2));
            bu[b][it] = bf16_bits_to_f32(__ldg(bi + (size_t)(I + n) * gpr + v / 2));
          }
        }
      }
    }
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      const int u = u0 + b * nw;
      if (u >= units) break;
      const int s = u / I, n = u - s * I;
      const int nr = S.slot_n[s];
      float ag[kDecodeMaxTokens], au[kDecodeMaxTokens];
#pragma unroll
      for (int j = 0; j < kDecodeMaxTokens; ++j) ag[j] = au[j] = 0.f;
#pragma unroll
      for (int it = 0; it < kDecMaxIt; ++it) {
        const int v = lane + 32 * it;
        if (v < nvec) {
#pragma unroll
          for (int j = 0; j < kDecodeMaxTokens; ++j) {
            if (j < nr) {
              const float* xr = xs + (S.slot_tok[s][j] * nvec + v) * kDecPad;
              ag[j] = dot32_f(cg[b][it], sg[b][it], bg[b][it], xr, ag[j]);
              au[j] = dot32_f(cu[b][it], su[b][it], bu[b][it], xr, au[j]);
            }
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kDecodeMaxTokens; ++j) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          ag[j] += __shfl_xor_sync(0xffffffffu, ag[j], o);
          au[j] += __shfl_xor_sync(0xffffffffu, au[j], o);
        }
      }
      if (lane < nr) {
        float gv = ag[0], uv = au[0];
#pragma unroll
        for (int j = 1; j < kDecodeMaxTokens; ++j)
          if (lane == j) {
            gv = ag[j];
            uv = au[j];
          }
        a.h[(size_t)S.slot_row[s][lane] * I + n] = silu_f32(gv) * uv;
      }
    }
  }

  // ---- phase 2: grid barrier (every block resident; bounded wait)
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    atomicAdd(a.bar, 1u);
    const uint64_t deadline = global_timer_ns() + (uint64_t)a.timeout_ns;
    while (ld_acquire_u32(a.bar) < (unsigned)G) {
      if (global_timer_ns() > deadline) {
        S.failed = 1;
        atomicExch(a.status, (int32_t)MOE_ERR_DEVICE_TIMEOUT);
        break;
      }
      __nanosleep(32);
    }
    __threadfence();
  }
  __syncthreads();
  if (S.failed || m0 >= H) return;

  // ---- phase 3: down projection of this block's output columns + combine
  const int R = A + (a.shared ? T : 0);
  const int ivec = I / 32, igpr = I / kGroup;
  float* hs = dsm;                                  // [R][I/32][kDecPad] (x is no longer needed)
  float* res = dsm + (size_t)R * ivec * kDecPad;    // [R][rows_per_blk]
  {
    const int hv = R * I / 4;  // float4 chunks of h; a batch of loads before any store
    for (int i0 = tid; i0 < hv; i0 += 4 * kDecThreads) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * kDecThreads;
        if (i < hv) v[u] = __ldcg(reinterpret_cast<const float4*>(a.h) + i);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * kDecThreads;
        if (i < hv) {
          const int r = (i * 4) / I, k = i * 4 - r * I;
          *reinterpret_cast<float4*>(hs + (r * ivec + (k >> 5)) * kDecPad + (k & 31)) = v[u];
        }
      }
    }
  }
  __syncthreads();
  int L = 1;  // lanes per W_down row: largest power of two <= min(32, I/32)
  while (L * 2 <= ivec && L * 2 <= 32) L *= 2;
  const int per_warp = 32 / L, sub = lane % L, rw = lane / L;
  const int its = (ivec + L - 1) / L;
  const int mrows = m1 - m0;
  const int dunits = nslots * mrows;
  constexpr int kSlots = 4;                  // (pass, load) entries issued together
  const int passes_per_batch = its >= kSlots ? 1 : kSlots / its;
  const int pass_stride = kDecWarps * per_warp;
  for (int ub0 = warp * per_warp; ub0 < dunits; ub0 += passes_per_batch * pass_stride) {
    uint4 c[kSlots];
    float sv[kSlots], bv[kSlots];
#pragma unroll
    for (int q = 0; q < kSlots; ++q) {
      const int pss = q / (its < kSlots ? its : kSlots), it = q - pss * (its < kSlots ? its : kSlots);
      const int u = ub0 + pss * pass_stride + rw;
      const int v = sub + L * it;
      if (pss < passes_per_batch && it < its && u < dunits && v < ivec) {
        const int s = u / mrows, m = m0 + (u - s * mrows);
        const int e = S.slot_e[s];
        const bool sh = e == E;
        const uint32_t* codes = sh ? a.dn.s_codes : a.dn.codes + (size_t)e * H * (I / 8);
        const uint16_t* sc = sh ? a.dn.s_scales : a.dn.scales + (size_t)e * H * igpr;
        const uint16_t* bi = sh ? a.dn.s_biases : a.dn.biases + (size_t)e * H * igpr;
        c[q] = *reinterpret_cast<const uint4*>(codes + (size_t)m * (I / 8) + 4 * v);
        sv[q] = bf16_bits_to_f32(sc[(size_t)m * igpr + v / 2]);
        bv[q] = bf16_bits_to_f32(bi[(size_t)m * igpr + v / 2]);
      }
    }
    for (int pss = 0; pss < passes_per_batch; ++pss) {
      const int u = ub0 + pss * pass_stride + rw;
      const bool live = u < dunits;
      const int s = live ? u / mrows : 0, ml = live ? u - s * mrows : 0;
      const int nr = live ? S.slot_n[s] : 0;
      float acc[kDecodeMaxTokens];
#pragma unroll
      for (int j = 0; j < kDecodeMaxTokens; ++j) acc[j] = 0.f;
#pragma unroll
      for (int q = 0; q < kSlots; ++q) {
        const int ip = its < kSlots ? its : kSlots;
        const int qp = q / ip, it = q - qp * ip;
        const int v = sub + L * it;
        if (qp == pss && it < its && live && v < ivec) {
#pragma unroll
          for (int j = 0; j < kDecodeMaxTokens; ++j)
            if (j < nr) acc[j] = dot32_f(c[q], sv[q], bv[q], hs + (S.slot_row[s][j] * ivec + v) * kDecPad, acc[j]);
        }
      }
      // more 16-byte loads than one batch holds (I > 2048): finish the row directly
      for (int it = kSlots; it < its; ++it) {
        const int v = sub + L * it;
        if (live && v < ivec) {
          const int e = S.slot_e[s];
          const bool sh = e == E;
          const int m = m0 + ml;
          const uint32_t* codes = sh ? a.dn.s_codes : a.dn.codes + (size_t)e * H * (I / 8);
          const uint16_t* sc = sh ? a.dn.s_scales : a.dn.scales + (size_t)e * H * igpr;
          const uint16_t* bi = sh ? a.dn.s_biases : a.dn.biases + (size_t)e * H * igpr;
          const uint4 cc = *reinterpret_cast<const uint4*>(codes + (size_t)m * (I / 8) + 4 * v);
          const float s1 = bf16_bits_to_f32(sc[(size_t)m * igpr + v / 2]);
          const float b1 = bf16_bits_to_f32(bi[(size_t)m * igpr + v / 2]);
#pragma unroll
          for (int j = 0; j < kDecodeMaxTokens; ++j)
            if (j < nr) acc[j] = dot32_f(cc, s1, b1, hs + (S.slot_row[s][j] * ivec + v) * kDecPad, acc[j]);
        }
      }
#pragma unroll
      for (int j = 0; j < kDecodeMaxTokens; ++j)
        for (int off = L >> 1; off > 0; off >>= 1) acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], off);
      if (live && sub == 0)
        for (int j = 0; j < nr; ++j) res[S.slot_row[s][j] * rows_per_blk + ml] = acc[j];
    }
  }
  __syncthreads();
  for (int i = tid; i < T * mrows; i += kDecThreads) {
    const int t = i / mrows, ml = i - t * mrows;
    float v = 0.f;
    for (int k = 0; k < K; ++k) v = fmaf(S.w[t * K + k], res[S.pos[t * K + k] * rows_per_blk + ml], v);
    if (a.shared) v = fmaf(S.g[t], res[(A + t) * rows_per_blk + ml], v);
    a.y[(size_t)t * H + m0 + ml] = v;
  }
}

size_t decode_smem_bytes(const Geometry& g, int rows_per_blk) {
  const int R = g.A + (g.shared ? g.T : 0);
  const size_t xs = (size_t)g.T * (g.H / 32) * kDecPad * sizeof(float);
  const size_t hs = (size_t)R * (g.I / 32) * kDecPad * sizeof(float) + (size_t)R * rows_per_blk * sizeof(float);
  return xs > hs ? xs : hs;
}

namespace {
int sm_count(int dev) {
  static int sms[64] = {0};
  if (dev < 0 || dev >= 64) return 0;
  if (sms[dev] == 0 && cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms[dev] = 0;
  return sms[dev];
}

template <int kIt>
cudaError_t launch_decode_it(const DecodeArgs& args, int grid, size_t smem, cudaStream_t stream) {
  static int configured = 0;
  cudaError_t e = ensure_smem(decode_layer_kernel<kIt>, smem, &configured);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kDecThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_layer_kernel<kIt>, args);
}
}  // namespace

// One block per SM (all resident: the grid barrier needs that).
bool decode_supported(const Geometry& g) {
  int dev = 0;
  if (g.T < 1 || g.T > kDecodeMaxTokens || g.H > 8192 || cudaGetDevice(&dev) != cudaSuccess) return false;
  const int sms = sm_count(dev);
  if (sms <= 0) return false;
  const int rows_per_blk = (g.H + sms - 1) / sms;
  return decode_smem_bytes(g, rows_per_blk) <= 200 * 1024;
}

cudaError_t launch_decode(const DecodeArgs& args, const Geometry& g, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int grid = sm_count(dev);
  if (grid <= 0) return cudaErrorInvalidDevice;
  const size_t smem = decode_smem_bytes(g, (g.H + grid - 1) / grid);
  const int its = (g.H / 32 + 31) / 32;
  if (its <= 1) return launch_decode_it<1>(args, grid, smem, stream);
  if (its <= 2) return launch_decode_it<2>(args, grid, smem, stream);
  if (its <= 4) return launch_decode_it<4>(args, grid, smem, stream);
  return launch_decode_it<8>(args, grid, smem, stream);
}

}  // namespace bgmoe
