// GPU-resident routing in one launch: top-k selection and weights, expert
// histogram, decoupled look-back prefix scan across blocks, stable scatter
// into expert-contiguous order, and the tile block map.
// [dothoosh.com "Perplexity Lily: 1.35x faster decode for Qwen3.6 on Apple
// silicon", "Prefill optimisations", GPU-resident routing item: histogram,
// prefix scan, scatter and block map in one GPU submission, no CPU sync.
// "Model specification": 256 experts scored, 8 picked, plus a shared expert.]
//
// Block b owns tokens [b*tpb, (b+1)*tpb) and so the assignments
// a = t*K + k of those tokens, a contiguous range. Stable positions follow
// from counts alone: pos(a) = offsets[e] + (assignments of e in earlier
// blocks) + (in earlier warps of this block) + (earlier in this warp step),
// so the result never depends on atomic ordering.
//
// Cross-block exchange: one 64-bit word per (block, expert) holds a flag in
// the high half (1 = block aggregate, 2 = inclusive prefix) and the count in
// the low half, so a single relaxed load sees both. Every wait is bounded by
// timeout_ns; on expiry the block writes MOE_ERR_DEVICE_TIMEOUT to the status
// word and returns. The grid is launched cooperatively, so all blocks are
// resident and the last block's inclusive prefix (the expert totals) is
// always produced.
#include "kernels.h"

namespace bgmoe {

constexpr int kRouteThreads = 512;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr unsigned long long kFlagAggregate = 1ull << 32;
constexpr unsigned long long kFlagInclusive = 2ull << 32;

// Exclusive scan of one int per thread over the block; returns the thread's
// exclusive prefix and writes the block total to *total.
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int s = lane < kRouteWarps ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += n;
    }
    if (lane < kRouteWarps) warp_sums[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const int before = warp > 0 ? warp_sums[warp - 1] : 0;
  *total = warp_sums[kRouteWarps - 1];
  __syncthreads();
  return before + incl - v;
}

__global__ void __launch_bounds__(kRouteThreads) route_kernel(RouteArgs a) {
  extern __shared__ __align__(16) int smem[];
  const int E = a.E, K = a.K;
  int* ids_s = smem;                          // [tpb*K]
  int* hist = ids_s + a.tpb * K;              // [warps][E]: counts, then running bases
  int* prefix_s = hist + kRouteWarps * E;     // [E] assignments of e in earlier blocks
  int* total_s = prefix_s + E;                // [E] assignments of e overall
  int* offs_s = total_s + E;                  // [E+2]
  int* tbase_s = offs_s + E + 2;              // [E+2] first tile of each expert
  int* scratch = tbase_s + E + 2;             // [kRouteWarps + 2]
  __shared__ int failed_s;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int blk = blockIdx.x, P = a.P;
  const int t0 = blk * a.tpb;
  const int nt = max(0, min(a.tpb, a.T - t0));
  const int A = a.T * K;
  if (tid == 0) failed_s = 0;

  // ---- top-k, renormalised softmax weights and shared gate (warp per token)
  for (int tl = warp; tl < nt; tl += kRouteWarps) {
    const int t = t0 + tl;
    int e;
    float w, g;
    warp_topk(a.logits + (size_t)t * (E + 1), a.bias, E, K, a.shared != 0, lane, &e, &w, &g);
    if (lane < K) {
      a.ids[(size_t)t * K + lane] = e;
      a.weights[(size_t)t * K + lane] = w;
      ids_s[tl * K + lane] = e;
    }
    if (lane == 0 && a.shared) a.gate[t] = g;
  }
  for (int i = tid; i < kRouteWarps * E; i += kRouteThreads) hist[i] = 0;
  __syncthreads();

  // ---- per-warp histograms of this block's assignments (warp-aggregated:
  // lanes holding the same expert elect one leader that adds the group size)
  const int na = nt * K;
  const int cw = (na + kRouteWarps - 1) / kRouteWarps;
  const int lo = warp * cw, hi = min(na, lo + cw);
  for (int base = lo; base < hi; base += 32) {
    const int i = base + lane;
    const bool valid = i < hi;
    const int e = valid ? ids_s[i] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (valid && lane == __ffs(peers) - 1) hist[warp * E + e] += __popc(peers);
  }
  __syncthreads();

  // ---- decoupled look-back over blocks, one expert per thread
  if (tid < E) {
    const int e = tid;
    int run = 0;
    for (int w = 0; w < kRouteWarps; ++w) {
      const int c = hist[w * E + e];
      hist[w * E + e] = run;
      run += c;
    }
    const int local = run;
    bool fail = false;
    unsigned long long* st = a.state;
    if (blk != a.stalled_block) st_relaxed_u64(&st[(size_t)blk * E + e], kFlagAggregate | (uint32_t)local);
    int prefix = 0;
    if (blk > 0) {
      int j = blk - 1;
      const uint64_t deadline = global_timer_ns() + (uint64_t)a.timeout_ns;
      while (true) {
        const unsigned long long v = ld_relaxed_u64(&st[(size_t)j * E + e]);
        const unsigned long long f = v & 0xFFFFFFFF00000000ull;
        if (f == kFlagInclusive) {
          prefix += (int)(uint32_t)v;
          break;
        }
        if (f == kFlagAggregate) {
          prefix += (int)(uint32_t)v;
          if (--j < 0) break;
          continue;
        }
        if (global_timer_ns() > deadline) {
          fail = true;
          break;
        }
        __nanosleep(64);
      }
    }
    int total = 0;
    if (!fail) {
      if (blk != a.stalled_block)
        st_relaxed_u64(&st[(size_t)blk * E + e], kFlagInclusive | (uint32_t)(prefix + local));
      if (blk == P - 1) {
        total = prefix + local;
      } else {
        const uint64_t deadline = global_timer_ns() + (uint64_t)a.timeout_ns;
        while (true) {
          const unsigned long long v = ld_relaxed_u64(&st[(size_t)(P - 1) * E + e]);
          if ((v & 0xFFFFFFFF00000000ull) == kFlagInclusive) {
            total = (int)(uint32_t)v;
            break;
          }
          if (global_timer_ns() > deadline) {
            fail = true;
            break;
          }
          __nanosleep(64);
        }
      }
    }
    prefix_s[e] = prefix;
    total_s[e] = total;
    if (fail) {
      failed_s = 1;
      atomicExch(a.status, (int32_t)MOE_ERR_DEVICE_TIMEOUT);
    }
  }
  __syncthreads();
  if (failed_s) return;

  // ---- expert offsets and tile bases (exclusive scans over the E+1 groups)
  int tot;
  {
    const int v = tid < E ? total_s[tid] : 0;
    const int ex = block_exclusive_scan(v, scratch, &tot);
    if (tid < E) offs_s[tid] = ex;
    if (tid == 0) {
      offs_s[E] = A;
      offs_s[E + 1] = A + (a.shared ? a.T : 0);
    }
  }
  {
    int ntl = 0;
    if (tid < E) ntl = (total_s[tid] + a.BM - 1) / a.BM;
    else if (tid == E && a.shared) ntl = (a.T + a.BM - 1) / a.BM;
    const int ex = block_exclusive_scan(ntl, scratch, &tot);
    if (tid <= E) tbase_s[tid] = ex;
    if (tid == 0) tbase_s[E + 1] = tot;
  }
  __syncthreads();

  // ---- stable scatter: warps walk their ranges in order
  for (int base = lo; base < hi; base += 32) {
    const int i = base + lane;
    const bool valid = i < hi;
    const int e = valid ? checked(ids_s[i], 0, E - 1, a.status) : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    if (valid) {
      const int pos = checked(offs_s[e] + prefix_s[e] + hist[warp * E + e] + __popc(peers & lanemask_lt()), 0,
                              a.T * K - 1, a.status);
      const int ag = t0 * K + i;
      a.sorted[pos] = ag;
      a.inv[ag] = pos;
    }
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) hist[warp * E + e] += __popc(peers);
    __syncwarp();
  }

  // ---- the last block publishes counts, offsets and the block map
  if (blk == P - 1) {
    const int ntiles = tbase_s[E + 1];
    for (int e = tid; e <= E; e += kRouteThreads)
      a.counts[e] = e < E ? total_s[e] : (a.shared ? a.T : 0);
    for (int e = tid; e <= E + 1; e += kRouteThreads) a.offsets[e] = offs_s[e];
    if (tid == 0) *a.num_tiles = ntiles;
    for (int idx = tid; idx < ntiles; idx += kRouteThreads) {
      int lo_e = 0, hi_e = E;  // largest e in [0, E] with tbase_s[e] <= idx
      while (lo_e < hi_e) {
        const int mid = (lo_e + hi_e + 1) >> 1;
        if (tbase_s[mid] <= idx) lo_e = mid;
        else hi_e = mid - 1;
      }
      const int e = lo_e;
      const int j = idx - tbase_s[e];
      const int cnt = e < E ? total_s[e] : a.T;
      a.tile_expert[idx] = e;
      a.tile_row0[idx] = offs_s[e] + j * a.BM;
      a.tile_rows[idx] = min(a.BM, cnt - j * a.BM);
    }
  }
}

size_t route_smem_bytes(const Geometry& g) {
  return sizeof(int) * ((size_t)g.tokens_per_block * g.K + (size_t)kRouteWarps * g.E + 2 * (size_t)g.E +
                        2 * ((size_t)g.E + 2) + kRouteWarps + 2);
}

cudaError_t launch_route(const RouteArgs& a, cudaStream_t stream) {
  Geometry g{};
  g.tokens_per_block = a.tpb;
  g.K = a.K;
  g.E = a.E;
  const size_t smem = route_smem_bytes(g);
  static SmemLimitMemo smem_memo;
  cudaError_t err = ensure_smem(route_kernel, smem, &smem_memo);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.P);
  cfg.blockDim = dim3(kRouteThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, route_kernel, a);
}

}  // namespace bgmoe
