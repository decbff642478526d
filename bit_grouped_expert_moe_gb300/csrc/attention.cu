// Single-token decode attention with grouped-query heads over a bf16 KV cache
// (sm_103a).
//
// [dothoosh.com "Perplexity Lily: 1.35x faster decode for Qwen3.6 on Apple
// silicon": "Model specification" gives the full-attention layers 16 query
// heads sharing 2 KV heads; "Decode optimisations" packs the query heads of a
// KV head into one thread group so that each cached row is read once, cuts
// the context into fixed blocks, and reads the cache with coalesced loads.]
//
// attn_block_kernel — persistent, one block per SM. The contexts of all
// (sequence, KV head) pairs are cut into fixed blocks of 64 positions, laid
// end to end in pair order (N blocks in all); block c of a grid of C takes the
// contiguous run [c*N/C, (c+1)*N/C). Warp 4 streams each block's K and V rows
// (64 x D bf16 each, 128-byte swizzle) into a 3-stage shared-memory ring by
// TMA; warps 0-3 take 16 positions each:
//   S^T  = K Q^T     mma.sync m16n8k16: M = 16 positions, N = 8 query heads
//                    (every head of the KV head at once), K = head dims;
//   online softmax per head on the base-2 scale (running max and sum);
//   P^T  fragments   the bf16 probabilities transposed in registers
//                    (movmatrix), no shared-memory round trip;
//   O^T += V^T P^T   mma.sync m16n8k16: M = 16 head dims, N = 8 heads,
//                    K = 16 positions.
// When the run leaves a pair (or ends), the four warps merge their states in
// shared memory and store one partial state per head — running maximum m,
// sum l and unnormalised output O — in slot (c + pair) of the workspace.
// Slots are unique: the blocks of the grid that cover a pair are consecutive
// and a block's pairs are consecutive, so c + pair never repeats.
//
// attn_merge_kernel — one block per (pair, head, 64 head dims) combines the
// partial states of the grid blocks that covered the pair:
//   M = max m_c,  L = sum 2^(m_c - M) l_c,  o = sum 2^(m_c - M) O_c / L.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <string.h>

#include "attention.h"
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace bgmoe {
namespace attn {

using tc::elect_one;
using tc::mbar_arrive;
using tc::mbar_arrive_expect_tx;
using tc::mbar_init;
using tc::mbar_wait;
using tc::smem_u32;

constexpr int kPos = 64;            // positions per fixed block (= ring stage)
constexpr int kStages = 3;
constexpr int kConsumers = 4;       // warps, 16 positions each
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kHeads = 8;           // MMA N: query heads of one KV head (padded)
constexpr int kMaxCtas = 256;       // workspace bound on the grid
constexpr int kSlab = kPos * 128;   // bytes of one 64-dim slab of a block (64 rows x 128 B)
constexpr long long kTimeoutNs = 1000000000ll;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kMinusBig = -1e30f; // running-max start: finite, so 2^(m - m_new) is never NaN

template <int D>
struct Smem {
  static constexpr int kSlabs = D / 64;
  static constexpr int kStageBytes = 2 * kSlabs * kSlab;  // K then V
  // A warp's softmax state as its lanes hold it: D/4 accumulators, then the
  // maxima and sums of the lane's two heads; stored [value][lane].
  static constexpr int kStateFloats = D / 4 + 4;
  static constexpr int kStateBytes = kStateFloats * 32 * 4;
  static constexpr int kMergeBytes = 3 * kStateBytes;     // warps 2, 3 (first fold) and warp 1 (second fold)
  static constexpr int kCtlOffset = kStages * kStageBytes + kMergeBytes;
  static constexpr int kBytes = kCtlOffset + 128 + 1024;  // + alignment slack
};

struct Ctl {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t mrg_full;   // first fold: warps 2 and 3 have stored their states
  uint64_t mrg_free;   // first fold: warps 0 and 1 have read them
  uint64_t mrg2_full;  // second fold: warp 1 has stored its state
  uint64_t mrg2_free;  // second fold: warp 0 has read it
  int abort;
};

struct Params {
  const uint16_t* q;
  const int32_t* lens;
  float* part;       // [slots][kHeads] m, then [slots][kHeads] l, then [slots][kHeads][D] O
  int32_t* flags;    // [C]: every grid block's outcome (0 or a moe_status), written each call
  float scale_log2;  // scale * log2(e)
  int B, Hq, Hkv, L_max, slots;
  long long timeout_ns;
  int stall_block;   // test only: this grid block's producer issues no cache loads (-1: none)
};

__device__ __forceinline__ int nblocks(int n) { return (n + kPos - 1) / kPos; }

// The grid block whose run holds fixed block s: the largest c with
// floor(c*N/C) <= s.
__device__ __forceinline__ int cta_of(long long s, long long N, int C) {
  return (int)(((s + 1) * C - 1) / N);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// d += A * B, A 16x16 (row), B 16x8 (col), bf16 in, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi, float* rlo, float* rhi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  *rlo = __low2float(v);
  *rhi = __high2float(v);
  uint32_t u;
  memcpy(&u, &v, 4);
  return u;
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// Position in the run: fixed block i of KV head g of sequence b, whose
// context has n positions (nb blocks).
struct Cursor {
  int b, g, i, n, nb;
  __device__ void advance(const Params& p) {
    if (++i < nb) return;
    i = 0;
    if (++g < p.Hkv) return;
    g = 0;
    do {
      ++b;
      n = b < p.B ? __ldg(p.lens + b) : 0;
      nb = nblocks(n);
    } while (nb == 0 && b < p.B);
  }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_block_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const Params p) {
  using S = Smem<D>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + S::kCtlOffset);
  float* mrg = reinterpret_cast<float*>(smem + kStages * S::kStageBytes);
  __shared__ long long s_lo, s_hi;
  __shared__ int s_b, s_g, s_i, s_bad;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = gridDim.x, c = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], kConsumers);
    }
    mbar_init(&ctl->mrg_full, 2);
    mbar_init(&ctl->mrg_free, 2);
    mbar_init(&ctl->mrg2_full, 1);
    mbar_init(&ctl->mrg2_free, 1);
    ctl->abort = 0;
    tc::fence_barrier_init();
  }
  if (warp == kConsumers) {
    tc::prefetch_tmap(&tm_k);
    tc::prefetch_tmap(&tm_v);
  }
  // Launched with programmatic dependent launch: the setup above overlaps the
  // previous kernel on the stream (often the previous call's merge, which
  // reads this workspace). Everything below may read what earlier kernels
  // wrote (q, the lengths, the caches) or overwrite what they read (the
  // partial states and flags), so it waits for them first. Only then may this
  // call's merge launch: it reads the lengths before its own wait.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (warp == 0) {
    // Count the fixed blocks (all pairs) and find where this block's run starts.
    long long total = 0;
    bool bad = false;
    for (int base = 0; base < p.B; base += 32) {
      const int b = base + lane;
      const int n = b < p.B ? __ldg(p.lens + b) : 0;
      bad |= n < 0 || n > p.L_max;
      long long v = n > 0 && n <= p.L_max ? nblocks(n) : 0;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      total += v;
    }
    bad = __any_sync(0xffffffffu, bad);
    total *= p.Hkv;
    const long long lo = (long long)c * total / C, hi = (long long)(c + 1) * total / C;
    int fb = 0, fg = 0, fi = 0;
    if (!bad && lo < hi) {
      long long acc = 0;
      for (int base = 0; base < p.B; base += 32) {
        const int b = base + lane;
        const long long v = b < p.B ? (long long)nblocks(__ldg(p.lens + b)) * p.Hkv : 0;
        long long incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const long long t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, acc + incl > lo);
        if (hit) {
          const int L = __ffs(hit) - 1;
          const long long before = acc + __shfl_sync(0xffffffffu, incl - v, L);
          const int nbL = nblocks(__ldg(p.lens + base + L));
          const long long off = lo - before;
          fb = base + L;
          fg = (int)(off / nbL);
          fi = (int)(off % nbL);
          break;
        }
        acc += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    if (lane == 0) {
      s_lo = lo;
      s_hi = hi;
      s_b = fb;
      s_g = fg;
      s_i = fi;
      s_bad = bad;
    }
  }
  __syncthreads();
  if (s_bad || s_lo >= s_hi) {
    if (threadIdx.x == 0) p.flags[c] = s_bad ? (int32_t)MOE_ERR_INVALID_ARG : 0;
    return;
  }
  const long long lo = s_lo, hi = s_hi;
  Cursor cur{s_b, s_g, s_i, __ldg(p.lens + s_b), 0};
  cur.nb = nblocks(cur.n);

  volatile int* abort_flag = &ctl->abort;
  const uint64_t deadline = global_timer_ns() + (uint64_t)p.timeout_ns;
  auto warp_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, deadline)) != 0;
  };

  if (warp == kConsumers) {
    // ------------------------------------------------------------ producer
    int it = 0, issued = 0;  // stages whose loads were issued (all of them unless stalled)
    const bool stalled = (int)blockIdx.x == p.stall_block;
    for (long long j = lo; j < hi; ++j, ++it) {
      const int s = it % kStages;
      if (it >= kStages && !warp_wait(&ctl->empty[s], ((it / kStages) & 1) ^ 1)) break;
      if (!stalled && elect_one()) {
        uint8_t* st = smem + s * S::kStageBytes;
        const int pair = cur.b * p.Hkv + cur.g;
        mbar_arrive_expect_tx(&ctl->full[s], (uint32_t)S::kStageBytes);
#pragma unroll
        for (int sl = 0; sl < S::kSlabs; ++sl) {
          tma_load_3d(st + sl * kSlab, &tm_k, sl * 64, cur.i * kPos, pair, &ctl->full[s]);
          tma_load_3d(st + (S::kSlabs + sl) * kSlab, &tm_v, sl * 64, cur.i * kPos, pair, &ctl->full[s]);
        }
      }
      __syncwarp();
      if (!stalled) issued = it + 1;
      cur.advance(p);
    }
    if (lane == 0 && *abort_flag) {  // let this block's own copies land before it exits
      int dummy = 0;
      const uint64_t dl = global_timer_ns() + 100000000ull;
      for (int k = issued - kStages < 0 ? 0 : issued - kStages; k < issued; ++k)
        mbar_wait(&ctl->full[k % kStages], (k / kStages) & 1, &dummy, dl);
    }
  } else {
    // ----------------------------------------------------------- consumers
    const int r = p.Hq / p.Hkv;
    const int qh = lane >> 2;          // the query head this lane feeds as an MMA column (B fragment)
    const int hA = 2 * (lane & 3);     // the two heads whose scores / outputs this lane holds
    // ldmatrix row addresses (relative to a slab): K as the A operand of S^T
    // (rows = positions), V transposed as the A operand of O^T.
    const int rowK = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8;
    const int chK = lane >> 4;
    const int rowV = 16 * warp + (lane & 7) + (lane >> 4) * 8;
    const int chV = (lane >> 3) & 1;
    const int sw = lane & 7;           // 128-byte swizzle: chunk ^= row % 8 (rows here are = lane % 8 mod 8)

    uint32_t qf[D / 16][2];
    float acc[D / 16][4];
    float mA = kMinusBig, mB = kMinusBig, lA = 0.f, lB = 0.f;
    auto load_q = [&]() {
      const bool live = qh < r;
      const uint16_t* qrow = p.q + ((size_t)cur.b * p.Hq + (size_t)cur.g * r + (live ? qh : 0)) * D;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        qf[ks][0] = live ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + hA)) : 0u;
        qf[ks][1] = live ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8 + hA)) : 0u;
      }
    };
    auto reset = [&]() {
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
      mA = mB = kMinusBig;
      lA = lB = 0.f;
    };
    reset();
    load_q();

    int it = 0, flushes = 0;
    bool ok = true;
    for (long long j = lo; j < hi; ++j, ++it) {
      const int s = it % kStages;
      if (!warp_wait(&ctl->full[s], (it / kStages) & 1)) {
        ok = false;
        break;
      }
      const uint32_t sK = smem_u32(smem + s * S::kStageBytes);
      const uint32_t sV = sK + S::kSlabs * kSlab;
      const int pos0 = cur.i * kPos + 16 * warp;  // first sequence position of this warp's 16
      if (pos0 < cur.n) {
        // S^T = K Q^T (two accumulators halve the dependent chain)
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int chunk = (ks & 3) * 2 + chK;
          uint32_t a[4];
          ldsm_x4(sK + (ks >> 2) * kSlab + rowK * 128 + ((chunk ^ sw) << 4), a);
          if (ks & 1)
            mma_bf16(sb, a, qf[ks][0], qf[ks][1]);
          else
            mma_bf16(sa, a, qf[ks][0], qf[ks][1]);
        }
        // online softmax on the base-2 scale; rows past the context are masked
        const int pr = pos0 + (lane >> 2);
        const bool v0 = pr < cur.n, v1 = pr + 8 < cur.n;
        const float x0 = v0 ? (sa[0] + sb[0]) * p.scale_log2 : -INFINITY;
        const float x1 = v0 ? (sa[1] + sb[1]) * p.scale_log2 : -INFINITY;
        const float x2 = v1 ? (sa[2] + sb[2]) * p.scale_log2 : -INFINITY;
        const float x3 = v1 ? (sa[3] + sb[3]) * p.scale_log2 : -INFINITY;
        float mxA = fmaxf(x0, x2), mxB = fmaxf(x1, x3);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, o));
          mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, o));
        }
        const float nA = fmaxf(mA, mxA), nB = fmaxf(mB, mxB);
        const float aA = exp2f(mA - nA), aB = exp2f(mB - nB);
        mA = nA;
        mB = nB;
        float r0, r1, r2, r3;
        const uint32_t p01 = pack_bf16(exp2f(x0 - nA), exp2f(x1 - nB), &r0, &r1);
        const uint32_t p23 = pack_bf16(exp2f(x2 - nA), exp2f(x3 - nB), &r2, &r3);
        lA = lA * aA + (r0 + r2);
        lB = lB * aB + (r1 + r3);
        if (__any_sync(0xffffffffu, aA != 1.f || aB != 1.f)) {
#pragma unroll
          for (int mt = 0; mt < D / 16; ++mt) {
            acc[mt][0] *= aA;
            acc[mt][1] *= aB;
            acc[mt][2] *= aA;
            acc[mt][3] *= aB;
          }
        }
        // P^T as the B fragment: rows (k) = positions, columns (n) = heads
        const uint32_t b0 = movmatrix_trans(p01), b1 = movmatrix_trans(p23);
        // V rows past the context may hold anything (even NaN): zero them
        const bool tail = pos0 + 16 > cur.n;
        const int kp = pos0 + 2 * (lane & 3);
        const uint32_t mlo = (kp < cur.n ? 0x0000FFFFu : 0u) | (kp + 1 < cur.n ? 0xFFFF0000u : 0u);
        const uint32_t mhi = (kp + 8 < cur.n ? 0x0000FFFFu : 0u) | (kp + 9 < cur.n ? 0xFFFF0000u : 0u);
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          const int chunk = (mt & 3) * 2 + chV;
          uint32_t a[4];
          ldsm_x4_trans(sV + (mt >> 2) * kSlab + rowV * 128 + ((chunk ^ sw) << 4), a);
          if (tail) {
            a[0] &= mlo;
            a[1] &= mlo;
            a[2] &= mhi;
            a[3] &= mhi;
          }
          mma_bf16(acc[mt], a, b0, b1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->empty[s]);

      if (cur.i == cur.nb - 1 || j == hi - 1) {
        // ---- the run leaves this pair: merge the four warps' states. The
        // warps hold their accumulators in the same lane layout, so a warp
        // folds another's state in lane by lane: warps 2, 3 into 0, 1, then
        // warp 1 into warp 0 (a fixed order), and warp 0 stores the result.
        float tA = lA, tB = lB;
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          tA += __shfl_xor_sync(0xffffffffu, tA, o);
          tB += __shfl_xor_sync(0xffffffffu, tB, o);
        }
        auto put = [&](float* st) {
#pragma unroll
          for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
            for (int k = 0; k < 4; ++k) st[(4 * mt + k) * 32 + lane] = acc[mt][k];
          st[(D / 4) * 32 + lane] = mA;
          st[(D / 4 + 1) * 32 + lane] = mB;
          st[(D / 4 + 2) * 32 + lane] = tA;
          st[(D / 4 + 3) * 32 + lane] = tB;
        };
        auto take = [&](const float* st) {
          const float m2A = st[(D / 4) * 32 + lane], m2B = st[(D / 4 + 1) * 32 + lane];
          const float nA = fmaxf(mA, m2A), nB = fmaxf(mB, m2B);
          const float a1A = exp2f(mA - nA), a2A = exp2f(m2A - nA);
          const float a1B = exp2f(mB - nB), a2B = exp2f(m2B - nB);
#pragma unroll
          for (int mt = 0; mt < D / 16; ++mt) {
            acc[mt][0] = acc[mt][0] * a1A + st[(4 * mt + 0) * 32 + lane] * a2A;
            acc[mt][1] = acc[mt][1] * a1B + st[(4 * mt + 1) * 32 + lane] * a2B;
            acc[mt][2] = acc[mt][2] * a1A + st[(4 * mt + 2) * 32 + lane] * a2A;
            acc[mt][3] = acc[mt][3] * a1B + st[(4 * mt + 3) * 32 + lane] * a2B;
          }
          tA = tA * a1A + st[(D / 4 + 2) * 32 + lane] * a2A;
          tB = tB * a1B + st[(D / 4 + 3) * 32 + lane] * a2B;
          mA = nA;
          mB = nB;
        };
        float* st1 = mrg + (warp & 1) * S::kStateFloats * 32;  // first-fold slot of warp 2 / warp 3
        float* st2 = mrg + 2 * S::kStateFloats * 32;           // second-fold slot
        bool fail = false;
        if (warp >= 2) {
          fail = flushes > 0 && !warp_wait(&ctl->mrg_free, (flushes - 1) & 1);
          if (!fail) {
            put(st1);
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->mrg_full);
          }
        } else {
          fail = !warp_wait(&ctl->mrg_full, flushes & 1);
          if (!fail) {
            take(st1);
            __syncwarp();
            if (lane == 0) mbar_arrive(&ctl->mrg_free);
            if (warp == 1) {
              fail = flushes > 0 && !warp_wait(&ctl->mrg2_free, (flushes - 1) & 1);
              if (!fail) {
                put(st2);
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->mrg2_full);
              }
            } else {
              fail = !warp_wait(&ctl->mrg2_full, flushes & 1);
              if (!fail) {
                take(st2);
                __syncwarp();
                if (lane == 0) mbar_arrive(&ctl->mrg2_free);
                const size_t slot = (size_t)c + cur.b * p.Hkv + cur.g;
                float* po = p.part + (size_t)2 * p.slots * kHeads + slot * kHeads * D;
#pragma unroll
                for (int mt = 0; mt < D / 16; ++mt) {
                  const int d = 16 * mt + (lane >> 2);
                  po[hA * D + d] = acc[mt][0];
                  po[(hA + 1) * D + d] = acc[mt][1];
                  po[hA * D + d + 8] = acc[mt][2];
                  po[(hA + 1) * D + d + 8] = acc[mt][3];
                }
                if (lane < 4) {
                  float* pm = p.part + slot * kHeads;
                  float* pl = p.part + (size_t)p.slots * kHeads + slot * kHeads;
                  pm[hA] = mA;
                  pm[hA + 1] = mB;
                  pl[hA] = tA;
                  pl[hA + 1] = tB;
                }
              }
            }
          }
        }
        if (fail) {
          ok = false;
          break;
        }
        ++flushes;
        reset();
        if (j + 1 < hi) {
          cur.advance(p);
          load_q();
        }
      } else {
        cur.advance(p);
      }
    }
    (void)ok;
  }
  __syncthreads();
  if (threadIdx.x == 0) p.flags[c] = *abort_flag ? (int32_t)MOE_ERR_DEVICE_TIMEOUT : 0;
}

struct MergeParams {
  const int32_t* lens;
  const float* part;
  const int32_t* flags;
  float* o;
  int32_t* status;
  int B, Hq, Hkv, D, L_max, slots, C;
};

// One block per (pair, head, 64 head dims). Thread t holds dims 4(t%16) ..
// +3 of the slice and takes the covering grid blocks c0 + t/16, c0 + t/16 + 8,
// ...: its loads of up to 8 partial states are all issued before any is
// used, then merged with a running maximum; the 8 partial lanes are merged in
// a fixed order at the end (results do not depend on timing).
constexpr int kMergeLanes = 8;
constexpr int kMergeBatch = 8;

__global__ void __launch_bounds__(128) attn_merge_kernel(const MergeParams p) {
  // The next call's block kernel may launch now: it waits for this grid to
  // finish before it touches the workspace.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // Everything up to the dependency wait reads only the lengths, which the
  // block kernel does not write (and which were final before it launched
  // this grid): it overlaps the block kernel's tail.
  const int r = p.Hq / p.Hkv;
  const int nslice = p.D / 64;
  const int slice = blockIdx.x % nslice;
  const int h = (blockIdx.x / nslice) % r;
  const int pair = blockIdx.x / (nslice * r);
  const int b = pair / p.Hkv, g = pair % p.Hkv;
  const int f = threadIdx.x & 15, pl = threadIdx.x >> 4;
  const int d = slice * 64 + 4 * f;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float4* out = reinterpret_cast<float4*>(p.o + ((size_t)b * p.Hq + (size_t)g * r + h) * p.D + d);
  __shared__ long long s_before[4], s_total[4];
  __shared__ int s_first_bad[4];
  __shared__ float s_m[kMergeLanes], s_l[kMergeLanes];
  __shared__ float4 s_o[kMergeLanes][16];
  long long before = 0, total = 0;
  bool bad = false;
  for (int bb = threadIdx.x; bb < p.B; bb += blockDim.x) {
    const int nbb = __ldg(p.lens + bb);
    bad |= nbb < 0 || nbb > p.L_max;
    const long long v = nblocks(nbb);
    total += v;
    if (bb < b) before += v;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    before += __shfl_xor_sync(0xffffffffu, before, o);
    total += __shfl_xor_sync(0xffffffffu, total, o);
  }
  if (lane == 0) {
    s_before[warp] = before;
    s_total[warp] = total;
  }
  bad = __syncthreads_or(bad);
  before = s_before[0] + s_before[1] + s_before[2] + s_before[3];
  total = s_total[0] + s_total[1] + s_total[2] + s_total[3];
  const int n = __ldg(p.lens + b);
  const int nb = bad ? 0 : nblocks(n);
  const long long N = total * p.Hkv, start = before * p.Hkv + (long long)g * nb;
  const int c0 = nb ? cta_of(start, N, p.C) : 0, c1 = nb ? cta_of(start + nb - 1, N, p.C) : -1;

  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (blockIdx.x == 0) {
    // the call's status: the outcome of the lowest-numbered grid block that failed
    int first = 0x7fffffff;
    for (int cc = threadIdx.x; cc < p.C; cc += blockDim.x)
      if (__ldcg(p.flags + cc) != 0) first = min(first, cc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) first = min(first, __shfl_xor_sync(0xffffffffu, first, o));
    if (lane == 0) s_first_bad[warp] = first;
    __syncthreads();
    if (threadIdx.x == 0) {
      first = min(min(s_first_bad[0], s_first_bad[1]), min(s_first_bad[2], s_first_bad[3]));
      *p.status = first == 0x7fffffff ? 0 : __ldcg(p.flags + first);
    }
  }
  if (bad) return;
  if (nb == 0) {
    if (pl == 0) *out = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }

  const float* pm = p.part;
  const float* pl_ = p.part + (size_t)p.slots * kHeads;
  const float* po = p.part + (size_t)2 * p.slots * kHeads;
  float M = kMinusBig, L = 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  int failed = 0;
  for (int base = c0 + pl; base <= c1; base += kMergeLanes * kMergeBatch) {
    float mc[kMergeBatch], lc[kMergeBatch];
    float4 oc[kMergeBatch];
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      const int cc = base + u * kMergeLanes;
      // with fewer fixed blocks than grid blocks some runs are empty (no slot written)
      const bool live = cc <= c1 && (long long)cc * N / p.C != (long long)(cc + 1) * N / p.C;
      const size_t slot = (size_t)(live ? cc : c0) + pair;
      failed |= live ? __ldcg(p.flags + cc) : 0;
      mc[u] = live ? __ldcg(pm + slot * kHeads + h) : kMinusBig;
      lc[u] = live ? __ldcg(pl_ + slot * kHeads + h) : 0.f;
      oc[u] = live ? __ldcg(reinterpret_cast<const float4*>(po + (slot * kHeads + h) * p.D + d))
                   : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      const float nm = fmaxf(M, mc[u]);
      const float fo = exp2f(M - nm), fc = exp2f(mc[u] - nm);
      O.x = O.x * fo + oc[u].x * fc;
      O.y = O.y * fo + oc[u].y * fc;
      O.z = O.z * fo + oc[u].z * fc;
      O.w = O.w * fo + oc[u].w * fc;
      L = L * fo + lc[u] * fc;
      M = nm;
    }
  }
  if (f == 0) {
    s_m[pl] = M;
    s_l[pl] = L;
  }
  s_o[pl][f] = O;
  if (__syncthreads_or(failed)) return;  // a covering grid block gave up: o is left as it was
  if (pl == 0) {
    float Mt = kMinusBig;
#pragma unroll
    for (int w = 0; w < kMergeLanes; ++w) Mt = fmaxf(Mt, s_m[w]);
    float Lt = 0.f;
    float4 Ot = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kMergeLanes; ++w) {
      const float e = exp2f(s_m[w] - Mt);
      Lt += e * s_l[w];
      Ot.x += e * s_o[w][f].x;
      Ot.y += e * s_o[w][f].y;
      Ot.z += e * s_o[w][f].z;
      Ot.w += e * s_o[w][f].w;
    }
    const float inv = 1.f / Lt;
    *out = make_float4(Ot.x * inv, Ot.y * inv, Ot.z * inv, Ot.w * inv);
  }
}

// ================================================================= host ===

PFN_cuTensorMapEncodeTiled_v12000 attn_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 3-D map of a cache [pairs][L_max][D] (bf16) with 64 x 64 boxes, 128-byte
// swizzle; rows past L_max read as zeros.
cudaError_t cache_map(CUtensorMap* m, const void* base, int D, int L_max, int pairs) {
  auto fn = attn_encode_fn();
  if (!fn) return cudaErrorNotSupported;
  memset(m, 0, sizeof(*m));
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)L_max, (cuuint64_t)pairs};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)L_max * D * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)kPos, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int attn_sm_count() {
  static int sms[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (sms[dev] == 0 && cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms[dev] = 0;
  return sms[dev];
}

bool shape_ok(const moe_attn_shape& s) {
  if (s.B < 1 || s.B > 4096 || s.Hkv < 1 || s.Hq < 1 || s.Hq % s.Hkv != 0) return false;
  const int r = s.Hq / s.Hkv;
  if (r > kHeads || (long long)s.B * s.Hkv > 65536) return false;
  if (s.D != 64 && s.D != 128 && s.D != 256) return false;
  return s.L_max >= 1 && s.L_max <= (1 << 26);
}

size_t workspace_bytes(const moe_attn_shape& s) {
  const size_t slots = (size_t)kMaxCtas + (size_t)s.B * s.Hkv;
  return 256 + kMaxCtas * sizeof(int32_t) + slots * kHeads * (2 + (size_t)s.D) * sizeof(float);
}

template <int D>
cudaError_t launch(const moe_attn_shape& s, const CUtensorMap& tk, const CUtensorMap& tv, const Params& prm,
                   int grid, bool early, cudaStream_t stream) {
  static SmemLimitMemo smem_memo;
  cudaError_t e = ensure_smem(attn_block_kernel<D>, Smem<D>::kBytes, &smem_memo);
  if (e != cudaSuccess) return e;
  // With `early`, programmatic dependent launch: the kernel waits for its
  // predecessors itself, after its setup. Otherwise an ordinary launch (the
  // wait then returns at once).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Smem<D>::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = early ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attn_block_kernel<D>, tk, tv, prm);
}

moe_status fail(cudaError_t e, const char* where) { return cuda_fail(e, where); }

// An event record that also works inside a stream capture (as an external
// event node of the graph).
cudaError_t record(void* ev, cudaStream_t s) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cap);
  if (e != cudaSuccess) return e;
  return cap == cudaStreamCaptureStatusActive
             ? cudaEventRecordWithFlags(static_cast<cudaEvent_t>(ev), s, cudaEventRecordExternal)
             : cudaEventRecord(static_cast<cudaEvent_t>(ev), s);
}

moe_status decode(const moe_attn_shape* shape, const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* lens, float scale, float* o, void* workspace, size_t ws_bytes, void* const* events,
                  void* stream_, int stall_block = -1, long long timeout_ns = kTimeoutNs) {
  if (!shape) return MOE_ERR_INVALID_ARG;
  const moe_attn_shape s = *shape;
  if (!shape_ok(s)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!q || !k_cache || !v_cache || !lens || !o || !workspace) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
       reinterpret_cast<uintptr_t>(v_cache)) & 15)
    return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(o) & 15) || (reinterpret_cast<uintptr_t>(lens) & 3) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255))
    return MOE_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !(scale < INFINITY)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < workspace_bytes(s)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const int sms = attn_sm_count();
  if (sms <= 0) return fail(cudaErrorInvalidDevice, "device query");
  const int grid = sms < kMaxCtas ? sms : kMaxCtas;
  const int pairs = s.B * s.Hkv;

  CUtensorMap tk, tv;
  cudaError_t e = cache_map(&tk, k_cache, s.D, s.L_max, pairs);
  if (e == cudaSuccess) e = cache_map(&tv, v_cache, s.D, s.L_max, pairs);
  if (e != cudaSuccess) return fail(e, "tensor map");

  int32_t* status = static_cast<int32_t*>(workspace);
  int32_t* flags = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + 256);
  float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + 256 + kMaxCtas * sizeof(int32_t));
  const int slots = kMaxCtas + pairs;
  Params prm{static_cast<const uint16_t*>(q), lens, part, flags, scale * kLog2e, s.B, s.Hq, s.Hkv, s.L_max, slots,
             timeout_ns, stall_block};
  if (events && (e = record(events[0], stream)) != cudaSuccess)
    return fail(e, "event record");
  // The block kernel starts early (beside the previous call's merge) only
  // when a merge grid fits on the SMs in one wave: an early block takes the
  // shared memory a waiting merge block would need, so a larger merge (a
  // batch of sequences) would run in more waves (measured at batch8:
  // 53.28 -> 53.77 us per layer early, against 22.82 -> 22.64 at 32K). The
  // call's own merge size stands for its predecessor's: calls in a sequence
  // share their shape.
  const int merge_blocks = pairs * (s.Hq / s.Hkv) * (s.D / 64);
  const bool early = merge_blocks <= sms;
  switch (s.D) {
    case 64: e = launch<64>(s, tk, tv, prm, grid, early, stream); break;
    case 128: e = launch<128>(s, tk, tv, prm, grid, early, stream); break;
    default: e = launch<256>(s, tk, tv, prm, grid, early, stream); break;
  }
  if (e != cudaSuccess) return fail(e, "block kernel launch");
  if (events && (e = record(events[1], stream)) != cudaSuccess)
    return fail(e, "event record");

  MergeParams mp{lens, part, flags, o, status, s.B, s.Hq, s.Hkv, s.D, s.L_max, slots, grid};
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(pairs * (s.Hq / s.Hkv) * (s.D / 64)));
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if ((e = cudaLaunchKernelEx(&cfg, attn_merge_kernel, mp)) != cudaSuccess) return fail(e, "merge kernel launch");
  if (events && (e = record(events[2], stream)) != cudaSuccess)
    return fail(e, "event record");
  return MOE_OK;
}

}  // namespace attn
}  // namespace bgmoe

using namespace bgmoe::attn;

extern "C" {

moe_status moe_attn_workspace_bytes(const moe_attn_shape* shape, size_t* bytes) {
  if (!shape || !bytes) return MOE_ERR_INVALID_ARG;
  if (!shape_ok(*shape)) return MOE_ERR_UNSUPPORTED_SHAPE;
  *bytes = workspace_bytes(*shape);
  return MOE_OK;
}

moe_status moe_attn_decode(const moe_attn_shape* shape, const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* lens, float scale, float* o, void* workspace, size_t ws_bytes,
                           void* stream) {
  return decode(shape, q, k_cache, v_cache, lens, scale, o, workspace, ws_bytes, nullptr, stream);
}

moe_status moe_attn_decode_timed(const moe_attn_shape* shape, const void* q, const void* k_cache,
                                 const void* v_cache, const int32_t* lens, float scale, float* o, void* workspace,
                                 size_t ws_bytes, void* const* events, void* stream) {
  if (!events || !events[0] || !events[1] || !events[2]) return MOE_ERR_INVALID_ARG;
  return decode(shape, q, k_cache, v_cache, lens, scale, o, workspace, ws_bytes, events, stream);
}

moe_status moe_attn_test_stall(const moe_attn_shape* shape, const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* lens, float scale, float* o, void* workspace, size_t ws_bytes,
                               int32_t stalled_block, int64_t timeout_ns, void* stream) {
  if (stalled_block < 0 || timeout_ns <= 0 || timeout_ns > kTimeoutNs) return MOE_ERR_INVALID_ARG;
  return decode(shape, q, k_cache, v_cache, lens, scale, o, workspace, ws_bytes, nullptr, stream, stalled_block,
                timeout_ns);
}

}  // extern "C"
