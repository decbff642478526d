// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05, TMEM
// accumulators) with 4-bit dequantisation fused into the mainloop.
// [dothoosh.com "Perplexity Lily: 1.35x faster decode for Qwen3.6 on Apple
// silicon", "Prefill optimisations", fused dequantisation: the grouped GEMM
// rebuilds the 4-bit group-64 weights tile by tile in on-chip memory and
// accumulates in FP32, so the dequantised array never goes back to memory;
// "tiling": tiles of more token rows per weight tile (16 -> 32 rows) paid.]
//
// Orientation (swap-AB): the weights are the MMA's M operand (128 rows per
// MMA) and the tile's token rows are N (16..128, rounded up to 16), so a
// small expert group wastes at most 15 token columns, not a 128-row tile.
// Both operands are fp16, K-major, in the 128-byte swizzled layout; the
// dequantised weights are rounded once to fp16 (W = scale*q + bias in one fp16
// FMA), and x and h carry the same in-group K permutation (0,4,1,5,2,6,3,7)
// that the nibble unpacking produces.
//
// Warp roles (512 threads):
//   warp 0      TMA producer: 4-bit code tiles (and, for the down GEMM, the
//               resident h tile)
//   warp 1      TMEM allocation and the single MMA-issuing thread
//   warps 2-3   gate/up only: gather of the tile's token rows of x (cp.async)
//   warps 4-11  dequantisation: codes -> fp16 weights in the swizzled layout
//   warps 12-15 epilogue: tcgen05.ld -> silu(gate)*up -> h (gate/up), or
//               -> o (down)
// Every mbarrier wait is bounded; on expiry the block raises an abort flag,
// drains its own copies, frees its TMEM and reports MOE_ERR_DEVICE_TIMEOUT.
#include <cudaTypedefs.h>

#include <cstring>

#include "kernels.h"
#include "tc_ptx.cuh"

namespace bgmoe {
using namespace tc;

constexpr int kTcThreads = 512;
constexpr int kStages = 3;
constexpr int kMaxBN = 128;          // token rows per tile (block_m <= 128)
constexpr int kTmemCols = 256;

// ----------------------------------------------------- shared layouts ---
// gate/up: per stage A = 256 weight rows x 64 k (gate 128 | up 128, 32 KB),
// B = 128 token rows x 64 k (16 KB), codes 256 rows x 32 B (8 KB).
constexpr int kGuA = 32768, kGuB = 16384, kGuC = 8192;
constexpr int kGuStage = kGuA + kGuB + kGuC;
// down: per stage A = 128 rows x 64 k (16 KB), codes 128 x 32 B (4 KB); the
// tile's h rows stay resident (I/64 boxes of block_m x 64).
constexpr int kDnA = 16384, kDnC = 4096;
constexpr int kDnStage = kDnA + kDnC;
constexpr int kMaxResidentH = 131072;

struct Ctl {                 // control block after the data
  uint64_t bar[4 * kStages + 8];
  int tok[kMaxBN];
  uint32_t tmem;
  int abort;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + (((a + 1023u) & ~1023u) - a);
}

__device__ __forceinline__ __half2 bf16_to_h2(uint32_t bits16) {
  const __half h = __float2half_rn(bf16_bits_to_f32(bits16));
  return __halves2half2(h, h);
}

__device__ __forceinline__ uint32_t u4_get(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// bf16 element g (0..7) of an 8-element uint4
__device__ __forceinline__ uint32_t bf16_of(const uint4& v, int g) {
  const uint32_t w = u4_get(v, g >> 1);
  return (g & 1) ? (w >> 16) : (w & 0xFFFFu);
}

// ============================================================ gate / up ===

struct GateUpTcParams {
  int H, I, E, K, A;
  const uint16_t* x16;       // [T][H] fp16 bits, K-permuted within groups of 8
  const uint16_t* scales;    // routed [E][2I][H/64] bf16
  const uint16_t* biases;
  const uint16_t* s_scales;  // shared [2I][H/64]
  const uint16_t* s_biases;
  TileArgs t;
  __half* h;                 // [rows][I], K-permuted within groups of 8
  int32_t* status;
  long long timeout_ns;
};

__global__ void __launch_bounds__(kTcThreads, 1)
gate_up_tc_kernel(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_s_codes,
                  const GateUpTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  const int tile = blockIdx.x, nb = blockIdx.y;
  if (device_failed(p.t.status) || tile >= *p.t.num_tiles) return;

  uint8_t* sm = align1024(smem_raw);
  uint8_t* sA = sm;
  uint8_t* sB = sA + kStages * kGuA;
  uint8_t* sC = sB + kStages * kGuB;
  Ctl* ctl = reinterpret_cast<Ctl*>(sC + kStages * kGuC);
  uint64_t* full_c = ctl->bar;
  uint64_t* a_full = full_c + kStages;
  uint64_t* b_full = a_full + kStages;
  uint64_t* empty = b_full + kStages;
  uint64_t* acc_full = empty + kStages;
  volatile int* abort_flag = &ctl->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = p.t.tile_expert[tile], row0 = p.t.tile_row0[tile], rows = p.t.tile_rows[tile];
  const bool sh = e == p.E;
  const int N = (rows + 15) & ~15;
  const int num_k = p.H / 64;
  const int I = p.I, H = p.H;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_c[s], 1);
      mbar_init(&a_full[s], 8);
      mbar_init(&b_full[s], 2);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    ctl->abort = 0;
    fence_barrier_init();
  }
  if (threadIdx.x < kMaxBN) {
    const int j = threadIdx.x;
    const int r = row0 + j;
    ctl->tok[j] = j < rows ? (r < p.A ? p.t.sorted[r] / p.K : r - p.A) : 0;
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;
  const uint64_t deadline = global_timer_ns() + (uint64_t)p.timeout_ns;

  if (warp == 0) {
    // ---------------------------------------------------- TMA producer
    if (lane == 0) {
      const CUtensorMap* map = sh ? &tm_s_codes : &tm_codes;
      prefetch_tmap(map);
      const int gate_row = (sh ? 0 : e * 2 * I) + nb * 128;
      int issued = 0;
      for (int it = 0; it < num_k; ++it) {
        const int s = it % kStages;
        if (it >= kStages && !mbar_wait(&empty[s], ((it / kStages) - 1) & 1, abort_flag, deadline)) break;
        mbar_arrive_expect_tx(&full_c[s], 8192);
        tma_load_2d(sC + s * kGuC, map, it * 8, gate_row, &full_c[s]);
        tma_load_2d(sC + s * kGuC + 4096, map, it * 8, gate_row + I, &full_c[s]);
        issued = it + 1;
      }
      if (*abort_flag) {  // let our own copies land before the block exits
        const uint64_t dl = global_timer_ns() + 100000000ull;
        int dummy = 0;
        for (int it = issued - kStages < 0 ? 0 : issued - kStages; it < issued; ++it)
          mbar_wait(&full_c[it % kStages], (it / kStages) & 1, &dummy, dl);
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_f32(128, N);
      for (int it = 0; it < num_k; ++it) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        if (!mbar_wait(&a_full[s], ph, abort_flag, deadline)) break;
        if (!mbar_wait(&b_full[s], ph, abort_flag, deadline)) break;
        tc_fence_after();
        const uint32_t a_g = smem_u32(sA + s * kGuA), a_u = a_g + 16384, b = smem_u32(sB + s * kGuB);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t acc = (it | kk) != 0;
          mma_f16(tmem, sw128_desc(a_g + kk * 32), sw128_desc(b + kk * 32), idesc, acc);
          mma_f16(tmem + 128, sw128_desc(a_u + kk * 32), sw128_desc(b + kk * 32), idesc, acc);
        }
        mma_commit(&empty[s]);
      }
      mma_commit(acc_full);  // arrives once every issued MMA has finished
    }
  } else if (warp < 4) {
    // ------------------------------------------- gather of x token rows
    const int gt = threadIdx.x - 64;
    constexpr int D = kStages - 1;  // stages in flight before publishing
    const int chunks = N * 8;
    int it = 0;
    for (; it < num_k; ++it) {
      const int s = it % kStages;
      if (it >= kStages && !mbar_wait(&empty[s], ((it / kStages) - 1) & 1, abort_flag, deadline)) break;
      uint8_t* dst = sB + s * kGuB;
      for (int idx = gt; idx < chunks; idx += 64) {
        const int j = idx >> 3, c = idx & 7;
        const uint16_t* src = p.x16 + (size_t)ctl->tok[j] * H + it * 64 + c * 8;
        cp_async_16(dst + j * 128 + ((c ^ (j & 7)) << 4), src, j < rows ? 16u : 0u);
      }
      cp_async_commit();
      if (it >= D) {
        cp_async_wait<D>();
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(&b_full[(it - D) % kStages]);
      }
    }
    cp_async_wait<0>();
    fence_proxy_async();
    __syncwarp();
    if (lane == 0)
      for (int j2 = (it - D > 0 ? it - D : 0); j2 < it; ++j2) mbar_arrive(&b_full[j2 % kStages]);
  } else if (warp < 12) {
    // ------------------------------------------------ dequantisation
    const int r = threadIdx.x - 128;  // 0..255: gate rows 0..127, up rows 128..255
    const int wrow = (r < 128 ? 0 : I) + nb * 128 + (r & 127);
    const size_t grow = sh ? (size_t)wrow : (size_t)e * 2 * I + wrow;
    const int gpr = H / 64;
    const uint16_t* srow = (sh ? p.s_scales : p.scales) + grow * gpr;
    const uint16_t* brow = (sh ? p.s_biases : p.biases) + grow * gpr;
    uint8_t* arow = sA + (r < 128 ? 0 : 16384) + (r & 127) * 128;
    const uint8_t* crow = sC + (r < 128 ? 0 : 4096) + (r & 127) * 32;
    uint4 sc = ldg_nc_v4(srow), bi = ldg_nc_v4(brow);
    uint4 sc_n = sc, bi_n = bi;
    if (gpr > 8) {
      sc_n = ldg_nc_v4(srow + 8);
      bi_n = ldg_nc_v4(brow + 8);
    }
    for (int it = 0; it < num_k; ++it) {
      const int s = it % kStages;
      if ((it & 7) == 0 && it > 0) {
        sc = sc_n;
        bi = bi_n;
        if (it + 8 < gpr) {
          sc_n = ldg_nc_v4(srow + it + 8);
          bi_n = ldg_nc_v4(brow + it + 8);
        }
      }
      const __half2 s2 = bf16_to_h2(bf16_of(sc, it & 7));
      const __half2 b2 = bf16_to_h2(bf16_of(bi, it & 7));
      if (!mbar_wait(&full_c[s], (it / kStages) & 1, abort_flag, deadline)) break;
      const uint4 c0 = *reinterpret_cast<const uint4*>(crow + s * kGuC);
      const uint4 c1 = *reinterpret_cast<const uint4*>(crow + s * kGuC + 16);
      uint8_t* dst = arow + s * kGuA;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        uint32_t o[4];
        dequant8_f16(q < 4 ? u4_get(c0, q) : u4_get(c1, q - 4), s2, b2, o);
        *reinterpret_cast<uint4*>(dst + ((q ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[s]);
    }
  } else {
    // ------------------------------------------------------- epilogue
    const int q = warp & 3;
    if (mbar_wait(acc_full, 0, abort_flag, deadline)) {
      tc_fence_after();
      const int n = nb * 128 + q * 32 + lane;
      const int pn = perm8_pos(n);
      const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
      for (int j0 = 0; j0 < N; j0 += 32) {
        float g[32], u[32];
        tmem_ld_32(lane_addr + j0, g);
        tmem_ld_32(lane_addr + 128 + j0, u);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int j = j0 + jj;
          if (j < rows) p.h[(size_t)(row0 + j) * I + pn] = __float2half_rn(silu_f32(g[jj]) * u[jj]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (*abort_flag) {  // no MMA may still be running when TMEM is freed
      int dummy = 0;
      mbar_wait(acc_full, 0, &dummy, global_timer_ns() + 100000000ull);
    }
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicExch(p.status, (int32_t)MOE_ERR_DEVICE_TIMEOUT);
}

// ================================================================= down ===

struct DownTcParams {
  int H, I, E, BM, mb_per_cta;
  const uint16_t* scales;    // routed [E][H][I/64] bf16
  const uint16_t* biases;
  const uint16_t* s_scales;  // shared [H][I/64]
  const uint16_t* s_biases;
  TileArgs t;
  __half* o;                 // [rows][H]
  int32_t* status;
  long long timeout_ns;
};

__global__ void __launch_bounds__(kTcThreads, 1)
down_tc_kernel(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_s_codes,
               const __grid_constant__ CUtensorMap tm_h, const DownTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  const int tile = blockIdx.x;
  if (device_failed(p.t.status) || tile >= *p.t.num_tiles) return;

  const int I = p.I, H = p.H;
  const int num_k = I / 64;
  const int hbox = p.BM * 128;  // bytes of one resident h box (BM rows x 64 fp16)
  uint8_t* sm = align1024(smem_raw);
  uint8_t* sH = sm;
  uint8_t* sA = sH + num_k * hbox;
  uint8_t* sC = sA + kStages * kDnA;
  Ctl* ctl = reinterpret_cast<Ctl*>(sC + kStages * kDnC);
  uint64_t* full_c = ctl->bar;
  uint64_t* a_full = full_c + kStages;
  uint64_t* empty = a_full + kStages;
  uint64_t* h_full = empty + kStages;
  uint64_t* acc_full = h_full + 1;   // [2]
  uint64_t* acc_empty = acc_full + 2; // [2]
  uint64_t* mma_done = acc_empty + 2;
  volatile int* abort_flag = &ctl->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = p.t.tile_expert[tile], row0 = p.t.tile_row0[tile], rows = p.t.tile_rows[tile];
  const bool sh = e == p.E;
  const int N = (rows + 15) & ~15;
  const int mb0 = blockIdx.y * p.mb_per_cta;
  const int nmb = p.mb_per_cta;
  const int total = nmb * num_k;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_c[s], 1);
      mbar_init(&a_full[s], 8);
      mbar_init(&empty[s], 1);
    }
    mbar_init(h_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(mma_done, 1);
    ctl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;
  const uint64_t deadline = global_timer_ns() + (uint64_t)p.timeout_ns;

  if (warp == 0) {
    if (lane == 0) {
      const CUtensorMap* map = sh ? &tm_s_codes : &tm_codes;
      prefetch_tmap(map);
      prefetch_tmap(&tm_h);
      mbar_arrive_expect_tx(h_full, (uint32_t)(num_k * hbox));
      for (int k = 0; k < num_k; ++k) tma_load_2d(sH + k * hbox, &tm_h, k * 64, row0, h_full);
      const int erow = sh ? 0 : e * H;
      int issued = 0;
      for (int it = 0; it < total; ++it) {
        const int s = it % kStages;
        const int mb = mb0 + it / num_k, k = it % num_k;
        if (it >= kStages && !mbar_wait(&empty[s], ((it / kStages) - 1) & 1, abort_flag, deadline)) break;
        mbar_arrive_expect_tx(&full_c[s], 4096);
        tma_load_2d(sC + s * kDnC, map, k * 8, erow + mb * 128, &full_c[s]);
        issued = it + 1;
      }
      int dummy = 0;
      const uint64_t dl = global_timer_ns() + 100000000ull;
      mbar_wait(h_full, 0, &dummy, dl);  // the resident tile must land before exit
      if (*abort_flag)
        for (int it = issued - kStages < 0 ? 0 : issued - kStages; it < issued; ++it)
          mbar_wait(&full_c[it % kStages], (it / kStages) & 1, &dummy, dl);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_f32(128, N);
      bool ok = mbar_wait(h_full, 0, abort_flag, deadline);
      for (int it = 0; ok && it < total; ++it) {
        const int s = it % kStages;
        const int mbi = it / num_k, k = it % num_k;
        const int buf = mbi & 1;
        if (k == 0 && mbi >= 2 && !mbar_wait(&acc_empty[buf], ((mbi >> 1) - 1) & 1, abort_flag, deadline)) break;
        if (!mbar_wait(&a_full[s], (it / kStages) & 1, abort_flag, deadline)) break;
        tc_fence_after();
        const uint32_t a = smem_u32(sA + s * kDnA), b = smem_u32(sH + k * hbox);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f16(tmem + buf * 128, sw128_desc(a + kk * 32), sw128_desc(b + kk * 32), idesc, (k | kk) != 0);
        mma_commit(&empty[s]);
        if (k == num_k - 1) mma_commit(&acc_full[buf]);
      }
      mma_commit(mma_done);  // arrives once every issued MMA has finished
    }
  } else if (warp >= 4 && warp < 12) {
    const int dt = threadIdx.x - 128;
    const int r = dt >> 1, half = dt & 1;  // two threads per weight row
    const int gpr = I / 64;
    for (int mbi = 0; mbi < nmb; ++mbi) {
      const int mrow = (mb0 + mbi) * 128 + r;
      const size_t grow = sh ? (size_t)mrow : (size_t)e * H + mrow;
      const uint16_t* srow = (sh ? p.s_scales : p.scales) + grow * gpr;
      const uint16_t* brow = (sh ? p.s_biases : p.biases) + grow * gpr;
      for (int k = 0; k < num_k; ++k) {
        const int it = mbi * num_k + k;
        const int s = it % kStages;
        const __half2 s2 = bf16_to_h2(__ldg(srow + k));
        const __half2 b2 = bf16_to_h2(__ldg(brow + k));
        if (!mbar_wait(&full_c[s], (it / kStages) & 1, abort_flag, deadline)) { mbi = nmb; break; }
        const uint4 c = *reinterpret_cast<const uint4*>(sC + s * kDnC + r * 32 + half * 16);
        uint8_t* dst = sA + s * kDnA + r * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t o[4];
          dequant8_f16(u4_get(c, q), s2, b2, o);
          const int ch = half * 4 + q;
          *reinterpret_cast<uint4*>(dst + ((ch ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[s]);
      }
    }
  } else if (warp >= 12) {
    const int q = warp & 3;
    for (int mbi = 0; mbi < nmb; ++mbi) {
      const int buf = mbi & 1;
      if (!mbar_wait(&acc_full[buf], (mbi >> 1) & 1, abort_flag, deadline)) break;
      tc_fence_after();
      const int m = (mb0 + mbi) * 128 + q * 32 + lane;
      const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16) + buf * 128;
      for (int j0 = 0; j0 < N; j0 += 32) {
        float v[32];
        tmem_ld_32(lane_addr + j0, v);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int j = j0 + jj;
          if (j < rows) p.o[(size_t)(row0 + j) * H + m] = __float2half_rn(v[jj]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    int dummy = 0;  // no MMA may still be running when TMEM is freed
    mbar_wait(mma_done, 0, &dummy, global_timer_ns() + 100000000ull);
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicExch(p.status, (int32_t)MOE_ERR_DEVICE_TIMEOUT);
}

// ================================================================= host ===

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D tensor map of a row-major [outer][inner] array.
cudaError_t tmap_2d(CUtensorMap* m, CUtensorMapDataType dt, size_t esize, const void* base, uint64_t inner,
                    uint64_t outer, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  memset(m, 0, sizeof(*m));
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * esize};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

size_t gate_up_smem() { return kStages * kGuStage + sizeof(Ctl) + 1024; }
size_t down_smem(int I, int BM) { return (size_t)(I / 64) * BM * 128 + kStages * kDnStage + sizeof(Ctl) + 1024; }

}  // namespace

bool tc_path_supported(const Geometry& g) {
  if (g.H % 512 != 0 || g.I % 128 != 0 || g.BM > kMaxBN) return false;
  if ((size_t)(g.I / 64) * g.BM * 128 > (size_t)kMaxResidentH) return false;
  if (down_smem(g.I, g.BM) > 232448 || gate_up_smem() > 232448) return false;
  return encode_fn() != nullptr;
}

cudaError_t launch_gate_up_tc(const Geometry& g, const uint16_t* x16, const ExpertArgs& w, const TileArgs& t,
                              __half* h, int32_t* status, long long timeout_ns, cudaStream_t stream) {
  CUtensorMap tm, tms;
  cudaError_t e = tmap_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, w.codes, g.H / 8, (uint64_t)g.E * 2 * g.I, 8, 128,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  if (g.shared) {
    e = tmap_2d(&tms, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, w.s_codes, g.H / 8, (uint64_t)2 * g.I, 8, 128,
                CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
  } else {
    tms = tm;
  }
  GateUpTcParams p{g.H, g.I, g.E, g.K, g.A, x16, w.scales, w.biases, w.s_scales, w.s_biases, t, h, status,
                   timeout_ns};
  const size_t smem = gate_up_smem();
  static int configured = 0;
  e = ensure_smem(gate_up_tc_kernel, smem, &configured);
  if (e != cudaSuccess) return e;
  dim3 grid(g.max_tiles, g.I / 128);
  gate_up_tc_kernel<<<grid, kTcThreads, smem, stream>>>(tm, tms, p);
  return cudaGetLastError();
}

cudaError_t launch_down_tc(const Geometry& g, const __half* h, const ExpertArgs& w, const TileArgs& t, __half* o,
                           int32_t* status, long long timeout_ns, cudaStream_t stream) {
  CUtensorMap tm, tms, tmh;
  cudaError_t e = tmap_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, w.codes, g.I / 8, (uint64_t)g.E * g.H, 8, 128,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  if (g.shared) {
    e = tmap_2d(&tms, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, w.s_codes, g.I / 8, (uint64_t)g.H, 8, 128,
                CU_TENSOR_MAP_SWIZZLE_NONE);
    if (e != cudaSuccess) return e;
  } else {
    tms = tm;
  }
  e = tmap_2d(&tmh, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, h, g.I, (uint64_t)g.rows, 64, g.BM,
              CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  const int mb_total = g.H / 128;
  int mbc = 4;
  while (mbc > 1 && mb_total % mbc) --mbc;
  DownTcParams p{g.H, g.I, g.E, g.BM, mbc, w.scales, w.biases, w.s_scales, w.s_biases, t, o, status, timeout_ns};
  const size_t smem = down_smem(g.I, g.BM);
  static int configured = 0;
  e = ensure_smem(down_tc_kernel, smem, &configured);
  if (e != cudaSuccess) return e;
  dim3 grid(g.max_tiles, mb_total / mbc);
  down_tc_kernel<<<grid, kTcThreads, smem, stream>>>(tm, tms, tmh, p);
  return cudaGetLastError();
}

}  // namespace bgmoe
