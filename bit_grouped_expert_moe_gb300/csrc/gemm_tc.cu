// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05, TMEM
// accumulators) with 4-bit dequantisation fused into the mainloop.
// [dothoosh.com "Perplexity Lily: 1.35x faster decode for Qwen3.6 on Apple
// silicon", "Prefill optimisations", fused dequantisation: the grouped GEMM
// rebuilds the 4-bit group-64 weights tile by tile in on-chip memory and
// accumulates in FP32, so the dequantised array never goes back to memory;
// "tiling": tiles of more token rows per weight tile (16 -> 32 rows) paid.]
//
// One kernel template serves both products:
//   gate/up: item = (block-map tile, 128 h columns): A = 128 gate rows and
//            the 128 matching up rows, B = the tile's token rows of x
//            (gathered), epilogue h = silu(gate) * up (fp16, K-permuted);
//   down:    item = (tile, 256 output rows): A = 256 rows of W_down, B = the
//            tile's contiguous h rows (TMA), epilogue o (fp16).
// Either way an item is two M=128 MMAs per 16-K step that share one B tile.
//
// Orientation (swap-AB): the weights are the MMA's M and the tile's token
// rows are N (rounded up to 16), so a small expert group wastes at most 15
// token columns. Operands are fp16, K-major, 128-byte swizzled; weights are
// rounded once to fp16 (W = scale*q + bias in one fp16 FMA), and x and h carry
// the in-group K order 0,4,1,5,2,6,3,7 in which the nibbles unpack.
//
// Persistent blocks (one per SM) walk the items with a stride of the grid;
// every ring runs on across item boundaries and the TMEM accumulator is
// double buffered, so one item's epilogue overlaps the next item's MMAs.
// Rings: codes (TMA) 4 deep, dequantised A 3 deep (down: 4), B 4 deep; the
// MMAs of each stage are committed once, to a ring of 8 stage-done barriers
// that every producer of a slot waits on.
// Warp roles (576 threads):
//   warp 0      TMA producer: code tiles (and h boxes for the down GEMM)
//   warp 1      TMEM allocation and the single MMA-issuing thread
//   warps 2-5   gate/up: gather of token rows of x with cp.async
//   warps 6-13  dequantisation: codes -> fp16 weights in the swizzled layout
//   warps 14-17 epilogue: tcgen05.ld -> h or o
// Every mbarrier wait is bounded; on expiry the block raises an abort flag,
// drains its own copies and MMAs, frees its TMEM and reports
// MOE_ERR_DEVICE_TIMEOUT.
#include <cudaTypedefs.h>

#include <cstring>

#include "kernels.h"
#include "tc_ptx.cuh"

namespace bgmoe {
using namespace tc;

constexpr int kTcThreads = 576;
#ifndef BGMOE_TC_CS
#define BGMOE_TC_CS 4
#endif
#ifndef BGMOE_TC_AS
#define BGMOE_TC_AS 3
#endif
#ifndef BGMOE_TC_BS
#define BGMOE_TC_BS 4
#endif
#ifndef BGMOE_TC_AS_DOWN
#define BGMOE_TC_AS_DOWN 4
#endif
#ifndef BGMOE_TC_A_MARGIN
#define BGMOE_TC_A_MARGIN 1
#endif
// Ring depths: codes, A (gate/up and down GEMM), B. Any depths within the
// stage_done ring and the shared-memory limit are correct (the macros let a
// test build others). The defaults are the fastest measured: on gate/up at
// 4096 tokens a 5-deep B ring was 4 % slower than 4 and a 3-deep one 17 %
// slower, and a 4-deep A ring 2 % slower than 3; the down GEMM (8 stages an
// item) is 1-6 % faster with a 4-deep A ring than with 3.
constexpr int kCS = BGMOE_TC_CS, kBS = BGMOE_TC_BS;
template <bool kGateUp>
constexpr int kAStages = kGateUp ? BGMOE_TC_AS : BGMOE_TC_AS_DOWN;
constexpr int kASMax = BGMOE_TC_AS > BGMOE_TC_AS_DOWN ? BGMOE_TC_AS : BGMOE_TC_AS_DOWN;
// Generic-proxy stores into an A slot wait for the commit of the MMAs of
// kAMargin stages AFTER the slot's previous use. Measured on GB300: rewriting
// a slot as soon as the commit of the MMAs that read it had arrived corrupted
// the last-read rows of the slot in about 1 item in 200 at 128-token tiles
// (the two accumulator chains of an item finish at different times); with a
// one-stage margin no corruption was seen in any repeated run.
constexpr int kAMargin = BGMOE_TC_A_MARGIN;
static_assert(kAMargin >= 0 && kAMargin < kAStages<true> && kAMargin < kAStages<false>,
              "A-slot margin must leave the dequant a stage of lead");
// An earlier layout, in which every dequantisation warp wrote one row of
// every stage, gave wrong h rows with a 4-deep A ring and this margin (the
// dequant waiting for the MMAs three iterations back). With the two groups
// below, 3-, 4- and 5-deep rings give bit-identical results in every repeat
// (a GPU test builds them), so the depth is free.
#ifndef BGMOE_TC_B_MARGIN
#define BGMOE_TC_B_MARGIN 1
#endif
// The same rule for the gather's cp.async stores into a B slot.
constexpr int kBMargin = BGMOE_TC_B_MARGIN;
static_assert(kBMargin >= 0 && kBMargin < kBS, "B-slot margin must leave the gather a stage of lead");
// One commit per stage: the MMAs of stage s arrive on stage_done[s % kDone],
// which the dequantisation, the gather and the down kernel's B copies all
// wait on. A waiter checks every stage in order, so it has seen the phase
// kDone stages back before it tests a parity, and no waiter falls kDone
// stages behind the MMAs (they need its output first).
constexpr int kDone = 8;
static_assert(kDone >= kASMax && kDone >= kBS, "stage_done ring shorter than a data ring");
constexpr int kMaxBN = 128;               // token rows per tile (block_m <= 128)
constexpr int kTmemCols = 512;            // 2 buffers x (2 x 128 columns)
constexpr int kCBytes = 8192;             // 256 rows x 32 B of codes
constexpr int kABytes = 32768;            // 256 rows x 64 k fp16
constexpr int kBBytes = 16384;            // 128 rows x 64 k fp16
template <bool kGateUp>
constexpr int kSmemData = kCS * kCBytes + kAStages<kGateUp> * kABytes + kBS * kBBytes;

struct TcCtl {
  uint64_t c_full[kCS], c_empty[kCS];
  uint64_t a_full[kASMax];
  uint64_t b_full[kBS];
  uint64_t stage_done[kDone];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t mma_done;
  uint32_t tmem;
  int abort;
};

struct TcParams {
  int H, I, E, K, A, BM;
  int items, per_tile;        // items = num_tiles * per_tile is computed on the device
  const uint16_t* scales;     // routed [E][rows][k/64] bf16
  const uint16_t* biases;
  const uint16_t* s_scales;   // shared [rows][k/64]
  const uint16_t* s_biases;
  const uint16_t* x16;        // gate/up: [T][H] fp16, K-permuted
  TileArgs t;
  __half* out;                // gate/up: h [rows][I]; down: o [rows][H]
  int32_t* status;
  long long timeout_ns;
  int rows;                   // rows of h and o: A (+ T with a shared expert)
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + (((a + 1023u) & ~1023u) - a);
}

__device__ __forceinline__ uint32_t u4_get(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// silu(a) = a / (1 + e^-a) with the approximate divide: a few ulp of fp32
// before h is rounded to fp16 (2^-11 relative), and for a < -87 (where the
// divisor passes 2^126) it returns 0 for a value below 1e-36. The IEEE divide
// cost the epilogue warps issue slots that the dequantisation warps beside
// them on each scheduler need (gate/up 233 -> 224 us at 4096 tokens).
__device__ __forceinline__ float silu_fast(float a) { return __fdividef(a, 1.0f + __expf(-a)); }

// 16 bytes to a shared-memory address
__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

__device__ __forceinline__ uint32_t bf16_of(const uint4& v, int g) {
  const uint32_t w = u4_get(v, g >> 1);
  return (g & 1) ? (w >> 16) : (w & 0xFFFFu);
}

template <bool kGateUp>
__global__ void __launch_bounds__(kTcThreads, 1)
expert_tc_kernel(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_s_codes,
                 const __grid_constant__ CUtensorMap tm_h, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  constexpr int kAS = kAStages<kGateUp>;  // A-ring depth of this GEMM
  if (block_failed(p.t.status)) return;
  const int num_tiles = *p.t.num_tiles;
  const int items = num_tiles * p.per_tile;
  if ((int)blockIdx.x >= items) return;

  uint8_t* sm = align1024(smem_raw);
  uint8_t* sA = sm;                        // 1024-aligned stages
  uint8_t* sB = sA + kAS * kABytes;
  uint8_t* sC = sB + kBS * kBBytes;
  TcCtl* ctl = reinterpret_cast<TcCtl*>(sC + kCS * kCBytes);
  volatile int* abort_flag = &ctl->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = p.H, I = p.I;
  const int kdim = kGateUp ? H : I;        // reduction length
  const int num_k = kdim / 64;
  const int G = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kCS; ++s) {
      mbar_init(&ctl->c_full[s], 1);
      mbar_init(&ctl->c_empty[s], 4);
    }
    for (int s = 0; s < kAS; ++s) mbar_init(&ctl->a_full[s], 4);
    for (int s = 0; s < kBS; ++s) mbar_init(&ctl->b_full[s], kGateUp ? 128 : 1);
    for (int s = 0; s < kDone; ++s) mbar_init(&ctl->stage_done[s], 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl->acc_full[b], 1);
      mbar_init(&ctl->acc_empty[b], 4);
    }
    mbar_init(&ctl->mma_done, 1);
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

  // Warps 0 and 1 run their loops with all 32 lanes, so loop values stay
  // warp-uniform; every lane waits and one elected lane issues.
  auto warp_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, deadline)) != 0;
  };
  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&tm_codes);
      prefetch_tmap(&tm_s_codes);
      if (!kGateUp) prefetch_tmap(&tm_h);
    }
    int it = 0, issued_c = 0, issued_b = 0;
    bool ok = true;
    // the next item's tile is looked up a whole item ahead
    int e_nx = p.t.tile_expert[blockIdx.x / p.per_tile], row0_nx = p.t.tile_row0[blockIdx.x / p.per_tile];
    for (int w = blockIdx.x; ok && w < items; w += G) {
      const int tile = w / p.per_tile, sub = w - tile * p.per_tile;
      const int e = e_nx, row0 = row0_nx;
      if (w + G < items) {
        e_nx = p.t.tile_expert[(w + G) / p.per_tile];
        row0_nx = p.t.tile_row0[(w + G) / p.per_tile];
      }
      const bool sh = e == p.E;
      const CUtensorMap* map = sh ? &tm_s_codes : &tm_codes;
      // first weight row of each half of the item (gate/up: gate and up rows)
      int r_lo, r_hi;
      if (kGateUp) {
        r_lo = (sh ? 0 : e * 2 * I) + sub * 128;
        r_hi = r_lo + I;
      } else {
        r_lo = (sh ? 0 : e * H) + sub * 256;
        r_hi = r_lo + 128;
      }
      for (int k = 0; k < num_k; ++k, ++it) {
        const int cs = it % kCS;
        if (it >= kCS && !warp_wait(&ctl->c_empty[cs], ((it / kCS) - 1) & 1)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          mbar_arrive_expect_tx(&ctl->c_full[cs], kCBytes);
          tma_load_2d(sC + cs * kCBytes, map, k * 8, r_lo, &ctl->c_full[cs]);
          tma_load_2d(sC + cs * kCBytes + 4096, map, k * 8, r_hi, &ctl->c_full[cs]);
        }
        __syncwarp();
        issued_c = it + 1;
        if (!kGateUp) {
          const int bs = it % kBS, j = it - kBS;  // the MMAs of stage j last read this slot
          if (j >= 0 && !warp_wait(&ctl->stage_done[j % kDone], (j / kDone) & 1)) {
            ok = false;
            break;
          }
          if (elect_one()) {
            mbar_arrive_expect_tx(&ctl->b_full[bs], (uint32_t)(p.BM * 128));
            tma_load_2d(sB + bs * kBBytes, &tm_h, k * 64, row0, &ctl->b_full[bs]);
          }
          __syncwarp();
          issued_b = it + 1;
        }
      }
    }
    if (lane == 0 && *abort_flag) {  // let this block's own copies land before it exits
      int dummy = 0;
      const uint64_t dl = global_timer_ns() + 100000000ull;
      for (int i = issued_c - kCS < 0 ? 0 : issued_c - kCS; i < issued_c; ++i)
        mbar_wait(&ctl->c_full[i % kCS], (i / kCS) & 1, &dummy, dl);
      for (int i = issued_b - kBS < 0 ? 0 : issued_b - kBS; i < issued_b; ++i)
        mbar_wait(&ctl->b_full[i % kBS], (i / kBS) & 1, &dummy, dl);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer
    int it = 0, ii = 0;
    bool ok = true;
    int rows_nx = p.t.tile_rows[blockIdx.x / p.per_tile];  // looked up a whole item ahead
    for (int w = blockIdx.x; ok && w < items; w += G, ++ii) {
      const int N = (checked(rows_nx, 1, p.BM, p.status) + 15) & ~15;  // TMEM holds N <= 128 columns
      if (w + G < items) rows_nx = p.t.tile_rows[(w + G) / p.per_tile];
      const uint32_t idesc = idesc_f16_f32(128, N);
      const int buf = ii & 1;
      if (ii >= 2 && !warp_wait(&ctl->acc_empty[buf], ((ii >> 1) - 1) & 1)) break;
      const uint32_t d0 = tmem + buf * 256, d1 = d0 + 128;
      for (int k = 0; k < num_k; ++k, ++it) {
        const int as = it % kAS, bs = it % kBS;
        // Both barriers are tested at once, so a ready stage (the usual
        // case) costs one shared-memory round trip, not two: the tensor pipe
        // holds about one queued MMA, so it idles while this warp waits.
        const bool ra = mbar_test_wait(&ctl->a_full[as], (it / kAS) & 1);
        const bool rb = mbar_test_wait(&ctl->b_full[bs], (it / kBS) & 1);
        if (!__all_sync(0xffffffffu, ra && rb) &&
            (!warp_wait(&ctl->a_full[as], (it / kAS) & 1) || !warp_wait(&ctl->b_full[bs], (it / kBS) & 1))) {
          ok = false;
          break;
        }
        // the gathered rows were written by cp.async (generic proxy): after
        // the barrier made them visible to this warp, order them before the
        // MMAs' async-proxy reads
        if (kGateUp) fence_proxy_async();
        tc_fence_after();
        // descriptor start addresses count 16-byte units: 16 fp16 along K
        // is +2, the second 128-row half of the A stage (+16384 B) is +1024
        const uint64_t da = sw128_desc(smem_u32(sA + as * kABytes));
        const uint64_t db = sw128_desc(smem_u32(sB + bs * kBBytes));
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t acc = (k | kk) != 0;
            mma_f16(d0, da + 2 * kk, db + 2 * kk, idesc, acc);
            mma_f16(d1, da + 1024 + 2 * kk, db + 2 * kk, idesc, acc);
          }
          mma_commit(&ctl->stage_done[it % kDone]);
        }
        __syncwarp();
      }
      if (ok && lane == 0) mma_commit(&ctl->acc_full[buf]);
      __syncwarp();
    }
    if (lane == 0) mma_commit(&ctl->mma_done);  // arrives once every issued MMA has finished
  } else if (warp < 6) {
    // ------------------------------------------ gather of x token rows
    if (kGateUp) {
      const int gt = threadIdx.x - 64;       // 0..127
      const int j0 = gt >> 3, c = gt & 7;    // rows j0 + 16 q, 16-byte chunk c
      int it = 0;
      bool ok = true;
      for (int w = blockIdx.x; ok && w < items; w += G) {
        const int tile = w / p.per_tile;
        const int rows = checked(p.t.tile_rows[tile], 1, p.BM, p.status);
        const int row0 = checked(p.t.tile_row0[tile], 0, p.rows - rows, p.status);
        const int N = (rows + 15) & ~15;
        int tok[kMaxBN / 16];
#pragma unroll
        for (int q = 0; q < kMaxBN / 16; ++q) {
          const int j = j0 + 16 * q, r = row0 + j;
          tok[q] = j < rows ? checked(r < p.A ? p.t.sorted[r] / p.K : r - p.A, 0, p.A / p.K - 1, p.status) : 0;
        }
        for (int k = 0; k < num_k; ++k, ++it) {
          const int bs = it % kBS;
          const int j = it - kBS + kBMargin;  // the MMAs of stage j must be complete
          if (j >= 0 && !mbar_wait(&ctl->stage_done[j % kDone], (j / kDone) & 1, abort_flag, deadline)) {
            ok = false;
            break;
          }
          fence_proxy_async();  // async-proxy reads of this slot before the new copies
          uint8_t* dst = sB + bs * kBBytes;
#pragma unroll
          for (int q = 0; q < kMaxBN / 16; ++q) {
            const int j = j0 + 16 * q;
            if (j < N)
              cp_async_16(dst + j * 128 + ((c ^ (j & 7)) << 4), p.x16 + (size_t)tok[q] * H + k * 64 + c * 8,
                          j < rows ? 16u : 0u);
          }
          // the slot's barrier counts this thread's arrival once its copies land
          cp_async_mbar_arrive_noinc(&ctl->b_full[bs]);
        }
      }
      cp_async_wait_all();
    }
  } else if (warp < 14) {
    // -------------------------------------------------- dequantisation
    // Two groups of 4 warps take alternate stages (group g the stages with
    // it % 2 == g; an item has an even number of stages). Thread gt of a
    // group owns weight rows gt and gt + 128 of the item (gate/up: the gate
    // and the up row of one h column), so each hand-off of a warp covers two
    // rows while the other group works on the next stage.
    const int grp = (warp - 6) >> 2;
    const int gt = threadIdx.x - 192 - grp * 128;  // 0..127
    const int gpr = kdim / 64;                     // groups (scale, bias) and stages per weight row
    uint8_t* arow0 = sA + gt * 128;                // row gt in the first 128-row half of a stage
    const uint8_t* crow0 = sC + gt * 32;
    const bool chunked = (gpr & 7) == 0;
    auto rows_of = [&](int w, int r, const uint16_t*& srow, const uint16_t*& brow) {
      const int tile = w / p.per_tile, sub = w - tile * p.per_tile;
      const int e = checked(p.t.tile_expert[tile], 0, p.E, p.status);
      const bool sh = e == p.E;
      size_t wrow;
      if (kGateUp) wrow = (size_t)(r < 128 ? 0 : I) + sub * 128 + (r & 127) + (sh ? 0 : (size_t)e * 2 * I);
      else wrow = (size_t)sub * 256 + r + (sh ? 0 : (size_t)e * H);
      srow = (sh ? p.s_scales : p.scales) + wrow * gpr;
      brow = (sh ? p.s_biases : p.biases) + wrow * gpr;
    };
    bool ok = true;
    int it = grp;
    // One stage of this group: the codes of both rows, the wait for the
    // MMAs that last read this A slot, both rows dequantised into the slot,
    // then one lane releases the A slot and the code slot.
    // sa, ba / sb, bb: scale * 2^14 and bias of this group in rows 0 and 1
    // (group_scale_bias), in both halves.
    auto stage = [&](__half2 sa, __half2 ba, __half2 sb, __half2 bb) -> bool {
      const int cs = it % kCS, as = it % kAS;
      if (!mbar_wait(&ctl->c_full[cs], (it / kCS) & 1, abort_flag, deadline)) return false;
      // Each row's 32 bytes of codes as two 16-byte loads. The code tiles land
      // with the 32-byte TMA swizzle (16-byte chunk c of row r at chunk
      // c ^ ((r >> 2) & 1)), so the 8 rows of an access phase cover all 8
      // bank groups instead of 4.
      const int hf = (gt >> 2) & 1;
      const uint8_t* cr = crow0 + cs * kCBytes;
      const uint4 a0 = *reinterpret_cast<const uint4*>(cr + 16 * hf);
      const uint4 a1 = *reinterpret_cast<const uint4*>(cr + 16 * (hf ^ 1));
      const uint4 b0 = *reinterpret_cast<const uint4*>(cr + 4096 + 16 * hf);
      const uint4 b1 = *reinterpret_cast<const uint4*>(cr + 4096 + 16 * (hf ^ 1));
      {
        const int j = it - kAS + kAMargin;  // the MMAs of stage j must be complete
        if (j >= 0 && !mbar_wait(&ctl->stage_done[j % kDone], (j / kDone) & 1, abort_flag, deadline)) return false;
      }
      // the slot was last read by the tensor core (async proxy): order
      // those reads before these generic-proxy stores
      fence_proxy_async();
      // row gt's chunk q sits at chunk q ^ (gt & 7) of its 128-byte row (the
      // 128-byte swizzle); the row starts 128-byte aligned, so its address is
      // (row | (gt & 7) << 4) ^ q << 4: one XOR per store
      const uint32_t dsx = smem_u32(arow0 + as * kABytes) | ((uint32_t)(gt & 7) << 4);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        uint32_t o[4], u[4];
        dequant8_f16(q < 4 ? u4_get(a0, q) : u4_get(a1, q - 4), sa, ba, o);
        dequant8_f16(q < 4 ? u4_get(b0, q) : u4_get(b1, q - 4), sb, bb, u);
        sts128(dsx ^ (uint32_t)(q << 4), o[0], o[1], o[2], o[3]);
        sts128((dsx ^ (uint32_t)(q << 4)) + 16384u, u[0], u[1], u[2], u[3]);
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&ctl->a_full[as]);
        mbar_arrive(&ctl->c_empty[cs]);
      }
      it += 2;
      return true;
    };
    // One item, given its scale and bias rows and their first 8-group chunk.
    auto run_item = [&](const uint16_t* srow0, const uint16_t* brow0, const uint16_t* srow1, const uint16_t* brow1,
                        uint4 s0, uint4 c0, uint4 s1, uint4 c1) {
      if (chunked) {
        // scales/biases 8 groups per 16-byte load; this group's 4 (scale,
        // bias) pairs of each row are picked out once per chunk and the next
        // chunk is loaded while the 4 stages run
        for (int k0 = 0; ok && k0 < num_k; k0 += 8) {
          uint32_t pa[4], pb[4];
          bool fits = true;  // every scale below 4 (group_scale_bias)
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const int g = grp + 2 * m;
            fits &= group_scale_bias(bf16_bits_to_f32(bf16_of(s0, g)), bf16_bits_to_f32(bf16_of(c0, g)), pa[m]);
            fits &= group_scale_bias(bf16_bits_to_f32(bf16_of(s1, g)), bf16_bits_to_f32(bf16_of(c1, g)), pb[m]);
          }
          if (!fits) flag_range(p.status);
          if (k0 + 8 < num_k) {
            s0 = ldg_nc_v4(srow0 + k0 + 8);
            c0 = ldg_nc_v4(brow0 + k0 + 8);
            s1 = ldg_nc_v4(srow1 + k0 + 8);
            c1 = ldg_nc_v4(brow1 + k0 + 8);
          }
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const __half2 ha = *reinterpret_cast<const __half2*>(&pa[m]);
            const __half2 hb = *reinterpret_cast<const __half2*>(&pb[m]);
            if (!stage(__low2half2(ha), __high2half2(ha), __low2half2(hb), __high2half2(hb))) {
              ok = false;
              break;
            }
          }
        }
      } else {
        for (int k = grp; ok && k < num_k; k += 2) {
          uint32_t pa, pb;
          const bool fits = group_scale_bias(bf16_bits_to_f32(__ldg(srow0 + k)), bf16_bits_to_f32(__ldg(brow0 + k)), pa) &
                            group_scale_bias(bf16_bits_to_f32(__ldg(srow1 + k)), bf16_bits_to_f32(__ldg(brow1 + k)), pb);
          if (!fits) flag_range(p.status);
          const __half2 ha = *reinterpret_cast<const __half2*>(&pa), hb = *reinterpret_cast<const __half2*>(&pb);
          ok = stage(__low2half2(ha), __high2half2(ha), __low2half2(hb), __high2half2(hb));
        }
      }
    };
    const uint4 z4 = make_uint4(0, 0, 0, 0);
    if (kGateUp) {
      // 32-stage items: the rows and the first chunk are loaded at the item start
      for (int w = blockIdx.x; ok && w < items; w += G) {
        const uint16_t *srow0, *brow0, *srow1, *brow1;
        rows_of(w, gt, srow0, brow0);
        rows_of(w, gt + 128, srow1, brow1);
        if (chunked)
          run_item(srow0, brow0, srow1, brow1, ldg_nc_v4(srow0), ldg_nc_v4(brow0), ldg_nc_v4(srow1), ldg_nc_v4(brow1));
        else
          run_item(srow0, brow0, srow1, brow1, z4, z4, z4, z4);
      }
    } else {
      // 8-stage down items: the next item's rows and first chunk are looked
      // up a whole item ahead
      const uint16_t *srow0, *brow0, *srow1, *brow1;
      rows_of(blockIdx.x, gt, srow0, brow0);
      rows_of(blockIdx.x, gt + 128, srow1, brow1);
      uint4 n0 = z4, n1 = z4, n2 = z4, n3 = z4;
      if (chunked) {
        n0 = ldg_nc_v4(srow0);
        n1 = ldg_nc_v4(brow0);
        n2 = ldg_nc_v4(srow1);
        n3 = ldg_nc_v4(brow1);
      }
      for (int w = blockIdx.x; ok && w < items; w += G) {
        const uint16_t *cs0 = srow0, *cb0 = brow0, *cs1 = srow1, *cb1 = brow1;
        const uint4 s0 = n0, c0 = n1, s1 = n2, c1 = n3;
        if (w + G < items) {
          rows_of(w + G, gt, srow0, brow0);
          rows_of(w + G, gt + 128, srow1, brow1);
          if (chunked) {
            n0 = ldg_nc_v4(srow0);
            n1 = ldg_nc_v4(brow0);
            n2 = ldg_nc_v4(srow1);
            n3 = ldg_nc_v4(brow1);
          }
        }
        run_item(cs0, cb0, cs1, cb1, s0, c0, s1, c1);
      }
    }
  } else {
    // -------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quadrant of this warp
    int ii = 0;
    for (int w = blockIdx.x; w < items; w += G, ++ii) {
      const int tile = w / p.per_tile, sub = w - tile * p.per_tile;
      const int rows = checked(p.t.tile_rows[tile], 1, p.BM, p.status);
      const int row0 = checked(p.t.tile_row0[tile], 0, p.rows - rows, p.status);
      const int N = (rows + 15) & ~15;
      const int buf = ii & 1;
      if (!mbar_wait(&ctl->acc_full[buf], (ii >> 1) & 1, abort_flag, deadline)) break;
      tc_fence_after();
      const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16) + buf * 256;
      // Largest |h| or |o| this lane stores: past fp16 (>= 65520, where the
      // value rounds to inf) is MOE_ERR_RANGE; so is a warp's h tile that is
      // all under the fp16 floor and not all zero (o is checked row by row
      // where it is combined). One max per value keeps the check cheap.
      float mx = 0.f;
      if (kGateUp) {
        const int pn = perm8_pos(sub * 128 + q * 32 + lane);
        __half* hcol = p.out + (size_t)row0 * I + pn;  // this lane's column of the tile's rows
        for (int j0 = 0; j0 < N; j0 += 32, hcol += (size_t)32 * I) {
          float g[32], u[32];
          tmem_ld_32(lane_addr + j0, g);
          tmem_ld_32(lane_addr + 128 + j0, u);
          const int lim = rows - j0;  // rows of this 32-row block that exist
          if (lim >= 32) {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
              const float hf = silu_fast(g[jj]) * u[jj];
              mx = fmaxf(mx, fabsf(hf));
              hcol[jj * I] = __float2half_rn(hf);
            }
          } else {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
              if (jj < lim) {
                const float hf = silu_fast(g[jj]) * u[jj];
                mx = fmaxf(mx, fabsf(hf));
                hcol[jj * I] = __float2half_rn(hf);
              }
            }
          }
        }
      } else {
        const int m = sub * 256 + q * 32 + lane;
        __half* ocol = p.out + (size_t)row0 * H + m;  // this lane's column of the tile's rows
        for (int j0 = 0; j0 < N; j0 += 32, ocol += (size_t)32 * H) {
          float v0[32], v1[32];
          tmem_ld_32(lane_addr + j0, v0);
          tmem_ld_32(lane_addr + 128 + j0, v1);
          const int lim = rows - j0;
          if (lim >= 32) {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
              mx = fmaxf(mx, fmaxf(fabsf(v0[jj]), fabsf(v1[jj])));
              ocol[jj * H] = __float2half_rn(v0[jj]);
              ocol[jj * H + 128] = __float2half_rn(v1[jj]);
            }
          } else {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
              if (jj < lim) {
                mx = fmaxf(mx, fmaxf(fabsf(v0[jj]), fabsf(v1[jj])));
                ocol[jj * H] = __float2half_rn(v0[jj]);
                ocol[jj * H + 128] = __float2half_rn(v1[jj]);
              }
            }
          }
        }
      }
      bool inf = mx >= 65520.f;
      if (kGateUp && __any_sync(0xffffffffu, mx > 0.f) && !__any_sync(0xffffffffu, mx >= kFp16Floor))
        inf |= lane == 0;
      if (inf) flag_range(p.status);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->acc_empty[buf]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    int dummy = 0;  // no MMA may still be running when TMEM is freed
    mbar_wait(&ctl->mma_done, 0, &dummy, global_timer_ns() + 100000000ull);
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
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
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

template <bool kGateUp>
constexpr size_t kSmemBytes = kSmemData<kGateUp> + sizeof(TcCtl) + 1024;

int tc_sm_count() {
  static int sms[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (sms[dev] == 0 && cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms[dev] = 0;
  return sms[dev];
}

template <bool kGateUp>
cudaError_t launch_tc(const Geometry& g, const CUtensorMap& tm, const CUtensorMap& tms, const CUtensorMap& tmh,
                      const TcParams& p, cudaStream_t stream) {
  static SmemLimitMemo smem_memo;
  cudaError_t e = ensure_smem(expert_tc_kernel<kGateUp>, kSmemBytes<kGateUp>, &smem_memo);
  if (e != cudaSuccess) return e;
  const int sms = tc_sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  // at most one item per block beyond the upper bound of the item count
  const int max_items = g.max_tiles * p.per_tile;
  const int grid = max_items < sms ? max_items : sms;
  expert_tc_kernel<kGateUp><<<grid, kTcThreads, kSmemBytes<kGateUp>, stream>>>(tm, tms, tmh, p);
  return cudaGetLastError();
}

}  // namespace

bool tc_path_supported(const Geometry& g) {
  if (g.H % 256 != 0 || g.I % 128 != 0 || g.BM > kMaxBN) return false;
  if (kSmemBytes<true> > 232448 || kSmemBytes<false> > 232448) return false;
  return encode_fn() != nullptr;
}

cudaError_t launch_gate_up_tc(const Geometry& g, const uint16_t* x16, const ExpertArgs& w, const TileArgs& t,
                              __half* h, int32_t* status, long long timeout_ns, cudaStream_t stream) {
  CUtensorMap tm, tms;
  cudaError_t e = tmap_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, w.codes, g.H / 8, (uint64_t)g.E * 2 * g.I, 8, 128,
                          CU_TENSOR_MAP_SWIZZLE_32B);
  if (e != cudaSuccess) return e;
  if (g.shared) {
    e = tmap_2d(&tms, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, w.s_codes, g.H / 8, (uint64_t)2 * g.I, 8, 128,
                CU_TENSOR_MAP_SWIZZLE_32B);
    if (e != cudaSuccess) return e;
  } else {
    tms = tm;
  }
  TcParams p{g.H, g.I, g.E, g.K, g.A, g.BM, 0, g.I / 128, w.scales, w.biases, w.s_scales, w.s_biases, x16, t, h,
             status, timeout_ns, g.rows};
  return launch_tc<true>(g, tm, tms, tm, p, stream);
}

cudaError_t launch_down_tc(const Geometry& g, const __half* h, const ExpertArgs& w, const TileArgs& t, __half* o,
                           int32_t* status, long long timeout_ns, cudaStream_t stream) {
  CUtensorMap tm, tms, tmh;
  cudaError_t e = tmap_2d(&tm, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, w.codes, g.I / 8, (uint64_t)g.E * g.H, 8, 128,
                          CU_TENSOR_MAP_SWIZZLE_32B);
  if (e != cudaSuccess) return e;
  if (g.shared) {
    e = tmap_2d(&tms, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, w.s_codes, g.I / 8, (uint64_t)g.H, 8, 128,
                CU_TENSOR_MAP_SWIZZLE_32B);
    if (e != cudaSuccess) return e;
  } else {
    tms = tm;
  }
  e = tmap_2d(&tmh, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, h, g.I, (uint64_t)g.rows, 64, g.BM,
              CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  TcParams p{g.H, g.I, g.E, g.K, g.A, g.BM, 0, g.H / 256, w.scales, w.biases, w.s_scales, w.s_biases, nullptr, t, o,
             status, timeout_ns, g.rows};
  return launch_tc<false>(g, tm, tms, tmh, p, stream);
}

}  // namespace bgmoe
