// Router scores on the tensor cores, for calls with many tokens:
// l[t, e] = x[t, :] . W_r[e, :] (bf16 x bf16, fp32 accumulation in TMEM).
// [dothoosh.com "Perplexity Lily: 1.35x faster decode for Qwen3.6 on Apple
// silicon", "Model specification": the router scores 256 experts per token.]
//
// Swap-AB again: 128 experts are the MMA's M, kRtTok tokens its N; TMA loads
// both operands (128-byte swizzle) through a kRtStages-deep ring. Each block
// covers kRtTok tokens x 128 experts. In the blocks of the first expert block,
// two otherwise idle warps also compute the shared-gate logit x . w_sg of
// their tokens and write x as fp16, K-permuted within groups of 8
// (0,4,1,5,2,6,3,7) for the tensor-core expert GEMM. Every block also clears
// its share of the routing kernel's look-back words.
#include <cudaTypedefs.h>

#include <cstring>

#include "kernels.h"
#include "tc_ptx.cuh"

namespace bgmoe {
using namespace tc;

constexpr int kRtThreads = 256;
constexpr int kRtWarps = kRtThreads / 32;
constexpr int kMaxH = 2048;                 // largest H this kernel serves (larger: the CUDA-core router)
constexpr int kRtStages = 4;
constexpr int kRtTok = 64;                  // tokens per block (MMA N)
constexpr int kRtA = 128 * 128;             // 128 experts x 64 k bf16
constexpr int kRtB = kRtTok * 128;          // kRtTok tokens x 64 k bf16
constexpr int kRtStage = kRtA + kRtB;

struct RtCtl {
  uint64_t full[kRtStages];
  uint64_t empty[kRtStages];
  uint64_t acc_full;
  uint32_t tmem;
  int abort;
};

struct RouterTcParams {
  int T, H, E;
  const uint16_t* x;      // bf16 [T][H]
  const uint16_t* wsg;    // bf16 [H] or null
  float* logits;          // [T][E+1]
  uint16_t* x16;          // fp16 [T][H] K-permuted, or null
  unsigned long long* state;
  int n_state;
  int32_t* status;
  long long timeout_ns;
};

__device__ __forceinline__ uint8_t* rt_align1024(uint8_t* p) {
  const uint32_t a = smem_u32(p);
  return p + (((a + 1023u) & ~1023u) - a);
}

__global__ void __launch_bounds__(kRtThreads, 1)
router_tc_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                 const RouterTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = rt_align1024(smem_raw);
  RtCtl* ctl = reinterpret_cast<RtCtl*>(sm + kRtStages * kRtStage);
  volatile int* abort_flag = &ctl->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kRtTok, eb = blockIdx.y;
  const int num_k = p.H / 64;

  {  // clear the look-back words of this call (the status word was cleared
     // in stream order before this kernel)
    const int nblocks = gridDim.x * gridDim.y;
    const int b = blockIdx.y * gridDim.x + blockIdx.x;
    for (int i = b * blockDim.x + threadIdx.x; i < p.n_state; i += nblocks * blockDim.x) p.state[i] = 0ull;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRtStages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    mbar_init(&ctl->acc_full, 1);
    ctl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem, 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem;
  const uint64_t deadline = global_timer_ns() + (uint64_t)p.timeout_ns;

  // Warps 0 and 1 run their loops with all 32 lanes (values stay
  // warp-uniform): every lane waits, one elected lane issues.
  auto warp_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, deadline)) != 0;
  };
  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tm_w);
      prefetch_tmap(&tm_x);
    }
    int issued = 0;
    for (int it = 0; it < num_k; ++it) {
      const int s = it % kRtStages;
      if (it >= kRtStages && !warp_wait(&ctl->empty[s], ((it / kRtStages) - 1) & 1)) break;
      uint8_t* st = sm + s * kRtStage;
      if (elect_one()) {
        mbar_arrive_expect_tx(&ctl->full[s], kRtStage);
        tma_load_2d(st, &tm_w, it * 64, eb * 128, &ctl->full[s]);
        tma_load_2d(st + kRtA, &tm_x, it * 64, t0, &ctl->full[s]);
      }
      __syncwarp();
      issued = it + 1;
    }
    if (lane == 0 && *abort_flag) {
      int dummy = 0;
      const uint64_t dl = global_timer_ns() + 100000000ull;
      for (int it = issued - kRtStages < 0 ? 0 : issued - kRtStages; it < issued; ++it)
        mbar_wait(&ctl->full[it % kRtStages], (it / kRtStages) & 1, &dummy, dl);
    }
  } else if (warp == 1) {
    // kind::f16 with bf16 A and B (format 1), fp32 accumulator
    const uint32_t idesc = idesc_f16_f32(128, kRtTok) | (1u << 7) | (1u << 10);
    for (int it = 0; it < num_k; ++it) {
      const int s = it % kRtStages;
      if (!warp_wait(&ctl->full[s], (it / kRtStages) & 1)) break;
      tc_fence_after();
      const uint64_t da = sw128_desc(smem_u32(sm + s * kRtStage));
      const uint64_t db = sw128_desc(smem_u32(sm + s * kRtStage + kRtA));
      if (elect_one()) {
        // descriptor start addresses count 16-byte units: 16 bf16 along K is +2
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) mma_f16(tmem, da + 2 * kk, db + 2 * kk, idesc, (it | kk) != 0);
        mma_commit(&ctl->empty[s]);
      }
      __syncwarp();
    }
    if (lane == 0) mma_commit(&ctl->acc_full);
  }
  if (warp >= 2) {
    // Shared-gate logit and fp16 copy of x for this block's tokens, on warps
    // 2-7 (the epilogue warps have nothing to do until the accumulator is
    // ready): w_sg stays in registers, and all of a token's x loads go out
    // before any is used.
    if (eb == 0 && (p.wsg != nullptr || p.x16 != nullptr)) {
      const int per_lane = p.H / 256;  // 16-byte chunks per lane (H % 512 == 0 on this path)
      constexpr int kMaxPer = kMaxH / 256;
      uint4 wv[kMaxPer];
#pragma unroll
      for (int i = 0; i < kMaxPer; ++i)
        if (i < per_lane && p.wsg != nullptr) wv[i] = ldg_nc_v4(p.wsg + (lane + 32 * i) * 8);
      // one token's shared-gate logit and fp16 copy from its x row xv
      auto token = [&](int t, const uint4 (&xv)[kMaxPer]) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < kMaxPer; ++i) {
          if (i >= per_lane) break;
          const int k0 = (lane + 32 * i) * 8;
          const uint32_t xw[4] = {xv[i].x, xv[i].y, xv[i].z, xv[i].w};
          float xf[8];
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            xf[2 * m] = bf16_bits_to_f32(xw[m] & 0xFFFFu);
            xf[2 * m + 1] = bf16_bits_to_f32(xw[m] >> 16);
          }
          if (p.wsg != nullptr) {
            const uint32_t ww[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              acc = fmaf(xf[2 * m], bf16_bits_to_f32(ww[m] & 0xFFFFu), acc);
              acc = fmaf(xf[2 * m + 1], bf16_bits_to_f32(ww[m] >> 16), acc);
            }
          }
          if (p.x16 != nullptr) {
            bool big = false;
#pragma unroll
            for (int m = 0; m < 8; ++m) big |= fp16_overflows(xf[m]);
            if (big) flag_range(p.status);
            // K order 0,4,1,5,2,6,3,7 inside the group of 8
            const __half2 h0 = __floats2half2_rn(xf[0], xf[4]), h1 = __floats2half2_rn(xf[1], xf[5]);
            const __half2 h2 = __floats2half2_rn(xf[2], xf[6]), h3 = __floats2half2_rn(xf[3], xf[7]);
            uint4 o;
            o.x = *reinterpret_cast<const uint32_t*>(&h0);
            o.y = *reinterpret_cast<const uint32_t*>(&h1);
            o.z = *reinterpret_cast<const uint32_t*>(&h2);
            o.w = *reinterpret_cast<const uint32_t*>(&h3);
            *reinterpret_cast<uint4*>(p.x16 + (size_t)t * p.H + k0) = o;
          }
        }
        if (p.wsg != nullptr) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
          if (lane == 0) p.logits[(size_t)t * (p.E + 1) + p.E] = acc;
        }
      };
      // two tokens per pass: both rows' loads go out before either is used
      constexpr int kStride = kRtWarps - 2;
      for (int tl = warp - 2; tl < kRtTok; tl += 2 * kStride) {
        const int ta = t0 + tl, tb = ta + kStride;
        if (ta >= p.T) break;
        const bool has_b = tl + kStride < kRtTok && tb < p.T;
        uint4 xa[kMaxPer], xb[kMaxPer];
#pragma unroll
        for (int i = 0; i < kMaxPer; ++i)
          if (i < per_lane) xa[i] = ldg_nc_v4(p.x + (size_t)ta * p.H + (lane + 32 * i) * 8);
        if (has_b)
#pragma unroll
          for (int i = 0; i < kMaxPer; ++i)
            if (i < per_lane) xb[i] = ldg_nc_v4(p.x + (size_t)tb * p.H + (lane + 32 * i) * 8);
        token(ta, xa);
        if (has_b) token(tb, xb);
      }
    }
  }
  if (warp >= 4) {
    // epilogue: lane = expert, column = token
    const int q = warp & 3;
    if (mbar_wait(&ctl->acc_full, 0, abort_flag, deadline)) {
      tc_fence_after();
      const int e = eb * 128 + q * 32 + lane;
      float v[32];
      for (int j0 = 0; j0 < kRtTok; j0 += 32) {
        tmem_ld_32(tmem + ((uint32_t)(q * 32) << 16) + j0, v);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int t = t0 + j0 + jj;
          if (t < p.T && e < p.E) p.logits[(size_t)t * (p.E + 1) + e] = v[jj];
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    int dummy = 0;
    mbar_wait(&ctl->acc_full, 0, &dummy, global_timer_ns() + 100000000ull);
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
  if (threadIdx.x == 0 && *abort_flag) atomicExch(p.status, (int32_t)MOE_ERR_DEVICE_TIMEOUT);
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 rt_encode_fn() {
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

cudaError_t bf16_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_outer) {
  auto fn = rt_encode_fn();
  if (!fn) return cudaErrorNotSupported;
  memset(m, 0, sizeof(*m));
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {64, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}
}  // namespace

bool router_tc_supported(const Geometry& g) { return g.H % 512 == 0 && g.H <= kMaxH && rt_encode_fn() != nullptr; }

cudaError_t launch_router_tc(const Geometry& g, const void* x, const void* wr, const void* wsg, float* logits,
                             unsigned long long* state, int n_state, int32_t* status, uint16_t* x16,
                             long long timeout_ns, cudaStream_t stream) {
  CUtensorMap tw, tx;
  cudaError_t e = bf16_map(&tw, wr, g.H, g.E, 128);
  if (e != cudaSuccess) return e;
  e = bf16_map(&tx, x, g.H, g.T, kRtTok);
  if (e != cudaSuccess) return e;
  RouterTcParams p{g.T, g.H, g.E, static_cast<const uint16_t*>(x), static_cast<const uint16_t*>(wsg), logits, x16,
                   state, n_state, status, timeout_ns};
  const size_t smem = kRtStages * kRtStage + sizeof(RtCtl) + 1024;
  static SmemLimitMemo smem_memo;
  e = ensure_smem(router_tc_kernel, smem, &smem_memo);
  if (e != cudaSuccess) return e;
  dim3 grid((g.T + kRtTok - 1) / kRtTok, (g.E + 127) / 128);
  router_tc_kernel<<<grid, kRtThreads, smem, stream>>>(tw, tx, p);
  return cudaGetLastError();
}

}  // namespace bgmoe
