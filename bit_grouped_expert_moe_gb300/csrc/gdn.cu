// Gated DeltaNet recurrence with the state held in registers (sm_103a).
//
// [dothoosh.com "Perplexity Lily: 1.35x faster decode for Qwen3.6 on Apple
// silicon": "Model specification" (30 Gated DeltaNet layers, a fixed-size
// recurrence) and "Prefill optimisations" (a register-resident scan); the
// gated delta rule of Yang, Kautz and Hatamizadeh, "Gated Delta Networks".]
//
// The rows of the [Dv][Dk] state evolve independently: row j needs only its
// own dot products with k^ and q^ and its own value v_j. So one block takes 16
// rows of one (sequence, value head) and its 128 threads hold them in
// registers, 8 threads per row and 16 columns each, for the whole sequence:
//   u   = S_j . k^          partial dot + 3-step shuffle over the row's 8 threads
//   v'  = beta (v_j - alpha u)
//   S_j = alpha S_j + v' k^
//   o_j = S_j . q^          partial dot + shuffle
// The token inputs of the block (q and k of its key head, its 16 values of v,
// gate and beta) arrive 32 tokens at a time by cp.async into a double buffer.
// A pass over each chunk then writes what every row needs, once per block
// instead of once per row: k^ and q^ (normalised, fp32), alpha = exp(gate),
// beta and v, so the per-token chain is loads, two dot products and the update.
// Thread t of a row holds the 16-byte column pieces t, t+8, t+16, t+24, so the
// 8 threads of a row read 8 consecutive pieces (no bank conflicts; the rows
// of the staged and prepared arrays are padded so that the prepare pass,
// which spans two tokens per access phase, has none either).
#include <cuda_bf16.h>

#include "common.cuh"
#include "gdn.h"
#include "kernels.h"

namespace bgmoe {
namespace gdn {

constexpr int kD = 128;          // Dk = Dv
constexpr int kRows = 16;        // state rows per block
constexpr int kTPR = 8;          // threads per row
constexpr int kCols = kD / kTPR; // columns per thread
constexpr int kThreads = kRows * kTPR;
constexpr float kEps = 1e-6f;
constexpr int kChunk = 32;       // tokens staged per shared-memory buffer

// Row paddings of the shared-memory arrays. The prepare pass has 4 threads
// per token, so each 8-thread phase of a 16-byte access covers two tokens:
// with unpadded rows (256 B of bf16, 512 B of fp32, both multiples of the
// 128-byte bank cycle) the two tokens hit the same banks. A bf16 row of 320 B
// moves the next token by 4 bank groups of 16 B (the 8 accesses of a phase
// then cover all 8 groups, and a cp.async target stays 16-byte aligned); an
// fp32 row of 132 floats moves it by one group, which interleaves the two
// tokens' groups the same way; 17 floats per value row spread the scalar v
// stores.
constexpr int kPadH = 32;  // bf16 elements
constexpr int kPadF = 4;   // fp32 elements

struct Stage {  // raw inputs of one chunk (cp.async target)
  uint16_t k[kChunk][kD + kPadH];
  uint16_t q[kChunk][kD + kPadH];
  uint16_t v[kChunk][kRows];
  float gate[kChunk];
  float beta[kChunk];
};

struct Prepared {  // what the token loop reads
  float k[kChunk][kD + kPadF];  // k^
  float q[kChunk][kD + kPadF];  // q^ (with 1/sqrt(Dk))
  float v[kChunk][kRows + 1];
  float alpha[kChunk];
  float beta[kChunk];
};

struct Smem {
  Stage st[2];
  Prepared pr;
};

struct Params {
  const uint16_t* q;
  const uint16_t* k;
  const uint16_t* v;
  const float* gate;
  const float* beta;
  const int32_t* offsets;
  const float* state_in;
  float* state_out;
  float* o;
  int32_t* status;
  int B, T, Hqk, Hv;
};

__device__ __forceinline__ float row_sum(float x) {
#pragma unroll
  for (int o = 1; o < kTPR; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Two fp32 lanes packed in 64 bits (lane 0 in the low half, as a float2 in
// memory). The packed operations round each lane exactly as the scalar ones
// (fma.rn / mul.rn per lane), so a pair of scalar chains run as one packed
// chain gives the same bits with half the instructions.
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ float2 unpack2(uint64_t v) {
  float2 f;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(v));
  return f;
}

__device__ __forceinline__ void cp_async(void* dst, const void* src, int bytes16) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(dst));
  if (bytes16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src) : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(d), "l"(src) : "memory");
}

__global__ void __launch_bounds__(kThreads) gdn_scan_kernel(const Params p) {
  const int blocks_per_head = kD / kRows;
  const int rb = blockIdx.x % blocks_per_head;
  const int h = (blockIdx.x / blocks_per_head) % p.Hv;
  const int b = blockIdx.x / (blocks_per_head * p.Hv);
  const int g = h / (p.Hv / p.Hqk);
  const int ri = threadIdx.x / kTPR;  // the block's row this thread holds
  const int row = rb * kRows + ri;
  const int tc = threadIdx.x % kTPR;   // column pieces tc, tc+8, tc+16, tc+24 (4 columns each)

  const size_t srow = (((size_t)b * p.Hv + h) * kD + row) * kD;
  // this thread's 16 state columns as 8 packed pairs: S2[2j], S2[2j + 1] hold
  // columns 32j + 4tc + {0, 1} and {2, 3}
  uint64_t S2[kCols / 2];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const ulonglong2 s4 = __ldcs(reinterpret_cast<const ulonglong2*>(p.state_in + srow + 32 * j + 4 * tc));
    S2[2 * j] = s4.x;
    S2[2 * j + 1] = s4.y;
  }
  int t0 = __ldg(p.offsets + b), t1 = __ldg(p.offsets + b + 1);
  if (t0 < 0 || t1 > p.T || t0 > t1) {
    if (threadIdx.x == 0 && rb == 0 && h == 0 && p.status) atomicExch(p.status, (int32_t)MOE_ERR_INVALID_ARG);
    t1 = t0;  // skipped: the state passes through unchanged
  }
  const float qscale = rsqrtf((float)kD);
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);

  // Stage tokens c .. c+n-1 (n <= kChunk) into buffer `buf`; every thread
  // issues its copies and commits one group (possibly empty).
  auto stage = [&](int c, int buf) {
    const int n = min(kChunk, t1 - c);
    const int tid = threadIdx.x;
    Stage& st = sm.st[buf];
#pragma unroll
    for (int j = tid; j < kChunk * (kD / 8); j += kThreads) {  // q and k: 16-byte pieces
      const int r = j / (kD / 8), piece = j % (kD / 8);
      if (r < n) {
        const size_t off = ((size_t)(c + r) * p.Hqk + g) * kD + piece * 8;
        cp_async(&st.k[r][piece * 8], p.k + off, 1);
        cp_async(&st.q[r][piece * 8], p.q + off, 1);
      }
    }
    if (tid < 2 * kChunk) {  // v: the block's 16 values (32 bytes) per token
      const int r = tid >> 1, half = tid & 1;
      if (r < n) cp_async(&st.v[r][half * 8], p.v + ((size_t)(c + r) * p.Hv + h) * kD + rb * kRows + half * 8, 1);
    } else if (tid < 3 * kChunk) {
      const int r = tid - 2 * kChunk;
      if (r < n) cp_async(&st.gate[r], p.gate + (size_t)(c + r) * p.Hv + h, 0);
    } else {
      const int r = tid - 3 * kChunk;
      if (r < n) cp_async(&st.beta[r], p.beta + (size_t)(c + r) * p.Hv + h, 0);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };

  int buf = 0;
  if (t0 < t1) stage(t0, 0);
  for (int c = t0; c < t1; c += kChunk, buf ^= 1) {
    if (c + kChunk < t1) {
      stage(c + kChunk, buf ^ 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();  // chunk c has landed; the previous chunk's token loop is over
    const int n = min(kChunk, t1 - c);
    {
      // prepare: 4 threads per token, thread qt taking columns qt*8 + 32m ..
      // +7 (m = 0..3). Every lane runs the same shuffles; rows past the chunk
      // compute on whatever the buffer holds and store nothing.
      const Stage& st = sm.st[buf];
      const int r = threadIdx.x >> 2, qt = threadIdx.x & 3;
      const bool live = r < n;
      float kv[32], qv[32];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint4 kw = *reinterpret_cast<const uint4*>(&st.k[r][qt * 8 + 32 * m]);
        const uint4 qw = *reinterpret_cast<const uint4*>(&st.q[r][qt * 8 + 32 * m]);
        const uint32_t ka[4] = {kw.x, kw.y, kw.z, kw.w}, qa[4] = {qw.x, qw.y, qw.z, qw.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          kv[8 * m + 2 * i] = __uint_as_float(ka[i] << 16);
          kv[8 * m + 2 * i + 1] = __uint_as_float(ka[i] & 0xFFFF0000u);
          qv[8 * m + 2 * i] = __uint_as_float(qa[i] << 16);
          qv[8 * m + 2 * i + 1] = __uint_as_float(qa[i] & 0xFFFF0000u);
        }
      }
      float kk = 0.f, qq = 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        kk = fmaf(kv[i], kv[i], kk);
        qq = fmaf(qv[i], qv[i], qq);
      }
      kk += __shfl_xor_sync(0xffffffffu, kk, 1);
      qq += __shfl_xor_sync(0xffffffffu, qq, 1);
      kk += __shfl_xor_sync(0xffffffffu, kk, 2);
      qq += __shfl_xor_sync(0xffffffffu, qq, 2);
      const float rk = rsqrtf(kk + kEps), rq = rsqrtf(qq + kEps) * qscale;
      if (live) {
#pragma unroll
        for (int m = 0; m < 4; ++m)
#pragma unroll
          for (int i = 0; i < 8; i += 4) {
            *reinterpret_cast<float4*>(&sm.pr.k[r][qt * 8 + 32 * m + i]) =
                make_float4(kv[8 * m + i] * rk, kv[8 * m + i + 1] * rk, kv[8 * m + i + 2] * rk,
                            kv[8 * m + i + 3] * rk);
            *reinterpret_cast<float4*>(&sm.pr.q[r][qt * 8 + 32 * m + i]) =
                make_float4(qv[8 * m + i] * rq, qv[8 * m + i + 1] * rq, qv[8 * m + i + 2] * rq,
                            qv[8 * m + i + 3] * rq);
          }
#pragma unroll
        for (int i = 0; i < 4; ++i)
          sm.pr.v[r][qt * 4 + i] = __uint_as_float((uint32_t)st.v[r][qt * 4 + i] << 16);
        if (qt == 0) {
          sm.pr.alpha[r] = expf(st.gate[r]);
          sm.pr.beta[r] = st.beta[r];
        }
      }
    }
    __syncthreads();  // prepared values are visible
    const Prepared& x = sm.pr;
    for (int r8 = 0; r8 < n; r8 += 8) {
      // the state chain runs token by token; each token's partial output dot
      // waits in po[] and 8 tokens are reduced together at the end
      float po[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int r = r8 + jj;
        if (r >= n) {
          po[jj] = 0.f;
          continue;
        }
        // k^ and q^ as packed pairs, in the layout of S2
        uint64_t kv2[kCols / 2], qv2[kCols / 2];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const ulonglong2 k4 = *reinterpret_cast<const ulonglong2*>(&x.k[r][32 * j + 4 * tc]);
          const ulonglong2 q4 = *reinterpret_cast<const ulonglong2*>(&x.q[r][32 * j + 4 * tc]);
          kv2[2 * j] = k4.x;
          kv2[2 * j + 1] = k4.y;
          qv2[2 * j] = q4.x;
          qv2[2 * j + 1] = q4.y;
        }
        const float alpha = x.alpha[r];
        // u = S_j . k^ (before the decay; the decayed product is alpha u), in
        // four chains over columns 4i + c: chains 0 and 1 as one packed
        // chain, 2 and 3 as another
        uint64_t u01 = 0ull, u23 = 0ull;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          u01 = fma2(S2[2 * j], kv2[2 * j], u01);
          u23 = fma2(S2[2 * j + 1], kv2[2 * j + 1], u23);
        }
        const float2 ua = unpack2(u01), ub = unpack2(u23);
        const float u = row_sum((ua.x + ua.y) + (ub.x + ub.y));
        const float w = x.beta[r] * (x.v[r][ri] - alpha * u);
        // S = alpha S + w k^ per column, then the output dot with q^ in the
        // same four chains
        const uint64_t alpha2 = pack2(alpha, alpha), w2 = pack2(w, w);
        uint64_t o01 = 0ull, o23 = 0ull;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          S2[2 * j] = fma2(alpha2, S2[2 * j], mul2(w2, kv2[2 * j]));
          S2[2 * j + 1] = fma2(alpha2, S2[2 * j + 1], mul2(w2, kv2[2 * j + 1]));
          o01 = fma2(S2[2 * j], qv2[2 * j], o01);
          o23 = fma2(S2[2 * j + 1], qv2[2 * j + 1], o23);
        }
        const float2 oa = unpack2(o01), ob = unpack2(o23);
        po[jj] = (oa.x + oa.y) + (ob.x + ob.y);
      }
      // reduce-scatter over the row's 8 threads: thread tc ends with token r8 + tc
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const bool hi = tc & 4;
        const float send = hi ? po[i] : po[i + 4];
        const float keep = hi ? po[i + 4] : po[i];
        po[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
      }
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const bool hi = tc & 2;
        const float send = hi ? po[i] : po[i + 2];
        const float keep = hi ? po[i + 2] : po[i];
        po[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
      }
      {
        const bool hi = tc & 1;
        const float send = hi ? po[0] : po[1];
        const float keep = hi ? po[1] : po[0];
        po[0] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
      }
      if (r8 + tc < n) p.o[((size_t)(c + r8 + tc) * p.Hv + h) * kD + row] = po[0];
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j)
    __stcs(reinterpret_cast<ulonglong2*>(p.state_out + srow + 32 * j + 4 * tc), make_ulonglong2(S2[2 * j], S2[2 * j + 1]));
}

// Sequences of a token or two (decode): no staging, each thread reads its
// inputs straight from global memory (the next token's while the current one
// is computed), so the block needs no shared memory and many blocks fit on an
// SM to keep the state reads and writes in flight.
__global__ void __launch_bounds__(kThreads) gdn_short_kernel(const Params p) {
  const int blocks_per_head = kD / kRows;
  const int rb = blockIdx.x % blocks_per_head;
  const int h = (blockIdx.x / blocks_per_head) % p.Hv;
  const int b = blockIdx.x / (blocks_per_head * p.Hv);
  const int g = h / (p.Hv / p.Hqk);
  const int row = rb * kRows + threadIdx.x / kTPR;
  const int tc = threadIdx.x % kTPR;
  const size_t srow = (((size_t)b * p.Hv + h) * kD + row) * kD;
  float S[kCols];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float4 s4 = __ldcs(reinterpret_cast<const float4*>(p.state_in + srow + 32 * j + 4 * tc));
    S[4 * j] = s4.x;
    S[4 * j + 1] = s4.y;
    S[4 * j + 2] = s4.z;
    S[4 * j + 3] = s4.w;
  }
  int t0 = __ldg(p.offsets + b), t1 = __ldg(p.offsets + b + 1);
  if (t0 < 0 || t1 > p.T || t0 > t1) {
    if (threadIdx.x == 0 && rb == 0 && h == 0 && p.status) atomicExch(p.status, (int32_t)MOE_ERR_INVALID_ARG);
    t1 = t0;
  }
  const float qscale = rsqrtf((float)kD);
  for (int t = t0; t < t1; ++t) {
    float kv[kCols], qv[kCols];
#pragma unroll
    for (int j = 0; j < 4; ++j) {   // columns 32j + 4tc .. +3: two bf16 pairs each
      const uint2 kw = __ldg(reinterpret_cast<const uint2*>(p.k + ((size_t)t * p.Hqk + g) * kD + 32 * j + 4 * tc));
      const uint2 qw = __ldg(reinterpret_cast<const uint2*>(p.q + ((size_t)t * p.Hqk + g) * kD + 32 * j + 4 * tc));
      kv[4 * j] = __uint_as_float(kw.x << 16);
      kv[4 * j + 1] = __uint_as_float(kw.x & 0xFFFF0000u);
      kv[4 * j + 2] = __uint_as_float(kw.y << 16);
      kv[4 * j + 3] = __uint_as_float(kw.y & 0xFFFF0000u);
      qv[4 * j] = __uint_as_float(qw.x << 16);
      qv[4 * j + 1] = __uint_as_float(qw.x & 0xFFFF0000u);
      qv[4 * j + 2] = __uint_as_float(qw.y << 16);
      qv[4 * j + 3] = __uint_as_float(qw.y & 0xFFFF0000u);
    }
    const float vj = __uint_as_float((uint32_t)__ldg(p.v + ((size_t)t * p.Hv + h) * kD + row) << 16);
    const float alpha = expf(__ldg(p.gate + (size_t)t * p.Hv + h));
    const float beta = __ldg(p.beta + (size_t)t * p.Hv + h);
    float kk = 0.f, qq = 0.f;
#pragma unroll
    for (int i = 0; i < kCols; ++i) {
      kk = fmaf(kv[i], kv[i], kk);
      qq = fmaf(qv[i], qv[i], qq);
    }
    const float rk = rsqrtf(row_sum(kk) + kEps);
    const float rq = rsqrtf(row_sum(qq) + kEps) * qscale;
    float u0 = 0.f, u1 = 0.f, u2 = 0.f, u3 = 0.f;
#pragma unroll
    for (int i = 0; i < kCols; i += 4) {
      u0 = fmaf(S[i], kv[i], u0);
      u1 = fmaf(S[i + 1], kv[i + 1], u1);
      u2 = fmaf(S[i + 2], kv[i + 2], u2);
      u3 = fmaf(S[i + 3], kv[i + 3], u3);
    }
    const float u = row_sum((u0 + u1) + (u2 + u3)) * rk;
    const float w = beta * (vj - alpha * u) * rk;
    float o0 = 0.f, o1 = 0.f, o2 = 0.f, o3 = 0.f;
#pragma unroll
    for (int i = 0; i < kCols; i += 4) {
      S[i] = fmaf(alpha, S[i], w * kv[i]);
      S[i + 1] = fmaf(alpha, S[i + 1], w * kv[i + 1]);
      S[i + 2] = fmaf(alpha, S[i + 2], w * kv[i + 2]);
      S[i + 3] = fmaf(alpha, S[i + 3], w * kv[i + 3]);
      o0 = fmaf(S[i], qv[i], o0);
      o1 = fmaf(S[i + 1], qv[i + 1], o1);
      o2 = fmaf(S[i + 2], qv[i + 2], o2);
      o3 = fmaf(S[i + 3], qv[i + 3], o3);
    }
    const float ot = row_sum((o0 + o1) + (o2 + o3)) * rq;
    if (tc == 0) p.o[((size_t)t * p.Hv + h) * kD + row] = ot;
  }
#pragma unroll
  for (int j = 0; j < 4; ++j)
    __stcs(reinterpret_cast<float4*>(p.state_out + srow + 32 * j + 4 * tc),
           make_float4(S[4 * j], S[4 * j + 1], S[4 * j + 2], S[4 * j + 3]));
}

bool shape_ok(const moe_gdn_shape& s) {
  if (s.B < 1 || s.B > 65535 || s.T < 0 || s.T > (1 << 24)) return false;
  if (s.Hqk < 1 || s.Hv < s.Hqk || s.Hv % s.Hqk != 0 || s.Hv > 4096) return false;
  return s.Dk == kD && s.Dv == kD;
}

cudaError_t record(void* ev, cudaStream_t s) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cap);
  if (e != cudaSuccess) return e;
  return cap == cudaStreamCaptureStatusActive
             ? cudaEventRecordWithFlags(static_cast<cudaEvent_t>(ev), s, cudaEventRecordExternal)
             : cudaEventRecord(static_cast<cudaEvent_t>(ev), s);
}

moe_status scan(const moe_gdn_shape* shape, const void* q, const void* k, const void* v, const float* gate,
                const float* beta, const int32_t* offsets, const float* state_in, float* state_out, float* o,
                int32_t* status, void* const* events, void* stream_) {
  if (!shape) return MOE_ERR_INVALID_ARG;
  const moe_gdn_shape s = *shape;
  if (!shape_ok(s)) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (!offsets || !state_in || !state_out) return MOE_ERR_INVALID_ARG;
  if (s.T > 0 && (!q || !k || !v || !gate || !beta || !o)) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(state_in) |
       reinterpret_cast<uintptr_t>(state_out)) & 15)
    return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(v) & 15) |
      ((reinterpret_cast<uintptr_t>(gate) | reinterpret_cast<uintptr_t>(beta) | reinterpret_cast<uintptr_t>(o) |
        reinterpret_cast<uintptr_t>(offsets) | reinterpret_cast<uintptr_t>(status)) & 3))
    return MOE_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  cudaError_t e;
  if (events && (e = record(events[0], stream)) != cudaSuccess) return cuda_fail(e, "event record");
  Params prm{static_cast<const uint16_t*>(q), static_cast<const uint16_t*>(k), static_cast<const uint16_t*>(v),
             gate, beta, offsets, state_in, state_out, o, status, s.B, s.T, s.Hqk, s.Hv};
  const unsigned grid = (unsigned)s.B * (unsigned)s.Hv * (kD / kRows);
  if (s.T <= 2 * s.B) {  // a token or two per sequence on average: decode
    gdn_short_kernel<<<grid, kThreads, 0, stream>>>(prm);
  } else {
    static SmemLimitMemo smem_memo;
    if ((e = ensure_smem(gdn_scan_kernel, sizeof(Smem), &smem_memo)) != cudaSuccess)
      return cuda_fail(e, "shared-memory limit");
    gdn_scan_kernel<<<grid, kThreads, sizeof(Smem), stream>>>(prm);
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "scan kernel launch");
  if (events && (e = record(events[1], stream)) != cudaSuccess) return cuda_fail(e, "event record");
  return MOE_OK;
}

}  // namespace gdn
}  // namespace bgmoe

extern "C" {

moe_status moe_gdn_scan(const moe_gdn_shape* shape, const void* q, const void* k, const void* v, const float* gate,
                        const float* beta, const int32_t* offsets, const float* state_in, float* state_out,
                        float* o, int32_t* status, void* stream) {
  return bgmoe::gdn::scan(shape, q, k, v, gate, beta, offsets, state_in, state_out, o, status, nullptr, stream);
}

moe_status moe_gdn_scan_timed(const moe_gdn_shape* shape, const void* q, const void* k, const void* v,
                              const float* gate, const float* beta, const int32_t* offsets, const float* state_in,
                              float* state_out, float* o, int32_t* status, void* const* events, void* stream) {
  if (!events || !events[0] || !events[1]) return MOE_ERR_INVALID_ARG;
  return bgmoe::gdn::scan(shape, q, k, v, gate, beta, offsets, state_in, state_out, o, status, events, stream);
}

}  // extern "C"
