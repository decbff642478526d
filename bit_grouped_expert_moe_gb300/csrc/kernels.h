// Host-side launchers of the layer's kernels (one per .cu file).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace bgmoe {

// Records "where: CUDA error text" for moe_last_error_detail() and returns
// MOE_ERR_CUDA (every entry point of the library reports launch failures so).
moe_status cuda_fail(cudaError_t e, const char* where);


constexpr int kDecodeMaxTokens = 4;  // tokens per call handled by the fused decode kernel
constexpr int kDecodeMaxStages = 8;  // shared-memory ring depth of the fused decode kernel

struct RouteArgs {
  const float* logits;  // [T][E+1], column E = shared gate logit
  const float* bias;    // [E] or null
  int T, E, K, BM, shared, P, tpb;
  int32_t* ids;
  float* weights;
  float* gate;
  int32_t* counts;
  int32_t* offsets;
  int32_t* sorted;
  int32_t* inv;
  int32_t* tile_expert;
  int32_t* tile_row0;
  int32_t* tile_rows;
  int32_t* num_tiles;
  int32_t* status;
  unsigned long long* state;  // [P][E] look-back words, zeroed by the router kernel
  int stalled_block;          // test hook: this block never publishes (-1: none)
  long long timeout_ns;       // limit of every device-side wait
};

struct ExpertArgs {
  const uint32_t* codes;   // routed experts
  const uint16_t* scales;
  const uint16_t* biases;
  const uint32_t* s_codes; // shared expert (or null)
  const uint16_t* s_scales;
  const uint16_t* s_biases;
};

struct TileArgs {
  const int32_t* tile_expert;
  const int32_t* tile_row0;
  const int32_t* tile_rows;
  const int32_t* num_tiles;
  const int32_t* sorted;
  const int32_t* status;
};

cudaError_t launch_router_logits(const Geometry& g, const void* x, const void* wr, const void* wsg,
                                 float* logits, unsigned long long* state, int n_state,
                                 int32_t* status, uint16_t* x16, cudaStream_t stream,
                                 unsigned int* bar = nullptr);

// Router on the tensor cores (router_tc.cu), for calls with many tokens.
bool router_tc_supported(const Geometry& g);
cudaError_t launch_router_tc(const Geometry& g, const void* x, const void* wr, const void* wsg, float* logits,
                             unsigned long long* state, int n_state, int32_t* status, uint16_t* x16,
                             long long timeout_ns, cudaStream_t stream);

size_t route_smem_bytes(const Geometry& g);
cudaError_t launch_route(const RouteArgs& a, cudaStream_t stream);

cudaError_t launch_gemv_gate_up(const Geometry& g, const uint16_t* x, const ExpertArgs& w,
                                const TileArgs& t, __half* h, cudaStream_t stream);
cudaError_t launch_gemv_down(const Geometry& g, const __half* h, const ExpertArgs& w,
                             const TileArgs& t, __half* o, cudaStream_t stream);

// Tensor-core grouped GEMMs (gemm_tc.cu).
bool tc_path_supported(const Geometry& g);
cudaError_t launch_gate_up_tc(const Geometry& g, const uint16_t* x16, const ExpertArgs& w, const TileArgs& t,
                              __half* h, int32_t* status, long long timeout_ns, cudaStream_t stream);
cudaError_t launch_down_tc(const Geometry& g, const __half* h, const ExpertArgs& w, const TileArgs& t, __half* o,
                           int32_t* status, long long timeout_ns, cudaStream_t stream);

// Fused decode layer (decode.cu): router, top-k, tables, gate/up, down and
// combine in one kernel after a one-block prelude, for T <= kDecodeMaxTokens.
constexpr int kDecodeMaxSlots = kDecodeMaxTokens * kMaxTopK + 1;  // distinct routed experts + the shared one
struct DecodeArgs {
  int T, H, I, E, K, shared;
  const uint16_t* x;     // bf16 [T][H]: the layer input, or (norm) the residual stream r
  int norm;              // 1: the layer input is RMSNorm(r) (fp32, not rounded), r = x
  const uint16_t* norm_w;  // bf16 [H] RMSNorm gain, or null (gain 1)
  float norm_eps;
  const uint16_t* wr;    // bf16 [E][H] router weights
  const uint16_t* wsg;   // bf16 [H] shared-expert gate row, or null
  float* logits;         // [T][E+1], filled with a sentinel by the prelude, then written by the router rows
  const float* bias;     // [E] or null
  __half* h;             // fp16 [kDecodeMaxSlots][T][I] h of every slot (K order permuted within groups of 8),
                         // filled with a sentinel by the prelude, then written once per call
  ExpertArgs gu, dn;
  int32_t* ids;
  float* weights;
  float* gate;
  int32_t* counts;
  int32_t* offsets;
  int32_t* sorted;
  int32_t* inv;
  int32_t* tile_expert;
  int32_t* tile_row0;
  int32_t* tile_rows;
  int32_t* num_tiles;
  int32_t* status;
  float* y;              // fp32 [T][H]
  uint16_t* x_next;      // bf16 [T][H] = bf16(r + y) (the next layer's residual stream), or null
  long long timeout_ns;
  int stall_block;       // test only: this block never publishes its h (-1: none)
  // shared-memory layout, filled in by launch_decode
  long long sdn_offset, x16_offset, xf_offset, part_offset, hst_bytes;
};
bool decode_supported(const Geometry& g);
// Launches the prelude (sentinel logits and h, cleared status word) and then
// the decode kernel with programmatic dependent launch.
cudaError_t launch_decode(const DecodeArgs& args, const Geometry& g, cudaStream_t stream);

cudaError_t launch_combine(const Geometry& g, const __half* o, const int32_t* inv, const float* weights,
                           const float* gate, const int32_t* status, float* y, cudaStream_t stream);

}  // namespace bgmoe
