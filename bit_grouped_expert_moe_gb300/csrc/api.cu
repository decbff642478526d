// C ABI of the MoE layer: argument checks, workspace layout and the launch
// sequence router -> routing -> expert gate/up -> expert down -> combine, all
// enqueued on the caller's stream with no host synchronisation.
#include <cstdio>
#include <cstring>
#include <cuda.h>
#include <nvtx3/nvToolsExt.h>

#include "kernels.h"

// An NVTX range around the enqueue of one step of the path (K1 router,
// K2 route, K3 gate/up, K4 down, K5 combine, or the fused decode layer), so
// that a profiler can select a step's kernels by name, e.g.
// `ncu --nvtx --nvtx-include "K3 gate/up/"`. NVTX is header-only here: with
// no tool attached a range costs two calls through a null hook.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

namespace bgmoe {

thread_local char g_detail[256] = "";

namespace {
// Driver entry points for naming the current context (looked up once).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name, int version) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(p);
}
}  // namespace

cudaError_t current_device_context(int* dev, unsigned long long* ctx) {
  static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent", 4000);
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId", 12000);
  *ctx = 0;
  const cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return e;
  CUcontext c = nullptr;
  if (get_current == nullptr || get_current(&c) != CUDA_SUCCESS || c == nullptr) return cudaSuccess;
  unsigned long long id = 0;
  // A context's identifier is unique for the life of the process; without
  // it the handle stands in (a handle can be reused after a reset).
  *ctx = (get_id != nullptr && get_id(c, &id) == CUDA_SUCCESS) ? id + 1 : reinterpret_cast<uintptr_t>(c);
  return cudaSuccess;
}

moe_status cuda_fail(cudaError_t e, const char* where) {
  snprintf(g_detail, sizeof(g_detail), "%s: %s", where, cudaGetErrorString(e));
  return MOE_ERR_CUDA;
}

namespace {

constexpr long long kDefaultTimeoutNs = 1000000000ll;  // 1 s per device-side wait
constexpr int kMaxRouteBlocks = 128;
constexpr int kMinTokensPerRouteBlock = 16;
constexpr int kMaxTokens = 1 << 18;
constexpr int kTensorCoreMinTokens = 64;

moe_status check_shape(const moe_shape* s) {
  if (!s) return MOE_ERR_INVALID_ARG;
  if (s->T < 0 || s->H <= 0 || s->I <= 0 || s->E <= 0 || s->top_k <= 0 || s->I_shared < 0)
    return MOE_ERR_INVALID_ARG;
  if (s->T > kMaxTokens) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (s->group_size != kGroup) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (s->H % 64 || s->H < 64 || s->H > 8192) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (s->I % 64 || s->I < 64 || s->I > 4096) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (s->I_shared != 0 && s->I_shared != s->I) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (s->top_k > kMaxTopK || s->top_k > s->E || s->E > kMaxExperts) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (s->block_m != 16 && s->block_m != 32 && s->block_m != 64 && s->block_m != 128)
    return MOE_ERR_UNSUPPORTED_SHAPE;
  return MOE_OK;
}

Geometry geometry(const moe_shape& s) {
  Geometry g{};
  g.T = s.T;
  g.H = s.H;
  g.I = s.I;
  g.E = s.E;
  g.K = s.top_k;
  g.BM = s.block_m;
  g.shared = s.I_shared > 0 ? 1 : 0;
  g.A = s.T * s.top_k;
  g.rows = g.A + (g.shared ? s.T : 0);
  const int ce = (g.A + g.BM - 1) / g.BM;
  g.max_tiles = ce + (g.A < g.E ? g.A : g.E) + (g.shared ? (g.T + g.BM - 1) / g.BM : 0);
  int P = (g.T + kMinTokensPerRouteBlock - 1) / kMinTokensPerRouteBlock;
  if (P > kMaxRouteBlocks) P = kMaxRouteBlocks;
  if (P < 1) P = 1;
  g.route_blocks = P;
  g.tokens_per_block = (g.T + P - 1) / P;
  return g;
}

// Workspace regions, each 256-byte aligned, in this order.
struct Workspace {
  int32_t* status;
  float* logits;              // [T][E+1]
  unsigned long long* state;  // [P][E]
  int32_t* ids;               // routing tables kept here when the caller passes none
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
  uint16_t* x16;              // [T][H] fp16 activations for the tensor-core path
  __half* dh;                 // [kDecodeMaxSlots][T][I] h of the fused decode kernel (T <= 4 only)
  __half* h;                  // [rows][I]
  __half* o;                  // [rows][H]
  size_t bytes;
};

Workspace carve(const Geometry& g, void* base) {
  Workspace w{};
  size_t off = 0;
  char* b = static_cast<char*>(base);
  auto take = [&](size_t n) -> void* {
    void* p = b ? b + off : nullptr;
    off += (n + 255) & ~size_t(255);
    return p;
  };
  w.status = static_cast<int32_t*>(take(sizeof(int32_t)));
  w.logits = static_cast<float*>(take(sizeof(float) * (size_t)g.T * (g.E + 1)));
  w.state = static_cast<unsigned long long*>(take(sizeof(unsigned long long) * (size_t)g.route_blocks * g.E));
  w.ids = static_cast<int32_t*>(take(sizeof(int32_t) * (size_t)g.A));
  w.weights = static_cast<float*>(take(sizeof(float) * (size_t)g.A));
  w.gate = static_cast<float*>(take(sizeof(float) * (size_t)g.T));
  w.counts = static_cast<int32_t*>(take(sizeof(int32_t) * (size_t)(g.E + 1)));
  w.offsets = static_cast<int32_t*>(take(sizeof(int32_t) * (size_t)(g.E + 2)));
  w.sorted = static_cast<int32_t*>(take(sizeof(int32_t) * (size_t)g.A));
  w.inv = static_cast<int32_t*>(take(sizeof(int32_t) * (size_t)g.A));
  w.tile_expert = static_cast<int32_t*>(take(sizeof(int32_t) * (size_t)g.max_tiles));
  w.tile_row0 = static_cast<int32_t*>(take(sizeof(int32_t) * (size_t)g.max_tiles));
  w.tile_rows = static_cast<int32_t*>(take(sizeof(int32_t) * (size_t)g.max_tiles));
  w.num_tiles = static_cast<int32_t*>(take(sizeof(int32_t)));
  w.x16 = static_cast<uint16_t*>(take(sizeof(uint16_t) * (size_t)g.T * g.H));
  w.dh = static_cast<__half*>(take(g.T <= kDecodeMaxTokens ? sizeof(__half) * (size_t)kDecodeMaxSlots * g.T * g.I : 0));
  w.h = static_cast<__half*>(take(sizeof(__half) * (size_t)g.rows * g.I));
  w.o = static_cast<__half*>(take(sizeof(__half) * (size_t)g.rows * g.H));
  w.bytes = off;
  return w;
}

bool route_out_ok(const moe_route_out* o, bool shared) {
  return o && o->ids && o->weights && o->counts && o->offsets && o->sorted && o->inv && o->tile_expert &&
         o->tile_row0 && o->tile_rows && o->num_tiles && o->status && (!shared || o->gate);
}

moe_route_out ws_route_out(const Workspace& w) {
  moe_route_out r{};
  r.ids = w.ids;
  r.weights = w.weights;
  r.gate = w.gate;
  r.counts = w.counts;
  r.offsets = w.offsets;
  r.sorted = w.sorted;
  r.inv = w.inv;
  r.tile_expert = w.tile_expert;
  r.tile_row0 = w.tile_row0;
  r.tile_rows = w.tile_rows;
  r.num_tiles = w.num_tiles;
  r.status = w.status;
  return r;
}

// Router scores: tensor cores for calls with many tokens, the CUDA-core GEMV
// (one warp per expert row) for decode-sized calls.
cudaError_t launch_router(const Geometry& g, const void* x, const void* w_router, const void* wsg,
                          const Workspace& w, int32_t* status, uint16_t* x16, cudaStream_t stream) {
  if (g.T >= kTensorCoreMinTokens && router_tc_supported(g))
    return launch_router_tc(g, x, w_router, wsg, w.logits, w.state, g.route_blocks * g.E, status, x16,
                            kDefaultTimeoutNs, stream);
  return launch_router_logits(g, x, w_router, wsg, w.logits, w.state, g.route_blocks * g.E, status, x16, stream);
}

moe_status enqueue_routing_only(const Geometry& g, const float* router_bias, const moe_route_out& r,
                                const Workspace& w, int stalled_block, long long timeout_ns, cudaStream_t stream) {
  RouteArgs a{};
  a.logits = w.logits;
  a.bias = router_bias;
  a.T = g.T;
  a.E = g.E;
  a.K = g.K;
  a.BM = g.BM;
  a.shared = g.shared;
  a.P = g.route_blocks;
  a.tpb = g.tokens_per_block;
  a.ids = r.ids;
  a.weights = r.weights;
  a.gate = r.gate;
  a.counts = r.counts;
  a.offsets = r.offsets;
  a.sorted = r.sorted;
  a.inv = r.inv;
  a.tile_expert = r.tile_expert;
  a.tile_row0 = r.tile_row0;
  a.tile_rows = r.tile_rows;
  a.num_tiles = r.num_tiles;
  a.status = r.status;
  a.state = w.state;
  a.stalled_block = stalled_block;
  a.timeout_ns = timeout_ns;
  cudaError_t e;
  {
    NvtxRange nr("K2 route");
    e = launch_route(a, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e, "routing kernel launch");
  return MOE_OK;
}

moe_status enqueue_route(const Geometry& g, const void* x, const void* w_router, const float* router_bias,
                         const void* w_shared_gate, const moe_route_out& r, const Workspace& w,
                         int stalled_block, long long timeout_ns, cudaStream_t stream) {
  // The call's status word starts at zero in stream order, before any kernel
  // of the call can record a failure in it.
  cudaError_t e = cudaMemsetAsync(r.status, 0, sizeof(int32_t), stream);
  if (e != cudaSuccess) return cuda_fail(e, "status clear");
  {
    NvtxRange nr("K1 router");
    e = launch_router(g, x, w_router, g.shared ? w_shared_gate : nullptr, w, r.status, nullptr, stream);
  }
  if (e != cudaSuccess) return cuda_fail(e, "router kernel launch");
  return enqueue_routing_only(g, router_bias, r, w, stalled_block, timeout_ns, stream);
}

moe_status route_common(const moe_shape* shape, const void* x, const void* w_router, const float* router_bias,
                        const void* w_shared_gate, const moe_route_out* out, void* workspace, size_t ws_bytes,
                        int stalled_block, long long timeout_ns, void* stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  const Geometry g = geometry(*shape);
  if (!route_out_ok(out, g.shared)) return MOE_ERR_INVALID_ARG;
  if (g.T == 0) return MOE_OK;
  if (!x || !w_router || (g.shared && !w_shared_gate) || !workspace) return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return MOE_ERR_INVALID_ARG;
  const Workspace w = carve(g, workspace);
  if (ws_bytes < w.bytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return enqueue_route(g, x, w_router, router_bias, w_shared_gate, *out, w, stalled_block, timeout_ns,
                       static_cast<cudaStream_t>(stream));
}

}  // namespace
}  // namespace bgmoe

using namespace bgmoe;

extern "C" {

int32_t moe_abi_version(void) { return MOE_ABI_VERSION; }

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_RANGE: return "a value left the fp16 operand range";
    case MOE_ERR_BOUNDS: return "a device table index was out of range (bounds-checking build)";
  }
  return "unknown status";
}

const char* moe_last_error_detail(void) { return g_detail; }

moe_status moe_workspace_bytes(const moe_shape* shape, size_t* bytes) {
  if (!bytes) return MOE_ERR_INVALID_ARG;
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  *bytes = carve(geometry(*shape), nullptr).bytes;
  return MOE_OK;
}

moe_status moe_max_tiles(const moe_shape* shape, int32_t* max_tiles) {
  if (!max_tiles) return MOE_ERR_INVALID_ARG;
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  *max_tiles = geometry(*shape).max_tiles;
  return MOE_OK;
}

moe_status moe_route_blocks(const moe_shape* shape, int32_t* blocks) {
  if (!blocks) return MOE_ERR_INVALID_ARG;
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  *blocks = geometry(*shape).route_blocks;
  return MOE_OK;
}

moe_status moe_route(const moe_shape* shape, const void* x, const void* w_router, const float* router_bias,
                     const void* w_shared_gate, const moe_route_out* out, void* workspace, size_t ws_bytes,
                     void* stream) {
  return route_common(shape, x, w_router, router_bias, w_shared_gate, out, workspace, ws_bytes, -1,
                      kDefaultTimeoutNs, stream);
}

moe_status moe_test_route_stall(const moe_shape* shape, const void* x, const void* w_router,
                                const float* router_bias, const void* w_shared_gate, const moe_route_out* out,
                                void* workspace, size_t ws_bytes, int32_t stalled_block, int64_t timeout_ns,
                                void* stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  const Geometry g = geometry(*shape);
  if (stalled_block < 0 || stalled_block >= g.route_blocks || timeout_ns <= 0 || timeout_ns > kDefaultTimeoutNs)
    return MOE_ERR_INVALID_ARG;
  return route_common(shape, x, w_router, router_bias, w_shared_gate, out, workspace, ws_bytes, stalled_block,
                      timeout_ns, stream);
}

namespace {
// moe_forward_timed, plus the test-only fused-decode stall: with
// stall_block >= 0 that block of the fused decode kernel never publishes its
// h and every wait of the call gives up after timeout_ns.
moe_status forward_impl(const moe_shape* shape, const void* x, const void* w_router, const float* router_bias,
                        const moe_experts* experts, const moe_experts* shared, const void* w_shared_gate, float* y,
                        const moe_route_out* route_out, void* workspace, size_t ws_bytes, void* const* events,
                        int32_t expert_path, void* stream, int32_t stall_block, int64_t timeout_ns,
                        void* x_next = nullptr, const void* norm_w = nullptr, float norm_eps = 0.f) {
  moe_status st = check_shape(shape);
  if (expert_path < MOE_PATH_AUTO || expert_path > MOE_PATH_FUSED_DECODE) return MOE_ERR_INVALID_ARG;
  if (st != MOE_OK) return st;
  const Geometry g = geometry(*shape);
  if (route_out && !route_out_ok(route_out, g.shared)) return MOE_ERR_INVALID_ARG;
  if (g.T == 0) return MOE_OK;
  if (!x || !w_router || !y || !experts || !workspace) return MOE_ERR_INVALID_ARG;
  if (!experts->gate_up.codes || !experts->gate_up.scales || !experts->gate_up.biases || !experts->down.codes ||
      !experts->down.scales || !experts->down.biases)
    return MOE_ERR_INVALID_ARG;
  if (g.shared && (!shared || !w_shared_gate || !shared->gate_up.codes || !shared->gate_up.scales ||
                   !shared->gate_up.biases || !shared->down.codes || !shared->down.scales || !shared->down.biases))
    return MOE_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return MOE_ERR_INVALID_ARG;
  const Workspace w = carve(g, workspace);
  if (ws_bytes < w.bytes) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const moe_route_out r = route_out ? *route_out : ws_route_out(w);
  // Inside a stream capture a plain event record only orders streams; the
  // external flag makes it a timed event node of the graph.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (events && cudaStreamIsCapturing(s, &cap) != cudaSuccess) return cuda_fail(cudaGetLastError(), "capture query");
  auto mark = [&](int i) -> cudaError_t {
    if (!events) return cudaSuccess;
    cudaEvent_t ev = static_cast<cudaEvent_t>(events[i]);
    return cap == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal)
                                                : cudaEventRecord(ev, s);
  };
  cudaError_t e = mark(0);
  if (e != cudaSuccess) return cuda_fail(e, "event record");

  // Expert path: the fused decode kernel for decode-sized calls, tensor
  // cores once the tile rows are many enough to feed them, else the GEMV.
  // The fused decode kernel copies weight tiles with bulk async copies and
  // the tensor-core kernels read codes, scales and biases 16 bytes at a
  // time: both need 16-byte aligned weight arrays.
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  auto mat16 = [&](const moe_qmat& q) { return a16(q.codes) && a16(q.scales) && a16(q.biases); };
  const bool aligned = mat16(experts->gate_up) && mat16(experts->down) &&
                       (!g.shared || (mat16(shared->gate_up) && mat16(shared->down)));
  const bool dec_ok = decode_supported(g) && aligned;
  if (expert_path == MOE_PATH_FUSED_DECODE && !dec_ok) return MOE_ERR_UNSUPPORTED_SHAPE;
  const bool fused = expert_path == MOE_PATH_FUSED_DECODE || (expert_path == MOE_PATH_AUTO && dec_ok);
  // The pre-norm residual join is part of the fused decode kernel only.
  if (x_next != nullptr && !fused) {
    snprintf(g_detail, sizeof(g_detail), "the residual entry point runs on the fused decode path only");
    return MOE_ERR_UNSUPPORTED_SHAPE;
  }
  const bool tc_ok = tc_path_supported(g) && aligned;
  if (expert_path == MOE_PATH_TENSOR_CORE && !tc_ok) return MOE_ERR_UNSUPPORTED_SHAPE;
  const bool tc = expert_path == MOE_PATH_TENSOR_CORE ||
                  (expert_path == MOE_PATH_AUTO && !fused && g.T >= kTensorCoreMinTokens && tc_ok);

  if (fused) {
    // The fused kernel computes the router logits itself; events[1] and [2]
    // fall right after events[0].
    if ((e = mark(1)) != cudaSuccess || (e = mark(2)) != cudaSuccess) return cuda_fail(e, "event record");
    DecodeArgs d{};
    d.wr = static_cast<const uint16_t*>(w_router);
    d.wsg = g.shared ? static_cast<const uint16_t*>(w_shared_gate) : nullptr;
    d.T = g.T;
    d.H = g.H;
    d.I = g.I;
    d.E = g.E;
    d.K = g.K;
    d.shared = g.shared;
    d.x = static_cast<const uint16_t*>(x);
    d.norm = x_next != nullptr ? 1 : 0;
    d.norm_w = static_cast<const uint16_t*>(norm_w);
    d.norm_eps = norm_eps;
    d.logits = w.logits;
    d.bias = router_bias;
    d.gu = ExpertArgs{experts->gate_up.codes, experts->gate_up.scales, experts->gate_up.biases,
                      g.shared ? shared->gate_up.codes : nullptr, g.shared ? shared->gate_up.scales : nullptr,
                      g.shared ? shared->gate_up.biases : nullptr};
    d.dn = ExpertArgs{experts->down.codes, experts->down.scales, experts->down.biases,
                      g.shared ? shared->down.codes : nullptr, g.shared ? shared->down.scales : nullptr,
                      g.shared ? shared->down.biases : nullptr};
    d.ids = r.ids;
    d.weights = r.weights;
    d.gate = r.gate;
    d.counts = r.counts;
    d.offsets = r.offsets;
    d.sorted = r.sorted;
    d.inv = r.inv;
    d.tile_expert = r.tile_expert;
    d.tile_row0 = r.tile_row0;
    d.tile_rows = r.tile_rows;
    d.num_tiles = r.num_tiles;
    d.status = r.status;
    d.h = w.dh;
    d.y = y;
    d.x_next = static_cast<uint16_t*>(x_next);
    d.timeout_ns = timeout_ns;
    d.stall_block = stall_block;
    {
      NvtxRange nr("K1-K5 fused decode");
      e = launch_decode(d, g, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "fused decode launch");
    for (int i = 3; i < 6; ++i)
      if ((e = mark(i)) != cudaSuccess) return cuda_fail(e, "event record");
    return MOE_OK;
  }

  // Router logits, then the routing pipeline (two launches). The status word
  // is cleared in stream order first, so no kernel of the call can have
  // recorded a failure before it is cleared.
  e = cudaMemsetAsync(r.status, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) return cuda_fail(e, "status clear");
  {
    NvtxRange nr("K1 router");
    e = launch_router(g, x, w_router, g.shared ? w_shared_gate : nullptr, w, r.status, tc ? w.x16 : nullptr, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "router kernel launch");
  if ((e = mark(1)) != cudaSuccess) return cuda_fail(e, "event record");
  st = enqueue_routing_only(g, router_bias, r, w, -1, kDefaultTimeoutNs, s);
  if (st != MOE_OK) return st;
  if ((e = mark(2)) != cudaSuccess) return cuda_fail(e, "event record");

  TileArgs t{r.tile_expert, r.tile_row0, r.tile_rows, r.num_tiles, r.sorted, r.status};
  ExpertArgs gu{experts->gate_up.codes, experts->gate_up.scales, experts->gate_up.biases,
                g.shared ? shared->gate_up.codes : nullptr, g.shared ? shared->gate_up.scales : nullptr,
                g.shared ? shared->gate_up.biases : nullptr};
  ExpertArgs dn{experts->down.codes, experts->down.scales, experts->down.biases,
                g.shared ? shared->down.codes : nullptr, g.shared ? shared->down.scales : nullptr,
                g.shared ? shared->down.biases : nullptr};
  {
    NvtxRange nr("K3 gate/up");
    e = tc ? launch_gate_up_tc(g, w.x16, gu, t, w.h, r.status, kDefaultTimeoutNs, s)
           : launch_gemv_gate_up(g, static_cast<const uint16_t*>(x), gu, t, w.h, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "expert gate/up launch");
  if ((e = mark(3)) != cudaSuccess) return cuda_fail(e, "event record");
  {
    NvtxRange nr("K4 down");
    e = tc ? launch_down_tc(g, w.h, dn, t, w.o, r.status, kDefaultTimeoutNs, s)
           : launch_gemv_down(g, w.h, dn, t, w.o, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "expert down launch");
  if ((e = mark(4)) != cudaSuccess) return cuda_fail(e, "event record");
  {
    NvtxRange nr("K5 combine");
    e = launch_combine(g, w.o, r.inv, r.weights, r.gate, r.status, y, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  if ((e = mark(5)) != cudaSuccess) return cuda_fail(e, "event record");
  return MOE_OK;
}

}  // namespace

moe_status moe_forward_timed(const moe_shape* shape, const void* x, const void* w_router,
                             const float* router_bias, const moe_experts* experts, const moe_experts* shared,
                             const void* w_shared_gate, float* y, const moe_route_out* route_out, void* workspace,
                             size_t ws_bytes, void* const* events, int32_t expert_path, void* stream) {
  return forward_impl(shape, x, w_router, router_bias, experts, shared, w_shared_gate, y, route_out, workspace,
                      ws_bytes, events, expert_path, stream, -1, kDefaultTimeoutNs);
}

moe_status moe_test_decode_stall(const moe_shape* shape, const void* x, const void* w_router,
                                 const float* router_bias, const moe_experts* experts, const moe_experts* shared,
                                 const void* w_shared_gate, float* y, const moe_route_out* route_out,
                                 void* workspace, size_t ws_bytes, int32_t stalled_block, int64_t timeout_ns,
                                 void* stream) {
  if (stalled_block < 0 || timeout_ns <= 0 || timeout_ns > kDefaultTimeoutNs) return MOE_ERR_INVALID_ARG;
  return forward_impl(shape, x, w_router, router_bias, experts, shared, w_shared_gate, y, route_out, workspace,
                      ws_bytes, nullptr, MOE_PATH_FUSED_DECODE, stream, stalled_block, timeout_ns);
}

moe_status moe_forward_residual(const moe_shape* shape, const void* r, const void* norm_weight, float norm_eps,
                                const void* w_router, const float* router_bias, const moe_experts* experts,
                                const moe_experts* shared, const void* w_shared_gate, float* y, void* r_next,
                                const moe_route_out* route_out, void* workspace, size_t ws_bytes, void* stream) {
  if (!r || !r_next || r_next == r || !(norm_eps > 0.f)) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(r) & 15) || (reinterpret_cast<uintptr_t>(r_next) & 15) ||
      (reinterpret_cast<uintptr_t>(norm_weight) & 15))
    return MOE_ERR_INVALID_ARG;
  return forward_impl(shape, r, w_router, router_bias, experts, shared, w_shared_gate, y, route_out, workspace,
                      ws_bytes, nullptr, MOE_PATH_AUTO, stream, -1, kDefaultTimeoutNs, r_next, norm_weight, norm_eps);
}

moe_status moe_forward(const moe_shape* shape, const void* x, const void* w_router, const float* router_bias,
                       const moe_experts* experts, const moe_experts* shared, const void* w_shared_gate, float* y,
                       const moe_route_out* route_out, void* workspace, size_t ws_bytes, void* stream) {
  return moe_forward_timed(shape, x, w_router, router_bias, experts, shared, w_shared_gate, y, route_out,
                           workspace, ws_bytes, nullptr, MOE_PATH_AUTO, stream);
}

moe_status moe_status_read(const int32_t* device_status, void* stream, int32_t* host_status) {
  if (!device_status || !host_status) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(host_status, device_status, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (e != cudaSuccess) return cuda_fail(e, "status copy");
  e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "status sync");
  return MOE_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Routing for callers that cannot allocate device memory.
//
// moe_route needs a workspace from its caller. Some callers have none to give
// at the point where they route: code running inside a host callback or a
// real-time loop that must not enter the CUDA allocator (cudaMalloc can
// synchronise the device and take unbounded time), plugins that are handed
// only the buffers of their inputs and outputs, and embedders whose device
// memory is owned and budgeted by a host framework. moe_route_noalloc keeps
// its scratch (router logits and the routing kernel's look-back words) in
// the file-scope device array below, which every GPU that loads this library
// holds until the process exits. The router kernel clears the look-back
// words at the start of every call; the logits are overwritten.
static __device__ __align__(256) unsigned char g_noalloc_scratch[1u << 20];

namespace bgmoe {
namespace {

constexpr size_t kNoAllocScratchBytes = sizeof(g_noalloc_scratch);
PointerMemo g_noalloc_memo;

// Device address of the scratch array on the current device, looked up once
// per device and context with that device current (the host-side name of a
// __device__ array is a stand-in, not its address; a new context, as after
// cudaDeviceReset, reloads the module and may move the array, so its address
// is looked up again there).
cudaError_t noalloc_scratch(void** out) {
  int dev = 0;
  unsigned long long ctx = 0;
  cudaError_t e = current_device_context(&dev, &ctx);
  if (e != cudaSuccess) return e;
  return static_cast<cudaError_t>(g_noalloc_memo.get(dev, ctx, out, [](void** p) {
    return static_cast<int>(cudaGetSymbolAddress(p, g_noalloc_scratch));
  }));
}

size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

}  // namespace
}  // namespace bgmoe

extern "C" moe_status moe_route_noalloc(const moe_shape* shape, const void* x, const void* w_router,
                                        const float* router_bias, const void* w_shared_gate,
                                        const moe_route_out* out, void* stream) {
  moe_status st = check_shape(shape);
  if (st != MOE_OK) return st;
  const Geometry g = geometry(*shape);
  if (!route_out_ok(out, g.shared)) return MOE_ERR_INVALID_ARG;
  if (g.T == 0) return MOE_OK;
  if (!x || !w_router || (g.shared && !w_shared_gate)) return MOE_ERR_INVALID_ARG;
  const size_t logits_bytes = align256(sizeof(float) * (size_t)g.T * (g.E + 1));
  const size_t need = logits_bytes + align256(sizeof(unsigned long long) * (size_t)g.route_blocks * g.E);
  if (need > kNoAllocScratchBytes) {
    snprintf(g_detail, sizeof(g_detail),
             "moe_route_noalloc: this shape needs %zu bytes of scratch, the static buffer holds %zu", need,
             kNoAllocScratchBytes);
    return MOE_ERR_UNSUPPORTED_SHAPE;
  }
  void* base = nullptr;
  cudaError_t e = noalloc_scratch(&base);
  if (e != cudaSuccess) return cuda_fail(e, "moe_route_noalloc scratch address");
  Workspace w{};
  w.logits = static_cast<float*>(base);
  w.state = reinterpret_cast<unsigned long long*>(static_cast<char*>(base) + logits_bytes);
  return enqueue_route(g, x, w_router, router_bias, w_shared_gate, *out, w, -1, kDefaultTimeoutNs,
                       static_cast<cudaStream_t>(stream));
}
