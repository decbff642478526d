/*
 * bit_grouped_expert_moe_gb300 — C ABI of one Mixture-of-Experts layer with
 * 4-bit group-64 affine expert weights, for NVIDIA GB300 (sm_103a).
 *
 * The layer (Qwen3.6-35B-A3B shape, as described on the pages about
 * Perplexity's Lily engine):
 *   1. router:  l[t,e] = x[t,:] . W_r[e,:] (+ b[e]); the top_k experts by l
 *               (ties: lower index first); weights w[t,k] = softmax over the
 *               selected logits (= softmax over all E renormalised over the
 *               top_k); shared gate g[t] = sigmoid(x[t,:] . w_sg).
 *               [dothoosh.com "Perplexity Lily: 1.35x faster decode for
 *               Qwen3.6 on Apple silicon", section "Model specification":
 *               the router scores 256 experts and picks 8, plus one shared
 *               expert that processes every token.]
 *   2. routing: histogram, prefix scan, scatter and block map, all on the GPU
 *               with no host synchronisation. [same page, "Prefill
 *               optimisations", GPU-resident routing item.]
 *   3. experts: SwiGLU experts h = silu(x W_gate^T) * (x W_up^T),
 *               o = h W_down^T, whose weights are 4-bit codes with one bf16
 *               scale and one bf16 bias per 64 weights, dequantised inside the
 *               grouped GEMM with FP32 accumulation. [same page, "Prefill
 *               optimisations", fused-dequantisation item.]
 *   4. combine: y[t] = sum_k w[t,k] o[t,k] + g[t] o_shared[t].
 *
 * Data formats (shared by every entry point):
 *   bf16 values are passed as their 16-bit patterns (uint16_t / void*).
 *   A packed matrix W[N][K] (output-major, K contiguous) is
 *     codes  uint32_t [N][K/8]   code k in bits 4*(k%8)..+3 of word k/8;
 *     scales uint16_t [N][K/64]  bf16 scale of weights k = 64g .. 64g+63;
 *     biases uint16_t [N][K/64]  bf16 bias of the same group;
 *   and W[n][k] = scale[n][k/64] * code(n,k) + bias[n][k/64], code in 0..15.
 *   Expert e's matrices start at e * (matrix size) in each array.
 *
 * Ownership and synchronisation: every pointer is a DEVICE pointer owned by
 * the caller (except shape/struct pointers, which are host pointers read
 * during the call). The library allocates no memory, keeps no state between
 * calls and never synchronises the host, except moe_status_read. All work is
 * enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream);
 * buffers must stay valid until the stream passes the call.
 *
 * Errors: argument, shape and workspace errors, and launch errors, are
 * returned synchronously. A device-side failure (a bounded wait that expired,
 * or a value outside the fp16 range below) is written to the int32 status
 * word of the call (route_out->status, or the workspace's own status word for
 * moe_forward without route_out) and the kernels after it do no work; read it
 * with moe_status_read. On any nonzero status y (and r_next) are not valid.
 *
 * Numerics: logits, softmax, gate and y are fp32. The expert products take
 * fp16 operands with fp32 accumulation: each weight is formed in fp16 as
 * fma(q 2^-14, scale 2^14, bias), an exact product rounded once (the GEMV
 * path keeps weights and x in fp32); x is rounded from bf16 to fp16; h (and
 * o, except on the fused decode path, which writes y from fp32 sums) are
 * stored as fp16. fp16 holds 11 significant bits on 2^-14 <= |v| <= 65504
 * and a fixed step of 2^-24 below. Ranges:
 *   x      |x| < 65520 (larger becomes inf in fp16): else MOE_ERR_RANGE.
 *   h, o   |value| < 65520: else MOE_ERR_RANGE. At the other end, a slice of
 *          h or o held together by one warp or block (8 to 512 values of
 *          one row or tile) whose values are all below 2^-16 and not all
 *          zero: MOE_ERR_RANGE (fp16's fixed step there exceeds 2^-9 of the
 *          slice's largest value).
 *   scale  |scale| < 4 on the fused decode and tensor-core paths (scale 2^14
 *          must fit fp16), else MOE_ERR_RANGE; any bf16 on the GEMV path.
 *          Small scales lose nothing beyond the weight's own rounding: a
 *          weight below 2^-14 is an fp16 subnormal (absolute error at most
 *          2^-25). Scales spread over 1e-7 .. 1e-4, with biases -8 scale +
 *          N(0, 1e-3) or following the scale, keep the layer within its
 *          tolerance (rel-L2 3e-3, max-abs 1e-2 RMS on y).
 *   bias   any bf16 value (rounded once to fp16).
 * Results are bit-identical from run to run (no float atomics).
 */
#ifndef BGMOE_MOE_H
#define BGMOE_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ABI_VERSION 1

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,         /* null pointer, negative size, ... */
  MOE_ERR_UNSUPPORTED_SHAPE = 2,   /* shape outside the supported set below */
  MOE_ERR_WORKSPACE_TOO_SMALL = 3, /* ws_bytes < moe_workspace_bytes() */
  MOE_ERR_CUDA = 4,                /* a CUDA runtime call or launch failed */
  MOE_ERR_DEVICE_TIMEOUT = 5,      /* a bounded device-side wait expired */
  MOE_ERR_RANGE = 6,               /* a value left the fp16 range of the expert path's operands
                                      (|x|, |h| or |o| >= 65520, a slice of h or o all under
                                      2^-16, or |scale| >= 4 where weights are fp16; see
                                      Numerics); the outputs are not valid */
  MOE_ERR_BOUNDS = 7               /* debug build only (BGMOE_BOUNDS_CHECK): an index read from a
                                      device-written table was out of range; the outputs are not valid */
} moe_status;

/* Shape of one call. Supported: T >= 0; H and I multiples of 64 with
 * 64 <= H <= 8192 and 64 <= I <= 4096; I_shared == I (one shared expert of
 * the same shape) or 0 (none); 1 <= top_k <= 8; top_k <= E <= 256;
 * group_size == 64; block_m in {16, 32, 64, 128}. */
typedef struct moe_shape {
  int32_t T;          /* tokens in this call */
  int32_t H;          /* hidden size */
  int32_t I;          /* routed expert intermediate size */
  int32_t I_shared;   /* shared expert intermediate size (I or 0) */
  int32_t E;          /* routed experts */
  int32_t top_k;      /* experts per token */
  int32_t group_size; /* weights per scale/bias pair (64) */
  int32_t block_m;    /* rows per block-map tile */
} moe_shape;

/* One packed 4-bit matrix stack (device pointers; layout in the file header). */
typedef struct moe_qmat {
  const uint32_t* codes;
  const uint16_t* scales;
  const uint16_t* biases;
} moe_qmat;

/* The expert weights of a layer: gate_up is [n][2I][H] (gate rows 0..I-1,
 * up rows I..2I-1), down is [n][H][I]; n = E for the routed experts, 1 for
 * the shared expert. */
typedef struct moe_experts {
  moe_qmat gate_up;
  moe_qmat down;
} moe_experts;

/* Routing outputs (device pointers, caller-owned; A = T * top_k):
 *   ids        int32 [T][top_k]  chosen experts, best first
 *   weights    fp32  [T][top_k]  renormalised softmax weights
 *   gate       fp32  [T]         shared-expert gate (may be NULL if I_shared == 0)
 *   counts     int32 [E+1]       assignments per expert; counts[E] = T if a
 *                                shared expert exists, else 0
 *   offsets    int32 [E+2]       exclusive prefix sum of counts
 *   sorted     int32 [A]         assignment a = t*top_k + k at each position;
 *                                positions of one expert follow increasing a
 *   inv        int32 [A]         position of each assignment
 *   tile_expert, tile_row0, tile_rows  int32 [moe_max_tiles()]  block map:
 *                                for e = 0..E in order, ceil(counts[e]/block_m)
 *                                tiles of <= block_m consecutive positions;
 *                                rows A + t belong to the shared expert (token t)
 *   num_tiles  int32 [1]         number of valid block-map entries
 *   status     int32 [1]         MOE_OK, or MOE_ERR_DEVICE_TIMEOUT
 * [dothoosh.com "Perplexity Lily...", "Prefill optimisations": routing
 * histogram, prefix scan, scatter and block map kept on the GPU.] */
typedef struct moe_route_out {
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
} moe_route_out;

/* ABI version of the loaded library (MOE_ABI_VERSION). */
int32_t moe_abi_version(void);

/* Text of a status code (static storage; never NULL). */
const char* moe_status_string(moe_status s);

/* Detail of the last MOE_ERR_CUDA returned on the calling thread (the CUDA
 * call and its error string); "" if none. Thread-local storage. */
const char* moe_last_error_detail(void);

/* Workspace bytes moe_route / moe_forward need for `shape` (a pure function
 * of the shape; no CUDA call). Errors: INVALID_ARG, UNSUPPORTED_SHAPE. */
moe_status moe_workspace_bytes(const moe_shape* shape, size_t* bytes);

/* Upper bound on the block-map length for `shape`:
 * ceil(A/block_m) + min(E, A) + ceil(T/block_m) (the last term only with a
 * shared expert). The tile_* arrays must hold this many entries. */
moe_status moe_max_tiles(const moe_shape* shape, int32_t* max_tiles);

/* Steps 1-2: router, top-k, weights, gate and the routing tables.
 *   x              bf16 [T][H]
 *   w_router       bf16 [E][H]
 *   router_bias    fp32 [E] or NULL (added to the logits before selection)
 *   w_shared_gate  bf16 [H]; required iff I_shared > 0
 *   out            every field required, except gate when I_shared == 0
 *   workspace      device buffer of >= moe_workspace_bytes() bytes, 256-byte
 *                  aligned; its contents need no initialisation */
moe_status moe_route(const moe_shape* shape, const void* x, const void* w_router,
                     const float* router_bias, const void* w_shared_gate,
                     const moe_route_out* out, void* workspace, size_t ws_bytes,
                     void* stream);

/* Steps 1-4: the whole layer, y fp32 [T][H].
 *   experts        routed experts (n = E)
 *   shared         the shared expert (n = 1); required iff I_shared > 0
 *   route_out      NULL, or routing outputs to keep (as moe_route)
 * Other arguments as moe_route. T == 0 is a no-op. */
moe_status moe_forward(const moe_shape* shape, const void* x, const void* w_router,
                       const float* router_bias, const moe_experts* experts,
                       const moe_experts* shared, const void* w_shared_gate,
                       float* y, const moe_route_out* route_out,
                       void* workspace, size_t ws_bytes, void* stream);

/* One pre-norm MoE block, for stacks of layers run back to back: the layer's
 * input is the RMS-normalised residual row and its output joins the
 * residual stream, which is the next call's r:
 *   x[t]      = r[t] / sqrt(mean_h r[t,h]^2 + norm_eps) * norm_weight   (fp32)
 *   y         = the layer of moe_forward applied to x                   (fp32 [T][H])
 *   r_next[t] = bf16_rn(r[t] + y[t])                                     (bf16 [T][H])
 * The pages' decode path writes each step's result straight into the
 * device-resident input slot of the next step [dothoosh.com "Perplexity
 * Lily: 1.35x faster decode for Qwen3.6 on Apple silicon", "Decode
 * optimisations", kernel-fusion item]. What joins two MoE layers is not on
 * the pages: the reading taken is the transformer's pre-norm residual block
 * (without a normalisation the synthetic weights' gain makes a stack of
 * layers overflow within three layers). x stays fp32 for the router and is
 * rounded once to fp16 for the expert products.
 *   r            bf16 [T][H], 16-byte aligned; r_next distinct from r, 16-byte aligned
 *   norm_weight  bf16 [H] gain, or NULL for a gain of 1 (16-byte aligned)
 *   norm_eps     > 0 (1e-6 in the workloads)
 * Runs on the fused decode path only (the shapes MOE_PATH_FUSED_DECODE
 * accepts; else UNSUPPORTED_SHAPE); y and r_next come out of the same
 * kernel. Other arguments and errors as moe_forward. */
moe_status moe_forward_residual(const moe_shape* shape, const void* r, const void* norm_weight,
                                float norm_eps, const void* w_router, const float* router_bias,
                                const moe_experts* experts, const moe_experts* shared,
                                const void* w_shared_gate, float* y, void* r_next,
                                const moe_route_out* route_out, void* workspace, size_t ws_bytes,
                                void* stream);

/* Expert-GEMM implementations selectable through moe_forward_timed. */
typedef enum moe_expert_path {
  MOE_PATH_AUTO = 0,        /* fused decode for T <= 4 when its conditions hold, tensor
                               cores for T >= 64 when the shape allows, else GEMV */
  MOE_PATH_GEMV = 1,        /* bandwidth-bound grouped GEMV (CUDA cores), any shape */
  MOE_PATH_TENSOR_CORE = 2, /* tcgen05 grouped GEMM; needs H % 256 == 0, I % 128 == 0 and
                               16-byte aligned codes, scales and biases (else
                               UNSUPPORTED_SHAPE) */
  MOE_PATH_FUSED_DECODE = 3 /* a one-block prelude and one fused kernel for the router,
                               top-k, tables, expert products and combine; needs T <= 4,
                               H % 512 == 0, H <= 2048, H / 16 <= the SM count,
                               I % 128 == 0, I <= 1024, E (+1 with a shared expert)
                               <= 15 x (SM count - I / 32), one 512-thread block of
                               about 170 KB of shared memory resident on every SM (no
                               other kernel may hold SMs while it runs: its blocks wait
                               for one another's data, with a 1 s limit) and 16-byte
                               aligned codes, scales and biases (else
                               UNSUPPORTED_SHAPE). Its events[1] and events[2] follow
                               events[0] at once and events[4..5] == events[3] */
} moe_expert_path;

/* moe_forward with a chosen expert path that also records caller-owned CUDA
 * events (cudaEvent_t created by the caller; events may be NULL) on `stream`
 * around its kernels: events[0] before the router kernel, [1] after it, [2]
 * after the routing kernel, [3] after the expert gate/up kernel, [4] after
 * the expert down kernel, [5] after the combine kernel. With events == NULL
 * and MOE_PATH_AUTO it is exactly moe_forward. For per-kernel timing on the
 * launching stream and for comparing the two expert paths. */
moe_status moe_forward_timed(const moe_shape* shape, const void* x, const void* w_router,
                             const float* router_bias, const moe_experts* experts,
                             const moe_experts* shared, const void* w_shared_gate,
                             float* y, const moe_route_out* route_out,
                             void* workspace, size_t ws_bytes, void* const* events,
                             int32_t expert_path, void* stream);

/* moe_route without a workspace, for callers that cannot allocate device
 * memory where they route (a host callback or real-time loop that must not
 * enter the CUDA allocator, a plugin given only its input and output buffers,
 * an embedder whose device memory is budgeted by a host framework). The
 * pages have no counterpart: this is a deployment convenience, not a step
 * of the layer. Same arguments and outputs as moe_route, minus the workspace.
 *   Scratch: a 1 MiB file-scope device array that every GPU loading this
 *   library holds until the process exits. A shape whose router logits
 *   (T * (E+1) * 4 bytes) plus look-back words no longer fit is refused with
 *   MOE_ERR_UNSUPPORTED_SHAPE (moe_last_error_detail gives both sizes); at
 *   E = 256 that is about 900 tokens per call.
 *   The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any
 *   stream capture.
 *   Every call on a device shares the one array and leaves its contents
 *   behind; each call clears what must start at zero. Calls that overlap on
 *   the GPU (two streams, or two host threads) race on the array: serialise
 *   them. The library allocates nothing on this path. */
moe_status moe_route_noalloc(const moe_shape* shape, const void* x, const void* w_router,
                             const float* router_bias, const void* w_shared_gate,
                             const moe_route_out* out, void* stream);

/* Reads a device status word written by a previous call: synchronises
 * `stream`, copies the word to *host_status. */
moe_status moe_status_read(const int32_t* device_status, void* stream, int32_t* host_status);

/* Test hook: moe_route with routing block `stalled_block` never publishing
 * its histogram, so that the blocks after it wait out `timeout_ns` and the
 * call ends with MOE_ERR_DEVICE_TIMEOUT in out->status (no hang, no trap).
 * Requires T * top_k large enough for more than one routing block
 * (moe_route_blocks() > stalled_block). */
moe_status moe_test_route_stall(const moe_shape* shape, const void* x, const void* w_router,
                                const float* router_bias, const void* w_shared_gate,
                                const moe_route_out* out, void* workspace, size_t ws_bytes,
                                int32_t stalled_block, int64_t timeout_ns, void* stream);

/* Test hook for the fused decode kernel's failure path: moe_forward_timed
 * with MOE_PATH_FUSED_DECODE, except that block `stalled_block` of the
 * decode kernel never publishes the h of its gate/up items, so the blocks
 * that need that h wait out `timeout_ns` (0 < timeout_ns <= 1 s; every
 * device wait of the call gives up after it). The call's status word then
 * reads MOE_ERR_DEVICE_TIMEOUT, every block has returned (having let its own
 * copies land) and the context stays usable. Same arguments as moe_forward;
 * UNSUPPORTED_SHAPE where the fused path is refused; INVALID_ARG for a
 * negative block or a timeout out of range (a block index past the grid
 * stalls nothing). */
moe_status moe_test_decode_stall(const moe_shape* shape, const void* x, const void* w_router,
                                 const float* router_bias, const moe_experts* experts, const moe_experts* shared,
                                 const void* w_shared_gate, float* y, const moe_route_out* route_out,
                                 void* workspace, size_t ws_bytes, int32_t stalled_block, int64_t timeout_ns,
                                 void* stream);

/* Number of thread blocks the routing kernel uses for `shape` on the current
 * device (the co-resident grid of the single-launch routing pipeline). */
moe_status moe_route_blocks(const moe_shape* shape, int32_t* blocks);

#ifdef __cplusplus
}
#endif

#endif /* BGMOE_MOE_H */
