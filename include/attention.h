/*
 * bit_grouped_expert_moe_gb300 — C ABI of single-token decode attention with
 * grouped-query heads over a bf16 KV cache, for NVIDIA GB300 (sm_103a).
 *
 * The operation [dothoosh.com "Perplexity Lily: 1.35x faster decode for
 * Qwen3.6 on Apple silicon", section "Model specification": the model's
 * full-attention layers use grouped-query attention, 16 query heads sharing
 * 2 key/value heads, over a KV cache that grows with the context]:
 *
 *   o[b,h,:] = sum_{j < lens[b]} softmax_j(scale * q[b,h,:] . K[b,g,j,:]) V[b,g,j,:]
 *   with g = h / (Hq / Hkv)  (consecutive query heads share a KV head).
 *
 * The cache of sequence b holds lens[b] positions (the new token's own key and
 * value already appended); the query attends to all of them. lens[b] = 0 gives
 * o[b] = 0. How it is computed follows the same section's decode items: all
 * query heads of one KV head are packed into one block so that every cached
 * key/value row is read from memory once; the context is cut into fixed
 * blocks of 64 positions, each giving a partial softmax state that a second
 * kernel merges; cache rows are read by TMA in whole 128-byte lines.
 *
 * Layouts (row-major, bf16 values as their 16-bit patterns):
 *   q        uint16_t [B][Hq][D]
 *   k_cache  uint16_t [B][Hkv][L_max][D]
 *   v_cache  uint16_t [B][Hkv][L_max][D]
 *   lens     int32_t  [B]            0 <= lens[b] <= L_max
 *   o        float    [B][Hq][D]     fp32 output
 *
 * Ownership and synchronisation as in moe.h: every array is a DEVICE pointer
 * owned by the caller; the shape is a host pointer read during the call; the
 * library allocates nothing, keeps no state between calls, never synchronises
 * the host, and enqueues all work on `stream` (a cudaStream_t).
 *
 * Errors: argument, shape, alignment and workspace errors and launch errors
 * are returned synchronously. Device-side failures are written to the int32
 * status word at the start of the workspace (read it with moe_status_read):
 * MOE_ERR_INVALID_ARG when some lens[b] lies outside 0..L_max (o is then not
 * written), MOE_ERR_DEVICE_TIMEOUT when a bounded wait expired.
 *
 * Numerics: scores q.K in fp32 from exact bf16 products; softmax in fp32 on
 * the base-2 scale; the probabilities are rounded to bf16 for the P.V
 * product (fp32 accumulation), and the softmax denominators sum the same
 * rounded values, so every output is a convex combination of cached values.
 * Results are bit-identical from run to run.
 */
#ifndef BGMOE_ATTENTION_H
#define BGMOE_ATTENTION_H

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Shape of one call. Supported: 1 <= B <= 4096; 1 <= Hkv; Hq a multiple of
 * Hkv with 1 <= Hq / Hkv <= 8; B * Hkv <= 65536; D in {64, 128, 256};
 * 1 <= L_max <= 2^26. */
typedef struct moe_attn_shape {
  int32_t B;      /* sequences (one new token each) */
  int32_t Hq;     /* query heads */
  int32_t Hkv;    /* key/value heads */
  int32_t D;      /* head size */
  int32_t L_max;  /* cache rows per (sequence, KV head) */
} moe_attn_shape;

/* Bytes of device workspace moe_attn_decode needs for `shape` (the status word
 * and the partial softmax states of the fixed blocks). */
moe_status moe_attn_workspace_bytes(const moe_attn_shape* shape, size_t* bytes);

/* Decode attention of one new token per sequence (the formula above).
 * q, k_cache, v_cache and o must be 16-byte aligned and the
 * workspace 256-byte aligned, with ws_bytes >= moe_attn_workspace_bytes().
 * scale must be finite and > 0 (1/sqrt(D) is the usual value). */
moe_status moe_attn_decode(const moe_attn_shape* shape, const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* lens, float scale, float* o, void* workspace, size_t ws_bytes,
                           void* stream);

/* moe_attn_decode recording three caller-created CUDA events (cudaEvent_t
 * handles) on `stream`: before the block kernel, between the block kernel and
 * the merge kernel, and after the merge kernel. */
moe_status moe_attn_decode_timed(const moe_attn_shape* shape, const void* q, const void* k_cache,
                                 const void* v_cache, const int32_t* lens, float scale, float* o, void* workspace,
                                 size_t ws_bytes, void* const* events, void* stream);

/* Test hook for the block kernel's failure path: moe_attn_decode, except that
 * grid block `stalled_block` (0-based, below the grid of one block per SM; a
 * block past the grid changes nothing) issues none of its cache loads, so its
 * consumers' bounded waits run out after `timeout_ns` (0 < timeout_ns <= 1 s;
 * every wait of the call gives up after it). The call's status word (the
 * first 4 bytes of the workspace) then reads MOE_ERR_DEVICE_TIMEOUT, no block
 * exits with a copy in flight, o is not valid, and the context stays usable.
 * INVALID_ARG for a negative block or a timeout out of range; the other
 * checks are moe_attn_decode's. */
moe_status moe_attn_test_stall(const moe_attn_shape* shape, const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* lens, float scale, float* o, void* workspace, size_t ws_bytes,
                               int32_t stalled_block, int64_t timeout_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BGMOE_ATTENTION_H */
