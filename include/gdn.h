/*
 * bit_grouped_expert_moe_gb300 — C ABI of the Gated DeltaNet recurrence
 * (the model's linear-attention layers), for NVIDIA GB300 (sm_103a).
 *
 * [dothoosh.com "Perplexity Lily: 1.35x faster decode for Qwen3.6 on Apple
 * silicon": "Model specification" gives the model 30 Gated DeltaNet layers, a
 * recurrence with a fixed-size state; "Prefill optimisations" keeps the scan's
 * state in registers. The recurrence itself is the gated delta rule of Yang,
 * Kautz and Hatamizadeh, "Gated Delta Networks" (ICLR 2025).]
 *
 * Per sequence and value head h (query/key head g = h / (Hv / Hqk)), token t:
 *   k^ = k_t / sqrt(|k_t|^2 + 1e-6),   q^ = q_t / sqrt(|q_t|^2 + 1e-6) / sqrt(Dk)
 *   S  = exp(gate_t) S                                  (decay)
 *   S  = S + beta_t (v_t - S k^) k^T                    (delta-rule write)
 *   o_t = S q^
 * S is the [Dv][Dk] fp32 state, carried from state_in to state_out.
 *
 * Layouts (row-major; bf16 values as their 16-bit patterns). The B sequences
 * are packed end to end: sequence b owns tokens offsets[b] .. offsets[b+1]-1.
 *   q, k       uint16_t [T][Hqk][Dk]
 *   v          uint16_t [T][Hv][Dv]
 *   gate, beta float    [T][Hv]        gate = log of the decay (<= 0)
 *   offsets    int32_t  [B+1]          0 = offsets[0] <= ... <= offsets[B] = T
 *   state_in   float    [B][Hv][Dv][Dk]
 *   state_out  float    [B][Hv][Dv][Dk]  may be the same buffer as state_in
 *   o          float    [T][Hv][Dv]
 *   status     int32_t  (device word; may be NULL)
 *
 * Ownership, streams and errors as in moe.h: device pointers owned by the
 * caller, host shape pointer, no allocation, no host synchronisation; argument
 * errors are returned synchronously. A sequence whose offsets are out of order
 * or out of range is skipped and MOE_ERR_INVALID_ARG is written to *status
 * (when given); the caller zeroes *status before the call.
 *
 * Numerics: fp32 throughout (bf16 inputs widened exactly); no atomics, so
 * results are bit-identical from run to run.
 */
#ifndef BGMOE_GDN_H
#define BGMOE_GDN_H

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Supported: 1 <= B <= 65535; 0 <= T <= 2^24; Hqk >= 1; Hv a multiple of
 * Hqk, Hv <= 4096; Dk = Dv = 128. */
typedef struct moe_gdn_shape {
  int32_t B;    /* sequences */
  int32_t T;    /* tokens of all sequences */
  int32_t Hqk;  /* query/key heads */
  int32_t Hv;   /* value heads */
  int32_t Dk;   /* key head size */
  int32_t Dv;   /* value head size */
} moe_gdn_shape;

/* The recurrence over every sequence's tokens (formula above). q, k, v,
 * state_in and state_out must be 16-byte aligned, the rest 4-byte aligned. */
moe_status moe_gdn_scan(const moe_gdn_shape* shape, const void* q, const void* k, const void* v, const float* gate,
                        const float* beta, const int32_t* offsets, const float* state_in, float* state_out,
                        float* o, int32_t* status, void* stream);

/* moe_gdn_scan recording two caller-created CUDA events (cudaEvent_t) on
 * `stream` before and after its kernel. */
moe_status moe_gdn_scan_timed(const moe_gdn_shape* shape, const void* q, const void* k, const void* v,
                              const float* gate, const float* beta, const int32_t* offsets, const float* state_in,
                              float* state_out, float* o, int32_t* status, void* const* events, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* BGMOE_GDN_H */
