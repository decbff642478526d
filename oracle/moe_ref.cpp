// Plain, slow fp64 CPU statement of one bit-grouped-expert MoE layer, in C++.
//
// Test infrastructure only: the tests, the smoke check and the benchmark's
// CPU-baseline and reference legs load it; the CUDA library never does, and
// the two share no code (no header, helper or constant of the library is
// used here).
//
// Sources (three web pages on Perplexity's Lily engine for Qwen3.6-35B-A3B):
//   [dothoosh] "Perplexity Lily: 1.35x faster decode for Qwen3.6 on Apple
//              silicon", sections "Model specification", "Prefill
//              optimisations", "Decode optimisations"
//   [aikraft]  "Perplexity open-sources Lily, a Rust/Metal inference engine
//              for Qwen3.6", "Architecture of Qwen3.6-35B-A3B"
//   [droneth]  the Lily article on droneth.or.th, "a large model that touches
//              only part of its weights per token"
// Each function names the passage it follows and the reading taken where the
// pages are silent; the readings are the same as those of the numpy oracle
// (oracle/moe.py), which this file restates independently, loop by loop.
//
// Conventions (the data format, not arithmetic): bf16 values arrive as raw
// 16-bit patterns, packed 4-bit codes as uint32 words, arrays row-major.
//
// BGREF_MUTANT (compile-time, default 0) plants one plausible mistake per
// value; the planted-mistake tests build those variants and check that a pin
// fails for each. A normal build has no mutant.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#ifndef BGREF_MUTANT
#define BGREF_MUTANT 0
#endif

namespace {

constexpr int kGroup = 64;   // weights per bf16 scale/bias pair
constexpr int kNibbles = 8;  // 4-bit codes per uint32 word

// A bf16 value is the upper half of the fp32 value with the same bits; the
// widening to fp64 is exact.
double bf16(uint16_t bits) {
  const uint32_t u = (uint32_t)bits << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return (double)f;
}

double silu(double a) {
#if BGREF_MUTANT == 4
  return a / (1.0 + std::exp(a));
#else
  return a / (1.0 + std::exp(-a));
#endif
}

double sigmoid(double a) {
#if BGREF_MUTANT == 7
  return std::tanh(a);
#else
  return 1.0 / (1.0 + std::exp(-a));
#endif
}

}  // namespace

extern "C" {

void bgref_bf16_to_f64(int64_t n, const uint16_t* bits, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = bf16(bits[i]);
}

// Groupwise-affine 4-bit dequantisation [dothoosh "Prefill optimisations",
// fused-dequantisation item; droneth, "a large model ..."]: 4-bit weights in
// groups of 64 along k that share one bf16 scale and one bf16 bias.
// Readings: W[n][k] = scale[n][k / 64] * q + bias[n][k / 64] with q the
// unsigned code of weight k, which sits in bits 4 (k % 8) .. +3 of word k / 8.
// codes [N][K/8], scales and biases [N][K/64] -> W [N][K].
void bgref_dequant(int N, int K, const uint32_t* codes, const uint16_t* scales, const uint16_t* biases, double* W) {
  for (int n = 0; n < N; ++n) {
    for (int k = 0; k < K; ++k) {
      const uint32_t word = codes[(int64_t)n * (K / kNibbles) + k / kNibbles];
#if BGREF_MUTANT == 1
      const int shift = 4 * (7 - k % kNibbles);
#else
      const int shift = 4 * (k % kNibbles);
#endif
      const double q = (double)((word >> shift) & 15u);
#if BGREF_MUTANT == 11
      const int g = k / 32 < K / kGroup ? k / 32 : K / kGroup - 1;
#else
      const int g = k / kGroup;
#endif
      const double s = bf16(scales[(int64_t)n * (K / kGroup) + g]);
      const double b = bf16(biases[(int64_t)n * (K / kGroup) + g]);
#if BGREF_MUTANT == 2
      W[(int64_t)n * K + k] = s * q - b;
#else
      W[(int64_t)n * K + k] = s * q + b;
#endif
    }
  }
}

// Router scores [dothoosh "Model specification"; aikraft "Architecture of
// Qwen3.6-35B-A3B"]: every token is scored against all experts,
// l[t][e] = sum_h x[t][h] W_r[e][h], plus an optional fp32 per-expert bias.
void bgref_router_logits(int T, int H, int E, const double* x, const uint16_t* wr, const float* bias, double* l) {
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int h = 0; h < H; ++h) acc += x[(int64_t)t * H + h] * bf16(wr[(int64_t)e * H + h]);
#if BGREF_MUTANT == 10
      (void)bias;
#else
      if (bias != nullptr) acc += (double)bias[e];
#endif
      l[(int64_t)t * E + e] = acc;
    }
  }
}

// The top_k experts of each token, best first [dothoosh "Model
// specification": 8 of 256 experts]. Readings: the ranking compares the
// logits rounded to fp32 (the precision the kernels decide in); equal logits
// go to the lower expert index. Written as k rounds of a scan for the best
// expert not yet chosen.
void bgref_select_top_k(int T, int E, int K, const double* l, int32_t* ids) {
  std::vector<char> taken(E);
  for (int t = 0; t < T; ++t) {
    std::fill(taken.begin(), taken.end(), 0);
    for (int k = 0; k < K; ++k) {
      int best = -1;
      float bv = 0.f;
      for (int e = 0; e < E; ++e) {
        if (taken[e]) continue;
        const float v = (float)l[(int64_t)t * E + e];
#if BGREF_MUTANT == 3
        if (best < 0 || v >= bv) {
#else
        if (best < 0 || v > bv) {
#endif
          best = e;
          bv = v;
        }
      }
      taken[best] = 1;
      ids[(int64_t)t * K + k] = best;
    }
  }
}

// Router, top-k, renormalised softmax weights and the shared-expert gate.
// Readings: the weights are a softmax over all experts renormalised over the
// selected ones, i.e. exp(l_k - l_max) / sum over the selected j of
// exp(l_j - l_max); the shared expert, which processes every token
// [dothoosh "Model specification"], is scaled by sigmoid(sum_h x[t][h] w_sg[h]).
// x fp64 [T][H]; wsg may be null (no shared expert: gate untouched).
void bgref_route(int T, int H, int E, int K, const double* x, const uint16_t* wr, const float* bias,
                 const uint16_t* wsg, double* logits, int32_t* ids, double* weights, double* gate) {
  bgref_router_logits(T, H, E, x, wr, bias, logits);
  bgref_select_top_k(T, E, K, logits, ids);
  for (int t = 0; t < T; ++t) {
    const double* lt = logits + (int64_t)t * E;
    const double top = lt[ids[(int64_t)t * K]];
    double sum = 0.0;
#if BGREF_MUTANT == 6
    for (int e = 0; e < E; ++e) sum += std::exp(lt[e] - top);
#else
    for (int k = 0; k < K; ++k) sum += std::exp(lt[ids[(int64_t)t * K + k]] - top);
#endif
    for (int k = 0; k < K; ++k) weights[(int64_t)t * K + k] = std::exp(lt[ids[(int64_t)t * K + k]] - top) / sum;
    if (wsg != nullptr) {
      double s = 0.0;
      for (int h = 0; h < H; ++h) s += x[(int64_t)t * H + h] * bf16(wsg[h]);
      gate[t] = sigmoid(s);
    }
  }
}

// Expert-contiguous routing tables [dothoosh "Prefill optimisations",
// GPU-resident routing item; droneth, same list]: a histogram, a prefix scan,
// a scatter and a block map.
//   counts[e]  assignments a = t K + k with ids[a] == e; counts[E] = T for the
//              shared expert (every token), 0 without one
//   offsets    exclusive prefix sum of counts, E + 2 entries
//   sorted[p]  the assignment at position p; inside one expert, positions
//              follow increasing a (a stable counting sort)
//   inv[a]     the position of assignment a
//   tiles      for e = 0 .. E, ceil(counts[e] / block_m) runs of at most
//              block_m consecutive positions: (expert, first position, rows)
// The shared expert's rows are positions A .. A + T - 1. Returns the number
// of tiles, or -1 when more than max_tiles would be written.
int bgref_routing_tables(int T, int K, int E, int block_m, int shared, const int32_t* ids, int32_t* counts,
                         int32_t* offsets, int32_t* sorted, int32_t* inv, int32_t* tile_expert, int32_t* tile_row0,
                         int32_t* tile_rows, int max_tiles) {
  const int A = T * K;
  for (int e = 0; e <= E; ++e) counts[e] = 0;
  for (int a = 0; a < A; ++a) counts[ids[a]] += 1;
#if BGREF_MUTANT == 9
  (void)shared;
#else
  if (shared) counts[E] = T;
#endif
  offsets[0] = 0;
  for (int e = 0; e <= E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  std::vector<int32_t> fill(offsets, offsets + E);
  for (int a = 0; a < A; ++a) {
    const int e = ids[a];
    sorted[fill[e]] = a;
    inv[a] = fill[e];
    fill[e] += 1;
  }
  int n = 0;
  for (int e = 0; e <= E; ++e) {
    for (int j = 0; j * block_m < counts[e]; ++j) {
      if (n >= max_tiles) return -1;
      tile_expert[n] = e;
      tile_row0[n] = offsets[e] + j * block_m;
      tile_rows[n] = std::min(block_m, counts[e] - j * block_m);
      ++n;
    }
  }
  return n;
}

// One SwiGLU expert on n token rows, fp64 throughout. Readings: gate and up
// are the first and second halves of the [2I][H] gate_up matrix;
// h = silu(gate) * up with silu(a) = a / (1 + exp(-a)); o = W_down h with
// W_down stored [H][I]. The pages fix FP32 accumulation for the GPU
// [dothoosh "Prefill optimisations"]; here every value stays fp64.
void bgref_swiglu(int n, int H, int I, const double* x, const double* w_gu, const double* w_dn, double* o) {
  std::vector<double> h(I);
  for (int r = 0; r < n; ++r) {
    const double* xr = x + (int64_t)r * H;
    for (int i = 0; i < I; ++i) {
      double g = 0.0, u = 0.0;
      for (int k = 0; k < H; ++k) {
        g += w_gu[(int64_t)i * H + k] * xr[k];
        u += w_gu[(int64_t)(I + i) * H + k] * xr[k];
      }
#if BGREF_MUTANT == 5
      h[i] = silu(u) * g;
#else
      h[i] = silu(g) * u;
#endif
    }
    for (int m = 0; m < H; ++m) {
      double acc = 0.0;
      for (int i = 0; i < I; ++i) acc += w_dn[(int64_t)m * I + i] * h[i];
      o[(int64_t)r * H + m] = acc;
    }
  }
}

// The layer's output for n tokens given their routing [dothoosh "Model
// specification": 8 routed experts plus one shared expert for every token]:
//   y[t] = sum_k w[t][k] Expert_{ids[t][k]}(x_t) + gate[t] Shared(x_t).
// Packed weights come as tables of E + 1 pointers (entry E: the shared
// expert), gate_up codes [2I][H/8] with scales/biases [2I][H/64], down codes
// [H][I/8] with scales/biases [H][I/64]; only the experts the tokens use
// (and the shared one when gate is given) are read. Each used expert is
// dequantised once. Returns 0, or -1 when a needed pointer is null.
int bgref_moe_experts(int n, int H, int I, int E, int K, const double* x, const int32_t* ids, const double* weights,
                      const double* gate, const uint32_t* const* gu_codes, const uint16_t* const* gu_scales,
                      const uint16_t* const* gu_biases, const uint32_t* const* dn_codes,
                      const uint16_t* const* dn_scales, const uint16_t* const* dn_biases, double* y) {
  for (int64_t i = 0; i < (int64_t)n * H; ++i) y[i] = 0.0;
  std::vector<double> w_gu((size_t)2 * I * H), w_dn((size_t)H * I), o(H);
  for (int e = 0; e <= E; ++e) {
    bool used = false;
    if (e < E) {
      for (int a = 0; a < n * K && !used; ++a) used = ids[a] == e;
    } else {
      used = gate != nullptr;
    }
    if (!used) continue;
    if (!gu_codes[e] || !gu_scales[e] || !gu_biases[e] || !dn_codes[e] || !dn_scales[e] || !dn_biases[e]) return -1;
    bgref_dequant(2 * I, H, gu_codes[e], gu_scales[e], gu_biases[e], w_gu.data());
    bgref_dequant(H, I, dn_codes[e], dn_scales[e], dn_biases[e], w_dn.data());
    for (int t = 0; t < n; ++t) {
      double wt = 0.0;
      bool hit = false;
      if (e < E) {
        for (int k = 0; k < K; ++k)
          if (ids[(int64_t)t * K + k] == e) {
            wt = weights[(int64_t)t * K + k];
            hit = true;
          }
      } else {
#if BGREF_MUTANT == 8
        wt = 1.0;
#else
        wt = gate[t];
#endif
        hit = true;
      }
      if (!hit) continue;
      bgref_swiglu(1, H, I, x + (int64_t)t * H, w_gu.data(), w_dn.data(), o.data());
      for (int m = 0; m < H; ++m) y[(int64_t)t * H + m] += wt * o[m];
    }
  }
  return 0;
}

// The input of a pre-norm MoE block, fp64 [T][H]:
//   x[t] = r[t] / sqrt(mean_h r[t][h]^2 + eps) * gain.
// The pages do not say what joins two MoE layers; the reading taken is the
// transformer's pre-norm residual block. gain (bf16 [H]) may be null (1).
void bgref_rms_norm(int T, int H, const uint16_t* r, double eps, const uint16_t* gain, double* x) {
  for (int t = 0; t < T; ++t) {
    double ss = 0.0;
    for (int h = 0; h < H; ++h) {
      const double v = bf16(r[(int64_t)t * H + h]);
      ss += v * v;
    }
#if BGREF_MUTANT == 12
    const double inv = 1.0 / (ss / H + eps);
#else
    const double inv = 1.0 / std::sqrt(ss / H + eps);
#endif
    for (int h = 0; h < H; ++h) {
      const double g = gain != nullptr ? bf16(gain[h]) : 1.0;
      x[(int64_t)t * H + h] = bf16(r[(int64_t)t * H + h]) * inv * g;
    }
  }
}

}  // extern "C"
