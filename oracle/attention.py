"""fp64 CPU oracle of single-token decode attention with grouped-query heads
(test infrastructure only: the tests, the smoke check and the CPU-baseline leg
of the benchmark use it; the product path never does).

Source: dothoosh.com, "Perplexity Lily: 1.35x faster decode for Qwen3.6 on
Apple silicon". Its "Model specification" section gives the full-attention
layers of the model 16 query heads and 2 key/value heads (grouped-query
attention over a KV cache that grows with the context). Its "Decode
optimisations" section packs several query heads that share a KV head into
one thread group so that each cached key/value row is read once, splits the
context into fixed-size blocks, and reads the cache with coalesced loads. Those
are ways of computing the same attention; this file states the attention
itself, as its plain definition:

    o[b, h] = sum_j softmax_j(scale * q[b, h] . K[b, g(h), j]) V[b, g(h), j]

Readings taken where the page is silent (the CUDA path follows the same ones):
  * g(h) = h // (Hq / Hkv): consecutive query heads share a KV head;
  * the cache of sequence b holds lens[b] positions, the new token's own key and
    value included, and the new query attends to every one of them;
  * scale = 1 / sqrt(D) unless given;
  * an empty cache (lens[b] = 0) gives o[b] = 0;
  * the head size D is not stated; the workloads take D = 256.

Parity status: pinned by tests/oracle_pins.py (closed forms for one and two
positions, equal keys, the head mapping, masking past lens, permutation and
shift invariance, and torch's scaled_dot_product_attention on full caches).
"""
from __future__ import annotations

import math

import numpy as np

from .moe import bf16_bits_to_f64


def gqa_decode_attention(q_bits, k_bits, v_bits, lens, scale=None) -> np.ndarray:
    """Decode attention of one new token per sequence over its KV cache.

    q_bits uint16 bf16 patterns [B, Hq, D]; k_bits, v_bits uint16 [B, Hkv, L_max, D];
    lens int [B] with 0 <= lens[b] <= L_max. Returns fp64 [B, Hq, D].
    """
    q = bf16_bits_to_f64(q_bits)
    K = bf16_bits_to_f64(k_bits)
    V = bf16_bits_to_f64(v_bits)
    B, Hq, D = q.shape
    Hkv = K.shape[1]
    if Hq % Hkv != 0:
        raise ValueError(f"Hq={Hq} is not a multiple of Hkv={Hkv}")
    per_kv = Hq // Hkv
    s = 1.0 / math.sqrt(D) if scale is None else float(scale)
    lens = np.asarray(lens, dtype=np.int64)
    o = np.zeros((B, Hq, D), dtype=np.float64)
    for b in range(B):
        n = int(lens[b])
        if not 0 <= n <= K.shape[2]:
            raise ValueError(f"lens[{b}]={n} outside 0..{K.shape[2]}")
        if n == 0:
            continue
        for h in range(Hq):
            g = h // per_kv
            logits = s * (K[b, g, :n] @ q[b, h])
            w = np.exp(logits - logits.max())
            w /= w.sum()
            o[b, h] = w @ V[b, g, :n]
    return o
