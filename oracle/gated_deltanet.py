"""fp64 CPU oracle of the Gated DeltaNet recurrence (test infrastructure only:
the tests, the smoke check and the CPU-baseline leg of the benchmark use it;
the product path never does).

Sources. dothoosh.com, "Perplexity Lily: 1.35x faster decode for Qwen3.6 on
Apple silicon": its "Model specification" section gives the model 30 Gated
DeltaNet layers beside its 10 attention layers, a recurrence whose state has a
fixed size; its "Prefill optimisations" section credits a register-resident
Gated DeltaNet scan with a further 5.6 %. The page states no formula. The
recurrence is the gated delta rule as published by Yang, Kautz and
Hatamizadeh, "Gated Delta Networks: Improving Mamba2 with Delta Rule" (ICLR
2025), written out here per sequence and value head:

    S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
        = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T
    o_t = S_t q_t

with S a [Dv x Dk] matrix, alpha_t = exp(gate_t) in (0, 1] and beta_t in [0, 1].

Readings taken where the page is silent (the CUDA path follows the same ones):
  * q and k are L2-normalised per head and token (x / sqrt(sum x^2 + eps),
    eps = 1e-6) and q is then scaled by 1/sqrt(Dk), as in the paper's model;
  * Hv value heads share Hqk query/key heads in consecutive groups: value
    head h reads query/key head h // (Hv / Hqk);
  * the gate arrives as its logarithm (gate_t <= 0), beta directly;
  * every sequence starts from a given state and returns its final state
    (fp32 on the device); a sequence with no tokens returns its state as is;
  * sizes are not stated; the workloads take Hqk = 16, Hv = 32, Dk = Dv = 128.

Parity status: pinned by tests/oracle_pins.py (retrieval after a full write,
orthonormal keys reducing to linear attention, pure decay, head grouping,
invariance to the scale of q and k, and splitting a sequence in two calls).
"""
from __future__ import annotations

import math

import numpy as np

from .moe import bf16_bits_to_f64

EPS = 1e-6


def _l2n(x: np.ndarray) -> np.ndarray:
    return x / np.sqrt((x * x).sum() + EPS)


def gated_delta_scan(q_bits, k_bits, v_bits, gate, beta, state0, offsets):
    """The recurrence over packed sequences.

    q_bits, k_bits uint16 bf16 patterns [T, Hqk, Dk]; v_bits [T, Hv, Dv];
    gate, beta float [T, Hv]; state0 float [B, Hv, Dv, Dk]; offsets int [B+1]
    (sequence b owns tokens offsets[b] .. offsets[b+1]-1).
    Returns (o fp64 [T, Hv, Dv], state fp64 [B, Hv, Dv, Dk]).
    """
    q = bf16_bits_to_f64(q_bits)
    k = bf16_bits_to_f64(k_bits)
    v = bf16_bits_to_f64(v_bits)
    gate = np.asarray(gate, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    S_all = np.array(state0, dtype=np.float64, copy=True)
    offsets = np.asarray(offsets, dtype=np.int64)
    T, Hqk, Dk = q.shape
    Hv, Dv = v.shape[1], v.shape[2]
    if Hv % Hqk != 0:
        raise ValueError(f"Hv={Hv} is not a multiple of Hqk={Hqk}")
    per = Hv // Hqk
    qscale = 1.0 / math.sqrt(Dk)
    o = np.zeros((T, Hv, Dv), dtype=np.float64)
    for b in range(len(offsets) - 1):
        for h in range(Hv):
            g = h // per
            S = S_all[b, h]
            for t in range(int(offsets[b]), int(offsets[b + 1])):
                kh = _l2n(k[t, g])
                qh = _l2n(q[t, g]) * qscale
                a = math.exp(gate[t, h])
                S *= a
                vn = beta[t, h] * (v[t, h] - S @ kh)
                S += np.outer(vn, kh)
                o[t, h] = S @ qh
    return o, S_all
