"""fp64 CPU oracle of the MoE layer (test infrastructure; see the package
docstring for the sources and the rule that only tests, the smoke check and the
CPU-baseline leg of the benchmark use it).

Conventions shared with the library's C ABI (they are the data format, not
arithmetic): bf16 values arrive as their raw 16-bit patterns (uint16),
packed 4-bit codes as uint32 words, all arrays row-major.

Parity status: every function here is pinned by the `-m "not gpu"` tests in
tests/test_oracle_pins.py (hand-worked values, closed forms, invariants, brute
force on tiny inputs, and planted mistakes that those pins must catch).
"""
from __future__ import annotations

import numpy as np

GROUP = 64   # weights per bf16 scale/bias pair
NIBBLES = 8  # 4-bit codes per uint32 word


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Widen raw bf16 bit patterns (uint16) to fp64 exactly: a bf16 value is the
    upper half of the fp32 value with the same bits."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def dequant(codes, scales, biases, group: int = GROUP) -> np.ndarray:
    """Groupwise-affine 4-bit dequantisation, fp64, output-major [N, K].

    [dothoosh "Prefill optimisations", fused dequantisation item; droneth,
    "a large model that touches only part of its weights per token"]: the
    checkpoint stores 4-bit weights in groups of 64 that share one bf16 scale
    and one bf16 bias. Readings taken where the pages are silent:
      * affine form  W[n, k] = scale[n, k // 64] * q[n, k] + bias[n, k // 64],
        with q the unsigned code 0..15;
      * groups run along k, the input (reduction) dimension;
      * 8 codes per little-endian uint32 word, code k in bits 4*(k % 8) .. +3
        of word k // 8 (low nibble = lower k).
    codes uint32 [N, K/8]; scales, biases bf16 bits [N, K/64] -> fp64 [N, K].
    """
    codes = np.asarray(codes).view(np.uint32) if np.asarray(codes).dtype != np.uint32 else np.asarray(codes)
    N, KW = codes.shape
    K = KW * NIBBLES
    shifts = (4 * np.arange(NIBBLES, dtype=np.uint32))
    q = (codes[:, :, None] >> shifts[None, None, :]) & np.uint32(0xF)       # [N, K/8, 8]
    q = q.reshape(N, K).astype(np.float64)
    s = np.repeat(bf16_bits_to_f64(scales), group, axis=1)
    b = np.repeat(bf16_bits_to_f64(biases), group, axis=1)
    assert s.shape == (N, K), (s.shape, N, K)
    return s * q + b


def router_logits(x_bits, wr_bits, bias=None) -> np.ndarray:
    """Router scores of every token for every expert, fp64 [T, E].

    [dothoosh "Model specification"; aikraft "Architecture of Qwen3.6-35B-A3B";
    droneth, "a large model..."]: the router scores all 256 experts for each
    token. l[t, e] = sum_h x[t, h] * W_r[e, h] (+ b[e], an optional fp32
    per-expert logit bias added before selection and softmax)."""
    x = bf16_bits_to_f64(x_bits)
    w = bf16_bits_to_f64(wr_bits)
    l = x @ w.T
    if bias is not None:
        l = l + np.asarray(bias, dtype=np.float32).astype(np.float64)[None, :]
    return l


def select_top_k(logits, top_k: int) -> np.ndarray:
    """The top_k experts of every token, best first, int32 [T, top_k].

    [dothoosh "Model specification"]: the router picks 8 of the 256 experts.
    Readings: the ranking compares the logits rounded to fp32 (the precision
    the kernels decide in); equal logits are broken by the lower expert index.
    A stable sort on the negated logits does exactly that: it keeps equal keys
    in index order."""
    l32 = np.asarray(logits).astype(np.float32)
    order = np.argsort(-l32, axis=1, kind="stable")
    return order[:, :top_k].astype(np.int32)


def topk_gap(logits, top_k: int) -> np.ndarray:
    """l_(k) - l_(k+1) per token on the fp32 logits (inf when top_k == E): the
    margin that separates the selected experts from the first one left out."""
    l32 = np.sort(np.asarray(logits).astype(np.float32).astype(np.float64), axis=1)[:, ::-1]
    if top_k >= l32.shape[1]:
        return np.full(l32.shape[0], np.inf)
    return l32[:, top_k - 1] - l32[:, top_k]


def rms_norm(r_bits, eps: float, gain_bits=None) -> np.ndarray:
    """The input of a pre-norm MoE block, fp64 [T, H]:
    x[t] = r[t] / sqrt(mean_h r[t, h]^2 + eps) * gain.

    The pages do not say what joins two consecutive MoE layers. The reading
    taken for running layers back to back is the transformer's pre-norm
    residual block: each layer reads the RMS-normalised residual row and adds
    its output back to that row. `gain` (bf16 [H]) is the normalisation's
    per-channel scale, 1 when absent."""
    r = bf16_bits_to_f64(r_bits)
    x = r / np.sqrt(np.mean(r * r, axis=1, keepdims=True) + eps)
    if gain_bits is not None:
        x = x * bf16_bits_to_f64(gain_bits)[None, :]
    return x


def _logits_f64(x, wr_bits, bias):
    l = x @ bf16_bits_to_f64(wr_bits).T
    if bias is not None:
        l = l + np.asarray(bias, dtype=np.float32).astype(np.float64)[None, :]
    return l


def route(x_bits, wr_bits, bias, wsg_bits, top_k: int, x_f64=None):
    """Router + top-k + renormalised softmax weights + shared-expert gate.

    Returns (ids int32 [T, k], weights fp64 [T, k], gate fp64 [T] or None,
    logits fp64 [T, E]).
    Readings where the pages are silent: the weights are a softmax over all
    experts renormalised over the selected ones, which equals
    exp(l_k - l_max) / sum_j exp(l_j - l_max) over the selected j; the shared
    expert (which processes every token, [dothoosh "Model specification"]) is
    scaled by the gate sigmoid(sum_h x[t, h] * w_sg[h]). `x_f64`, when given,
    is the input itself in fp64 (a normalised residual row) and x_bits is
    ignored."""
    l = router_logits(x_bits, wr_bits, bias) if x_f64 is None else _logits_f64(x_f64, wr_bits, bias)
    ids = select_top_k(l, top_k)
    sel = np.take_along_axis(l, ids.astype(np.int64), axis=1)
    z = np.exp(sel - sel[:, :1])
    w = z / z.sum(axis=1, keepdims=True)
    gate = None
    if wsg_bits is not None:
        xs = bf16_bits_to_f64(x_bits) if x_f64 is None else x_f64
        s = xs @ bf16_bits_to_f64(wsg_bits)
        gate = 1.0 / (1.0 + np.exp(-s))
    return ids, w, gate, l


def routing_tables(ids, E: int, block_m: int, shared: bool = True) -> dict:
    """Expert-contiguous routing tables built from the chosen expert ids.

    [dothoosh "Prefill optimisations", GPU-resident routing item; droneth, same
    list]: a routing histogram, a prefix scan, a scatter and a block map.
      counts[e]   number of assignments a = t*top_k + k with ids[a] == e;
                  counts[E] = T for the shared expert (every token)
      offsets     exclusive prefix sum of counts, length E + 2
      sorted[p]   the assignment at position p; within one expert, positions
                  follow increasing a (a stable counting sort)
      inv[a]      the position of assignment a (sorted[inv[a]] == a)
      tiles       for e = 0..E in order, ceil(counts[e] / block_m) tiles of at
                  most block_m consecutive positions of one expert:
                  (expert, first position, rows)
    The shared expert's rows are positions A .. A + T - 1 (token t at A + t).
    Returns a dict of int32 numpy arrays and num_tiles."""
    ids = np.asarray(ids, dtype=np.int64)
    T = ids.shape[0]
    flat = ids.reshape(-1)
    A = flat.size
    counts = np.zeros(E + 1, dtype=np.int64)
    for e in flat:                     # histogram
        counts[e] += 1
    if shared:
        counts[E] = T
    offsets = np.zeros(E + 2, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)    # exclusive prefix scan
    sorted_ = np.zeros(A, dtype=np.int64)
    inv = np.zeros(A, dtype=np.int64)
    fill = offsets[:E].copy()
    for a in range(A):                 # stable scatter in assignment order
        e = flat[a]
        sorted_[fill[e]] = a
        inv[a] = fill[e]
        fill[e] += 1
    te, tr0, trows = [], [], []
    for e in range(E + 1):             # block map
        c = counts[e]
        j = 0
        while j * block_m < c:
            te.append(e)
            tr0.append(offsets[e] + j * block_m)
            trows.append(min(block_m, c - j * block_m))
            j += 1
    i32 = lambda v: np.asarray(v, dtype=np.int32)
    return dict(counts=i32(counts), offsets=i32(offsets), sorted=i32(sorted_), inv=i32(inv),
                tile_expert=i32(te), tile_row0=i32(tr0), tile_rows=i32(trows), num_tiles=len(te))


def swiglu_expert(xrows, w_gu, w_dn) -> np.ndarray:
    """One SwiGLU expert on token rows, fp64 end to end.

    Readings where the pages are silent: gate and up projections are the first
    and second halves of the [2I, H] gate_up matrix; h = silu(gate) * up with
    silu(a) = a / (1 + exp(-a)); o = W_down h with W_down [H, I]. The pages fix
    FP32 accumulation for the GPU ([dothoosh "Prefill optimisations"]); the
    oracle keeps every value in fp64, with no intermediate rounding."""
    I = w_gu.shape[0] // 2
    gu = xrows @ w_gu.T
    g, u = gu[:, :I], gu[:, I:]
    h = g / (1.0 + np.exp(-g)) * u
    return h @ w_dn.T


def moe_forward(x_bits, wr_bits, bias, wsg_bits, top_k: int, expert_fn, tokens=None, x_f64=None):
    """The whole layer for the tokens listed (all tokens by default).

    y[t] = sum_k w[t, k] * Expert_{ids[t, k]}(x_t) + g_t * Shared(x_t)
    [dothoosh "Model specification": 8 routed experts plus one shared expert
    for every token]. `expert_fn(e)` returns the packed weights of expert e
    (e == E: the shared expert, or None without one) as
    (gu_codes, gu_scales, gu_biases, dn_codes, dn_scales, dn_biases).
    Each used expert is dequantised once; rows are gathered per expert, the
    way the pages' grouped GEMM groups them, but the arithmetic is the plain
    definition (fp64 sums make the order of the additions immaterial at any
    tolerance the tests use).
    `x_f64`, when given, is the input in fp64 (a normalised residual row,
    see rms_norm) and x_bits is ignored.
    Returns (y fp64 [n, H], ids, weights, gate, logits) for the n tokens."""
    n_all = (np.asarray(x_f64) if x_f64 is not None else np.asarray(x_bits)).shape[0]
    tokens = np.arange(n_all) if tokens is None else np.asarray(tokens)
    if x_f64 is None:
        xs = np.asarray(x_bits)[tokens]
        ids, w, gate, logits = route(xs, wr_bits, bias, wsg_bits, top_k)
        x = bf16_bits_to_f64(xs)
    else:
        x = np.asarray(x_f64, dtype=np.float64)[tokens]
        ids, w, gate, logits = route(None, wr_bits, bias, wsg_bits, top_k, x_f64=x)
    n, H = x.shape
    E = np.asarray(wr_bits).shape[0]
    y = np.zeros((n, H), dtype=np.float64)
    for e in np.unique(ids):
        gu_c, gu_s, gu_b, dn_c, dn_s, dn_b = expert_fn(int(e))
        w_gu = dequant(gu_c, gu_s, gu_b)
        w_dn = dequant(dn_c, dn_s, dn_b)
        rows, ks = np.nonzero(ids == e)
        o = swiglu_expert(x[rows], w_gu, w_dn)
        y[rows] += w[rows, ks][:, None] * o
    if wsg_bits is not None:
        sh = expert_fn(E)
        if sh is not None:
            gu_c, gu_s, gu_b, dn_c, dn_s, dn_b = sh
            o = swiglu_expert(x, dequant(gu_c, gu_s, gu_b), dequant(dn_c, dn_s, dn_b))
            y += gate[:, None] * o
    return y, ids, w, gate, logits
