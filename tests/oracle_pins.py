"""Pins that tie the CPU oracle to something other than itself.

Each pin raises AssertionError when the oracle is wrong. They reach the oracle
through the module object (`M.<function>`) at call time, so that
test_planted_mistakes.py can swap in a mutated function and check that some
pin catches it. Sources of the facts pinned are named in each pin and in the
golden files they read.
"""
from __future__ import annotations

import itertools
import math

import numpy as np

import oracle.attention as A
import oracle.gated_deltanet as G
import oracle.moe as M
from tests._util import bf16_from_f64, read_golden

RNG = np.random.default_rng(20260099)


def _bits(vals):
    return bf16_from_f64(np.asarray(vals, dtype=np.float64))


# ---------------------------------------------------------------- format ---

def pin_dequant_handworked():
    """Hand-worked nibble values (tests/golden/dequant_handworked.txt)."""
    for (word, scale, bias), want in read_golden("dequant_handworked.txt"):
        w = int(word, 16)
        for j in range(8):   # the word at every position of a 64-weight group
            codes = np.zeros((1, 8), dtype=np.uint32)
            codes[0, j] = w
            s = _bits([[float(scale)]])
            b = _bits([[float(bias)]])
            W = M.dequant(codes, s, b)
            assert W.shape == (1, 64)
            got = W[0, 8 * j: 8 * j + 8]
            assert np.array_equal(got, np.array([float(v) for v in want])), (word, j, got, want)
            rest = np.delete(W[0], np.arange(8 * j, 8 * j + 8))
            assert np.all(rest == float(bias)), (word, j)


def pin_dequant_groups():
    """One scale/bias pair per row and per 64 weights along K
    (tests/golden/dequant_groups.txt)."""
    rows = read_golden("dequant_groups.txt")
    codes = np.full((2, 16), 0x33333333, dtype=np.uint32)
    s = np.zeros((2, 2))
    b = np.zeros((2, 2))
    want = np.zeros((2, 2))
    for (r, g, sc, bi), (v,) in rows:
        s[int(r), int(g)] = float(sc)
        b[int(r), int(g)] = float(bi)
        want[int(r), int(g)] = float(v)
    W = M.dequant(codes, _bits(s), _bits(b))
    assert W.shape == (2, 128)
    for r in range(2):
        for g in range(2):
            assert np.all(W[r, 64 * g: 64 * g + 64] == want[r, g]), (r, g)


def pin_checkpoint_bits_per_weight():
    """4-bit codes plus a bf16 scale and a bf16 bias per 64 weights is 4.5 bits
    per weight; 35e9 parameters at 4.5 bits is within 3 % of the 19.4 GB
    checkpoint the pages print, and 70 GB of bf16 is 2 bytes x 35e9
    (tests/golden/checkpoint_format.txt). The byte count comes from the array
    shapes the oracle accepts for one [N, K] matrix."""
    g = {r[0][0]: float(r[0][1]) for r in read_golden("checkpoint_format.txt")}
    N, K = 8, 512
    codes = np.zeros((N, K // 8), dtype=np.uint32)
    s = np.zeros((N, K // 64), dtype=np.uint16)
    b = np.zeros((N, K // 64), dtype=np.uint16)
    W = M.dequant(codes, s, b)
    assert W.shape == (N, K)
    bytes_per_weight = (codes.nbytes + s.nbytes + b.nbytes) / W.size
    assert bytes_per_weight * 8 == 4.5
    assert abs(g["params_total"] * bytes_per_weight - g["q4_bytes"]) / g["q4_bytes"] < 0.03
    assert abs(g["params_total"] * 2 - g["bf16_bytes"]) / g["bf16_bytes"] < 0.01


# ---------------------------------------------------------------- router ---

def _logit_inputs(logits, H=64):
    E = len(logits)
    x = np.zeros((1, H))
    x[0, 0] = 1.0
    wr = np.zeros((E, H))
    wr[:, 0] = logits
    return _bits(x), _bits(wr)


def pin_router_logits_exact():
    """Integer logits through x = e_0 come out exact (no dropped term, no
    transposed operand): l[t, e] = sum_h x[t, h] W_r[e, h] + b[e]."""
    x = np.zeros((3, 64))
    x[0, 0] = 1.0
    x[1, 5] = 2.0
    x[2, :] = 1.0
    wr = np.zeros((4, 64))
    wr[1, 0] = 3.0
    wr[2, 5] = -1.5
    wr[3, :] = 0.25
    b = np.array([0.0, 1.0, 0.0, -2.0], dtype=np.float32)
    l = M.router_logits(_bits(x), _bits(wr), b)
    want = np.array([[0, 3 + 1, 0, 0.25 - 2],
                     [0, 1, -3.0, 0.5 - 2],
                     [0, 3 + 1, -1.5, 16 - 2]])
    assert np.array_equal(l, want), l


def pin_topk_ties_golden():
    """Exact ties resolved toward the lower index (tests/golden/topk_ties.txt)."""
    for (k,), logits, want in read_golden("topk_ties.txt"):
        x, wr = _logit_inputs([float(v) for v in logits])
        ids, w, gate, l = M.route(x, wr, None, None, int(k))
        assert ids.tolist() == [[int(v) for v in want]], (logits, ids, want)


def _rank_topk(l32, k):
    """Brute force: expert e's rank is the number of experts that beat it
    (higher fp32 logit, or equal logit and lower index)."""
    T, E = l32.shape
    out = np.zeros((T, k), dtype=np.int64)
    for t in range(T):
        for e in range(E):
            r = sum(1 for j in range(E) if l32[t, j] > l32[t, e] or (l32[t, j] == l32[t, e] and j < e))
            if r < k:
                out[t, r] = e
    return out


def pin_topk_bruteforce():
    """Top-k against O(E^2) rank counting on random logits, some with ties."""
    for E, k in [(8, 1), (12, 4), (16, 8), (20, 8)]:
        x = RNG.standard_normal((6, 32))
        wr = RNG.standard_normal((E, 32))
        wr[E // 2] = wr[0]          # an exact tie between expert 0 and E/2
        xb, wb = _bits(x), _bits(wr)
        ids, w, gate, l = M.route(xb, wb, None, None, k)
        want = _rank_topk(l.astype(np.float32), k)
        assert np.array_equal(ids, want), (E, k)


def pin_softmax_closed_form():
    """Renormalised softmax: weights sum to 1, ratios are exp(l_i - l_j), and
    the weights do not change when every logit shifts by the same bias."""
    E, k = 16, 8
    x = RNG.standard_normal((5, 32))
    wr = RNG.standard_normal((E, 32)) * 0.3
    xb, wb = _bits(x), _bits(wr)
    ids, w, gate, l = M.route(xb, wb, None, None, k)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-12)
    for t in range(5):
        for i, j in itertools.combinations(range(k), 2):
            want = math.exp(l[t, ids[t, i]] - l[t, ids[t, j]])
            assert abs(w[t, i] / w[t, j] - want) <= 1e-9 * want
    assert np.all(np.diff(w, axis=1) <= 0)
    ids2, w2, _, _ = M.route(xb, wb, np.full(E, 0.75, dtype=np.float32), None, k)
    assert np.array_equal(ids2, ids) and np.allclose(w2, w, rtol=1e-12)
    ids1, w1, _, _ = M.route(xb, wb, None, None, 1)
    assert np.all(w1 == 1.0)


def pin_gate_closed_form():
    """Shared-expert gate: sigmoid of x . w_sg; 1/2 at 0, 3/4 at ln 3."""
    x = np.zeros((2, 64))
    x[0, 0] = 1.0
    x[1, 3] = 1.0
    wsg = np.zeros(64)
    wsg[3] = 1.1015625             # bf16(ln 3), 3e-3 above ln 3
    ids, w, g, l = M.route(_bits(x), _bits(np.ones((8, 64))), None, _bits(wsg), 8)
    assert g[0] == 0.5
    assert abs(g[1] - 0.75) < 1e-3     # slope 3/16 times the 3e-3 offset


# --------------------------------------------------------------- routing ---

def check_routing_invariants(ids, E, bm, tab, shared=True):
    """Properties every correct routing table has (shared with the GPU tests)."""
    ids = np.asarray(ids)
    T, K = ids.shape
    A = T * K
    c, off = tab["counts"], tab["offsets"]
    assert c[:E].sum() == A
    assert (not shared) or c[E] == T
    assert off[0] == 0 and np.array_equal(np.diff(off), c)
    srt, inv = tab["sorted"], tab["inv"]
    assert np.array_equal(np.sort(srt), np.arange(A))
    assert np.array_equal(srt[inv], np.arange(A)) and np.array_equal(inv[srt], np.arange(A))
    flat = ids.reshape(-1)
    for e in range(E):
        seg = srt[off[e]:off[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)
    n = tab["num_tiles"]
    te, tr0, tr = tab["tile_expert"][:n], tab["tile_row0"][:n], tab["tile_rows"][:n]
    want_tiles = sum(-(-int(c[e]) // bm) for e in range(E + 1))
    assert n == want_tiles
    covered = np.zeros(A + (T if shared else 0), dtype=np.int64)
    for e, r0, r in zip(te, tr0, tr):
        assert 1 <= r <= bm
        assert off[e] <= r0 and r0 + r <= off[e + 1]
        covered[r0:r0 + r] += 1
    assert np.all(covered == 1)
    assert np.all(np.diff(te) >= 0)


def pin_routing_invariants():
    for T, E, K, bm in [(1, 8, 8, 16), (7, 16, 4, 4), (64, 256, 8, 16), (33, 256, 8, 128), (100, 32, 8, 32)]:
        ids = np.stack([RNG.permutation(E)[:K] for _ in range(T)])
        tab = M.routing_tables(ids, E, bm)
        check_routing_invariants(ids, E, bm, tab)


def pin_routing_bruteforce():
    """Positions by their definition: pos(a) = offsets[e] + #{a' < a with the
    same expert}; offsets[e] = #{assignments with a lower expert}."""
    T, E, K, bm = 9, 12, 3, 4
    ids = np.stack([RNG.permutation(E)[:K] for _ in range(T)])
    tab = M.routing_tables(ids, E, bm)
    flat = ids.reshape(-1)
    for a in range(flat.size):
        e = flat[a]
        want = int((flat < e).sum() + (flat[:a] == e).sum())
        assert tab["inv"][a] == want, (a, tab["inv"][a], want)
    assert tab["offsets"][E] == T * K and tab["offsets"][E + 1] == T * K + T


# ------------------------------------------------------------ whole layer ---

def _const_layer(E, H, I, consts):
    """Experts whose weights are constants: scale 0, bias c_gate on the gate
    rows, c_up on the up rows, c_down on the down matrix."""
    def fn(e):
        cg, cu, cd = consts[e]
        gu_c = RNG.integers(0, 2 ** 32, size=(2 * I, H // 8), dtype=np.uint32)
        dn_c = RNG.integers(0, 2 ** 32, size=(H, I // 8), dtype=np.uint32)
        z_gu = _bits(np.zeros((2 * I, H // 64)))
        b_gu = np.zeros((2 * I, H // 64))
        b_gu[:I] = cg
        b_gu[I:] = cu
        return (gu_c, z_gu, _bits(b_gu), dn_c, _bits(np.zeros((H, I // 64))), _bits(np.full((H, I // 64), cd)))
    return fn


def pin_layer_constant_weights():
    """Constant weights reduce the layer to a closed form. With S_t = sum_h x[t,h]
    and expert e's constants (g_e, u_e, d_e): h = silu(g_e S_t) * u_e S_t on every
    column, o = d_e * I * h on every output, so
    y_t = sum_k w_tk d_e I silu(g_e S) u_e S + gate_t d_s I silu(g_s S) u_s S."""
    E, H, I, K, T = 12, 128, 64, 4, 5
    consts = {e: (0.25 * (e % 3 - 1) + 0.125, 0.5 - 0.0625 * e, 0.015625 * (e + 1)) for e in range(E + 1)}
    x = RNG.standard_normal((T, H))
    xb = _bits(x)
    xv = M.bf16_bits_to_f64(xb)
    wr = _bits(RNG.standard_normal((E, H)) * 0.2)
    wsg = _bits(RNG.standard_normal(H) * 0.1)
    y, ids, w, gate, l = M.moe_forward(xb, wr, None, wsg, K, _const_layer(E, H, I, consts))
    silu = lambda a: a / (1.0 + math.exp(-a))
    for t in range(T):
        S = xv[t].sum()
        want = 0.0
        for k in range(K):
            g_, u_, d_ = consts[int(ids[t, k])]
            want += w[t, k] * d_ * I * silu(g_ * S) * u_ * S
        g_, u_, d_ = consts[E]
        sgate = 1.0 / (1.0 + math.exp(-float(xv[t] @ M.bf16_bits_to_f64(wsg))))
        want += sgate * d_ * I * silu(g_ * S) * u_ * S
        assert np.allclose(y[t], want, rtol=1e-12, atol=1e-12), (t, y[t, :3], want)


def pin_silu_values():
    """silu at hand-known points through a one-weight expert (gate row = a,
    up row = 1, down = 1, so o = silu(a)): 0 at 0; 3/4 * a at a = ln 3, where
    the sigmoid is exactly 3/4 (a is bf16(ln 3), 2e-5 away, which moves the
    value by < 1e-5); about a at a = 20 and about 0 at a = -20."""
    H = I = 64
    a3 = 1.0986328125                   # bf16(ln 3)
    for a, want, tol in [(0.0, 0.0, 0.0), (a3, 0.75 * a3, 1e-5), (20.0, 20.0, 1e-6), (-20.0, 0.0, 1e-6)]:
        w_gu = np.zeros((2 * I, H))
        w_gu[0, 0] = a
        w_gu[I, 0] = 1.0
        w_dn = np.zeros((H, I))
        w_dn[0, 0] = 1.0
        x = np.zeros((1, H))
        x[0, 0] = 1.0
        o = M.swiglu_expert(x, w_gu, w_dn)
        assert abs(o[0, 0] - want) <= tol, (a, o[0, 0], want)
        assert np.all(o[0, 1:] == 0)


def pin_down_projection_orientation():
    """o = W_down h with W_down stored output-major [H, I]: with x = e_0, one
    gate weight of 20 (silu(20) = 20 to 1e-8) and one up weight of 1, h has a
    single non-zero h_0 = 20, so o_m = 20 * W_down[m, 0] exactly picks column 0.
    Row 0 of W_down holds other values that a transposed use would pick."""
    H = I = 64
    w_gu = np.zeros((2 * I, H))
    w_gu[0, 0] = 20.0
    w_gu[I, 0] = 1.0
    w_dn = np.zeros((H, I))
    w_dn[:, 0] = (np.arange(H) + 1) / 64.0
    w_dn[0, 1:] = 5.0
    x = np.zeros((1, H))
    x[0, 0] = 1.0
    o = M.swiglu_expert(x, w_gu, w_dn)
    want = 20.0 * (np.arange(H) + 1) / 64.0
    assert np.allclose(o[0], want, rtol=1e-7, atol=0), o[0, :4]


def _dense_reference(xb, wr, bias, wsg, K, fn, E):
    """Every expert on every token, masked by the brute-force top-k ranks and
    weighted by a softmax over the masked set."""
    x = M.bf16_bits_to_f64(xb)
    l = M.router_logits(xb, wr, bias)
    top = _rank_topk(l.astype(np.float32), K)
    T = x.shape[0]
    y = np.zeros_like(x)
    outs = {}
    for e in range(E):
        c = fn(e)
        outs[e] = M.swiglu_expert(x, M.dequant(*c[:3]), M.dequant(*c[3:]))
    for t in range(T):
        mask = np.zeros(E, dtype=bool)
        mask[top[t]] = True
        z = np.where(mask, np.exp(l[t] - l[t].max()), 0.0)
        wt = z / z.sum()
        for e in range(E):
            if mask[e]:
                y[t] += wt[e] * outs[e][t]
    if wsg is not None:
        c = fn(E)
        gate = 1.0 / (1.0 + np.exp(-(x @ M.bf16_bits_to_f64(wsg))))
        y += gate[:, None] * M.swiglu_expert(x, M.dequant(*c[:3]), M.dequant(*c[3:]))
    return y


def _random_layer(E, H, I):
    cache = {}

    def fn(e):
        if e not in cache:
            s_gu = np.abs(RNG.standard_normal((2 * I, H // 64))) * 0.02
            s_dn = np.abs(RNG.standard_normal((H, I // 64))) * 0.02
            cache[e] = (RNG.integers(0, 2 ** 32, size=(2 * I, H // 8), dtype=np.uint32), _bits(s_gu),
                        _bits(-8 * s_gu + 1e-3 * RNG.standard_normal(s_gu.shape)),
                        RNG.integers(0, 2 ** 32, size=(H, I // 8), dtype=np.uint32), _bits(s_dn),
                        _bits(-8 * s_dn + 1e-3 * RNG.standard_normal(s_dn.shape)))
        return cache[e]
    return fn


def pin_layer_dense_masked():
    """The routed layer equals the dense all-experts masked mixture."""
    E, H, I, K, T = 16, 128, 64, 4, 12
    fn = _random_layer(E, H, I)
    xb = _bits(RNG.standard_normal((T, H)))
    wr = _bits(RNG.standard_normal((E, H)) / math.sqrt(H))
    wsg = _bits(RNG.standard_normal(H) / math.sqrt(H))
    bias = (RNG.standard_normal(E) * 0.5).astype(np.float32)
    y, *_ = M.moe_forward(xb, wr, bias, wsg, K, fn)
    want = _dense_reference(xb, wr, bias, wsg, K, fn, E)
    assert np.allclose(y, want, rtol=1e-10, atol=1e-12)
    # the same layer evaluated for a subset of tokens gives the same rows
    sub = np.array([3, 0, 11])
    ys, *_ = M.moe_forward(xb, wr, bias, wsg, K, fn, tokens=sub)
    assert np.allclose(ys, y[sub], rtol=1e-12, atol=1e-14)


def pin_layer_all_experts():
    """top_k = E: the layer is the dense softmax mixture of every expert."""
    E, H, I, T = 8, 64, 64, 4
    fn = _random_layer(E, H, I)
    xb = _bits(RNG.standard_normal((T, H)))
    wr = _bits(RNG.standard_normal((E, H)) / math.sqrt(H))
    y, ids, w, g, l = M.moe_forward(xb, wr, None, None, E, fn)
    x = M.bf16_bits_to_f64(xb)
    p = np.exp(l - l.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    want = np.zeros_like(x)
    for e in range(E):
        c = fn(e)
        want += p[:, e:e + 1] * M.swiglu_expert(x, M.dequant(*c[:3]), M.dequant(*c[3:]))
    assert np.allclose(y, want, rtol=1e-10, atol=1e-12)


# ------------------------------------------------------ pre-norm residual ---

def pin_rms_norm_handworked():
    """Hand-worked rows: [1, 7] has mean square 25, so its RMS is 5 and the
    normalised row [0.2, 1.4]; a row of ones with eps = 3 divides by
    sqrt(1 + 3) = 2; a row of +-2 becomes +-1 (eps negligible)."""
    x = M.rms_norm(_bits([[1.0, 7.0]]), 1e-30)
    assert np.allclose(x, [[0.2, 1.4]], rtol=1e-14, atol=0)
    x = M.rms_norm(_bits([[1.0, 1.0, 1.0, 1.0]]), 3.0)
    assert np.allclose(x, [[0.5] * 4], rtol=1e-14, atol=0)
    r = np.array([[-2.0, 2.0, 2.0, -2.0, 2.0, 2.0, 2.0, 2.0]])
    assert np.allclose(M.rms_norm(_bits(r), 1e-30), r / 2, rtol=1e-14, atol=0)


def pin_rms_norm_invariants():
    """The output's mean square is 1 (eps negligible), scaling the row by a
    power of two changes nothing, and the gain multiplies each channel."""
    r = RNG.standard_normal((5, 96)) * 3
    x = M.rms_norm(_bits(r), 1e-30)
    assert np.allclose(np.mean(x * x, axis=1), 1.0, rtol=1e-12)
    assert np.allclose(M.rms_norm(_bits(r * 8), 1e-30), x, rtol=1e-12)
    gain = np.where(np.arange(96) % 2 == 0, 2.0, 0.5)
    assert np.allclose(M.rms_norm(_bits(r), 1e-30, _bits(gain)), x * gain[None, :], rtol=1e-12)


# -------------------------------------------------------- decode attention ---

def _attn(q, k, v, lens, scale=None):
    return A.gqa_decode_attention(_bits(q), _bits(k), _bits(v), lens, scale)


def pin_attn_single_position():
    """One cached position: the softmax weight is 1 and o = v_0 for every
    query head, whatever q is."""
    B, Hq, Hkv, D, L = 2, 4, 2, 16, 5
    q = RNG.standard_normal((B, Hq, D)) * 3
    k = RNG.standard_normal((B, Hkv, L, D))
    v = RNG.standard_normal((B, Hkv, L, D))
    vb = M.bf16_bits_to_f64(_bits(v))
    o = _attn(q, k, v, [1, 1])
    for b in range(B):
        for h in range(Hq):
            assert np.array_equal(o[b, h], vb[b, h // 2, 0]), (b, h)


def pin_attn_two_positions_closed_form():
    """Two positions whose scores differ by d = 1 (q = e_0, k_0 = 2 e_0,
    k_1 = 0, D = 4, default scale 1/2): weights sigmoid(1) and 1 - sigmoid(1)."""
    D = 4
    q = np.zeros((1, 1, D)); q[0, 0, 0] = 1.0
    k = np.zeros((1, 1, 2, D)); k[0, 0, 0, 0] = 2.0
    v = np.zeros((1, 1, 2, D)); v[0, 0, 0, 0] = 1.0; v[0, 0, 1, 1] = 1.0
    o = _attn(q, k, v, [2])
    sig = 1.0 / (1.0 + math.exp(-1.0))
    assert abs(o[0, 0, 0] - 0.7310585786300049) < 1e-15 and abs(sig - 0.7310585786300049) < 1e-15
    assert abs(o[0, 0, 1] - 0.2689414213699951) < 1e-15
    assert o[0, 0, 2] == 0 and o[0, 0, 3] == 0


def pin_attn_equal_keys_mean():
    """Identical keys (or q = 0) make every weight 1/n: o is the mean of the
    first n value rows."""
    B, Hq, Hkv, D, L = 1, 2, 1, 8, 9
    row = RNG.standard_normal(D)
    k = np.tile(row, (B, Hkv, L, 1))
    v = RNG.standard_normal((B, Hkv, L, D))
    q = RNG.standard_normal((B, Hq, D))
    vb = M.bf16_bits_to_f64(_bits(v))
    for n in (1, 4, 9):
        o = _attn(q, k, v, [n])
        assert np.allclose(o[0, 0], vb[0, 0, :n].mean(axis=0), rtol=0, atol=1e-13), n
    k2 = RNG.standard_normal((B, Hkv, L, D))
    o = _attn(np.zeros((B, Hq, D)), k2, v, [L])
    assert np.allclose(o[0, 1], vb[0, 0].mean(axis=0), rtol=0, atol=1e-13)


def pin_attn_head_mapping():
    """Query head h reads KV head h // (Hq/Hkv): with V of KV head g all equal
    to g + 1, every output element of head h is h // (Hq/Hkv) + 1."""
    B, Hq, Hkv, D, L = 1, 8, 2, 8, 6
    q = RNG.standard_normal((B, Hq, D))
    k = RNG.standard_normal((B, Hkv, L, D))
    v = np.zeros((B, Hkv, L, D))
    for g in range(Hkv):
        v[0, g] = g + 1
    o = _attn(q, k, v, [L])
    for h in range(Hq):
        assert np.allclose(o[0, h], h // 4 + 1, rtol=0, atol=1e-14), h


def pin_attn_masks_past_length():
    """Rows at or past lens[b] do not matter: poisoning them (large values in K
    and V) leaves o unchanged, and o equals the result on the truncated cache."""
    B, Hq, Hkv, D, L = 3, 4, 2, 16, 12
    q = RNG.standard_normal((B, Hq, D))
    k = RNG.standard_normal((B, Hkv, L, D))
    v = RNG.standard_normal((B, Hkv, L, D))
    lens = [5, 12, 0]
    o = _attn(q, k, v, lens)
    k2, v2 = k.copy(), v.copy()
    for b, n in enumerate(lens):
        k2[b, :, n:] = 1e4
        v2[b, :, n:] = -3e4
    assert np.array_equal(_attn(q, k2, v2, lens), o)
    assert np.array_equal(_attn(q[:1], k[:1, :, :5], v[:1, :, :5], [5]), o[:1])
    assert np.all(o[2] == 0)


def pin_attn_invariances():
    """Permuting cache positions (keys and values together) and adding one
    vector to every key (every score shifts by the same q . c) leave o
    unchanged; scaling every value by 2 doubles o."""
    B, Hq, Hkv, D, L = 1, 4, 1, 8, 10
    q = RNG.standard_normal((B, Hq, D))
    k = RNG.standard_normal((B, Hkv, L, D))
    v = RNG.standard_normal((B, Hkv, L, D))
    o = _attn(q, k, v, [L])
    perm = RNG.permutation(L)
    assert np.allclose(_attn(q, k[:, :, perm], v[:, :, perm], [L]), o, rtol=0, atol=1e-13)
    c = np.round(RNG.standard_normal(D) * 4) / 4   # exact in bf16 sums with the keys below
    kq = np.round(k * 8) / 8
    assert np.allclose(_attn(q, kq + c, v, [L]), _attn(q, kq, v, [L]), rtol=0, atol=1e-12)
    assert np.allclose(_attn(q, k, 2 * v, [L]), 2 * o, rtol=0, atol=1e-13)


def pin_attn_peaked_limit():
    """Scores hundreds apart put all the weight on the best position: with
    q = 64 e_0 and key j = j e_0 (scale 1/2, D = 4) the scores are 32 j, so
    o = v at the last position to fp64 precision (the others weigh at most
    e^-32), and nothing overflows even though exp(32 (L-1)) would."""
    D, L = 4, 40
    q = np.zeros((1, 1, D)); q[0, 0, 0] = 64.0
    k = np.zeros((1, 1, L, D)); k[0, 0, :, 0] = np.arange(L)
    v = RNG.standard_normal((1, 1, L, D))
    o = _attn(q, k, v, [L])
    vb = M.bf16_bits_to_f64(_bits(v))
    assert np.all(np.isfinite(o))
    assert np.allclose(o[0, 0], vb[0, 0, L - 1], rtol=0, atol=1e-12)


def pin_attn_matches_torch_sdpa():
    """Full caches reduce the oracle to torch's scaled_dot_product_attention
    (fp64, one query position, enable_gqa), an independent library routine, at
    the default scale and at an explicit one."""
    import torch
    B, Hq, Hkv, D, L = 2, 8, 2, 32, 17
    q = M.bf16_bits_to_f64(_bits(RNG.standard_normal((B, Hq, D)) * 2))
    k = M.bf16_bits_to_f64(_bits(RNG.standard_normal((B, Hkv, L, D))))
    v = M.bf16_bits_to_f64(_bits(RNG.standard_normal((B, Hkv, L, D))))
    for scale in (None, 0.3):
        want = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q)[:, :, None, :], torch.from_numpy(k), torch.from_numpy(v),
            scale=scale, enable_gqa=True)[:, :, 0, :].numpy()
        got = _attn(q, k, v, [L, L], scale)
        assert np.allclose(got, want, rtol=0, atol=1e-12), scale


# ---------------------------------------------------------- Gated DeltaNet ---

def _gdn(q, k, v, gate, beta, S0, offsets):
    return G.gated_delta_scan(_bits(q), _bits(k), _bits(v), gate, beta, S0, offsets)


# The closed forms below hold for unit keys; the eps inside the normalisation
# (|k^|^2 = |k|^2 / (|k|^2 + 1e-6)) moves results by about 1e-6 of the terms'
# size, hence the absolute tolerance of 1e-5 (the planted mistakes move them
# by 1e-1 and more).
def _gdn_case(T, Hqk=2, Hv=4, Dk=8, Dv=8, B=1):
    q = RNG.standard_normal((T, Hqk, Dk))
    k = RNG.standard_normal((T, Hqk, Dk))
    v = RNG.standard_normal((T, Hv, Dv))
    gate = -RNG.uniform(0.0, 0.5, (T, Hv))
    beta = RNG.uniform(0.1, 0.9, (T, Hv))
    S0 = RNG.standard_normal((B, Hv, Dv, Dk))
    return q, k, v, gate, beta, S0


def pin_gdn_full_write_is_retrieved():
    """With beta = 1 and no decay, one step writes v under the unit key k^:
    S_t k^ = v whatever S_{t-1} was, so q = k reads back v / sqrt(Dk)."""
    T, Dk = 5, 16
    q, k, v, gate, beta, S0 = _gdn_case(T, Dk=Dk, Dv=8)
    gate[:] = 0.0
    beta[:] = 1.0
    o, _ = _gdn(k, k, v, gate, beta, S0, [0, T])
    vb = M.bf16_bits_to_f64(_bits(v))
    assert np.allclose(o, vb / math.sqrt(Dk), rtol=1e-5, atol=1e-6)


def pin_gdn_orthonormal_keys_are_linear_attention():
    """From S_0 = 0 with no decay and orthonormal keys e_t the writes do not
    interfere: o_t = sum_{s<=t} beta_s v_s (q^_t)_s, q^ the unit q / sqrt(Dk)."""
    T, Dk, Dv = 6, 8, 4
    q, k, v, gate, beta, S0 = _gdn_case(T, Hqk=1, Hv=1, Dk=Dk, Dv=Dv)
    k[:] = 0.0
    for t in range(T):
        k[t, 0, t] = 1.0
    gate[:] = 0.0
    S0[:] = 0.0
    o, S = _gdn(q, k, v, gate, beta, S0, [0, T])
    qb = M.bf16_bits_to_f64(_bits(q))[:, 0]
    vb = M.bf16_bits_to_f64(_bits(v))[:, 0]
    for t in range(T):
        qh = qb[t] / np.linalg.norm(qb[t]) / math.sqrt(Dk)
        want = sum(beta[s, 0] * vb[s] * qh[s] for s in range(t + 1))
        assert np.allclose(o[t, 0], want, rtol=1e-5, atol=1e-5), t
    assert np.allclose(S[0, 0][:, :T], (beta[:, 0][None, :] * vb.T), rtol=1e-5, atol=1e-5)


def pin_gdn_orthonormal_keys_with_decay():
    """Orthonormal keys e_t from S_0 = 0 with decay: each write decays from the
    step after it, o_t = sum_{s<=t} (prod_{s<r<=t} alpha_r) beta_s v_s (q^_t)_s."""
    T, Dk, Dv = 5, 8, 3
    q, k, v, gate, beta, S0 = _gdn_case(T, Hqk=1, Hv=1, Dk=Dk, Dv=Dv)
    k[:] = 0.0
    for t in range(T):
        k[t, 0, t] = 1.0
    S0[:] = 0.0
    o, _ = _gdn(q, k, v, gate, beta, S0, [0, T])
    qb = M.bf16_bits_to_f64(_bits(q))[:, 0]
    vb = M.bf16_bits_to_f64(_bits(v))[:, 0]
    for t in range(T):
        qh = qb[t] / np.linalg.norm(qb[t]) / math.sqrt(Dk)
        want = sum(math.exp(gate[s + 1:t + 1, 0].sum()) * beta[s, 0] * vb[s] * qh[s] for s in range(t + 1))
        assert np.allclose(o[t, 0], want, rtol=1e-5, atol=1e-5), t


def pin_gdn_same_key_twice():
    """Writing under the same unit key twice, from S_0 = 0: the second step's
    delta is taken against the decayed state, so the memory then holds
    alpha (1 - beta) v_0 + beta v_1 under that key (beta_0 = 1)."""
    Dk, Dv = 8, 4
    q, k, v, gate, beta, S0 = _gdn_case(2, Hqk=1, Hv=1, Dk=Dk, Dv=Dv)
    k[:] = 0.0
    k[:, 0, 3] = 1.0
    q[:] = k
    S0[:] = 0.0
    gate[0, 0] = 0.0
    beta[0, 0] = 1.0
    o, S = _gdn(q, k, v, gate, beta, S0, [0, 2])
    vb = M.bf16_bits_to_f64(_bits(v))[:, 0]
    a, bt = math.exp(gate[1, 0]), beta[1, 0]
    held = a * (1 - bt) * vb[0] + bt * vb[1]
    assert np.allclose(S[0, 0][:, 3], held, rtol=1e-5, atol=1e-5)
    assert np.allclose(o[1, 0], held / math.sqrt(Dk), rtol=1e-5, atol=1e-5)


def pin_gdn_pure_decay():
    """beta = 0: no writes, the state only decays: S_t = prod alpha_s S_0 and
    o_t = (prod_{s<=t} alpha_s) S_0 q^_t."""
    T, Dk = 4, 8
    q, k, v, gate, beta, S0 = _gdn_case(T, Hqk=1, Hv=2, Dk=Dk, Dv=6)
    beta[:] = 0.0
    o, S = _gdn(q, k, v, gate, beta, S0, [0, T])
    qb = M.bf16_bits_to_f64(_bits(q))[:, 0]
    for h in range(2):
        decay = np.exp(np.cumsum(gate[:, h]))
        for t in range(T):
            qh = qb[t] / np.linalg.norm(qb[t]) / math.sqrt(Dk)
            assert np.allclose(o[t, h], decay[t] * (S0[0, h] @ qh), rtol=1e-6, atol=1e-9)
        assert np.allclose(S[0, h], decay[-1] * S0[0, h], rtol=1e-12)


def pin_gdn_head_grouping():
    """Value head h reads query/key head h // (Hv/Hqk): key head 0 has q = k
    (reads back v / sqrt(Dk) after a full write), key head 1 has q orthogonal
    to k (reads 0); value heads 0, 1 follow key head 0, heads 2, 3 key head 1."""
    Dk = 8
    q, k, v, gate, beta, S0 = _gdn_case(1, Hqk=2, Hv=4, Dk=Dk, Dv=4)
    k[0, 0] = 0.0
    k[0, 0, 0] = 1.0
    q[0, 0] = k[0, 0]
    k[0, 1] = 0.0
    k[0, 1, 1] = 1.0
    q[0, 1] = 0.0
    q[0, 1, 2] = 1.0
    gate[:] = 0.0
    beta[:] = 1.0
    S0[:] = 0.0
    o, _ = _gdn(q, k, v, gate, beta, S0, [0, 1])
    vb = M.bf16_bits_to_f64(_bits(v))
    for h in (0, 1):
        assert np.allclose(o[0, h], vb[0, h] / math.sqrt(Dk), rtol=1e-5)
    for h in (2, 3):
        assert np.allclose(o[0, h], 0.0, atol=1e-12)


def pin_gdn_scale_of_q_and_k_does_not_matter():
    """q and k enter only through their directions (L2-normalised)."""
    q, k, v, gate, beta, S0 = _gdn_case(7)
    o, S = _gdn(q, k, v, gate, beta, S0, [0, 7])
    o2, S2 = _gdn(4.0 * q, 0.25 * k, v, gate, beta, S0, [0, 7])
    # equal up to the eps inside the normalisation (1e-6 against |k|^2 ~ 1)
    assert np.allclose(o2, o, rtol=1e-5, atol=1e-5)
    assert np.allclose(S2, S, rtol=1e-5, atol=1e-5)


def pin_gdn_split_and_packing():
    """A sequence run in one call equals the same tokens in two calls that
    pass the state on; packing three sequences (one empty) in one call equals
    three separate calls (no state leaks across a sequence boundary)."""
    T = 9
    q, k, v, gate, beta, S0 = _gdn_case(T, B=1)
    o, S = _gdn(q, k, v, gate, beta, S0, [0, T])
    o1, S1 = _gdn(q[:4], k[:4], v[:4], gate[:4], beta[:4], S0, [0, 4])
    o2, S2 = _gdn(q[4:], k[4:], v[4:], gate[4:], beta[4:], S1, [0, T - 4])
    assert np.array_equal(np.concatenate([o1, o2]), o) and np.array_equal(S2, S)
    S03 = RNG.standard_normal((3, 4, 8, 8))
    offs = [0, 3, 3, T]
    op, Sp = _gdn(q, k, v, gate, beta, S03, offs)
    for b in range(3):
        lo, hi = offs[b], offs[b + 1]
        ob, Sb = _gdn(q[lo:hi], k[lo:hi], v[lo:hi], gate[lo:hi], beta[lo:hi], S03[b:b + 1], [0, hi - lo])
        assert np.array_equal(op[lo:hi], ob) and np.array_equal(Sp[b], Sb[0])
    assert np.array_equal(Sp[1], S03[1])


def _gdn_chunkwise(q, k, v, gate, beta, S0, chunk):
    """The same recurrence by the paper's chunkwise form, one value head with
    its key head: within a chunk with cumulative decay g_i = prod_{j<=i} alpha_j
    the state is S_i = g_i S_0 + sum_{l<=i} (g_i / g_l) u_l k^_l^T, where the
    pseudo-values u solve the unit lower-triangular system
        u_j + beta_j sum_{l<j} (g_j / g_l) (k^_l . k^_j) u_l = beta_j (v_j - g_j S_0 k^_j),
    and o_i = S_i q^_i. A different algebra from the token loop (a triangular
    solve and matrix products), written from the formula, not from the oracle."""
    import scipy.linalg
    T, Dk = k.shape
    kh = k / np.sqrt((k * k).sum(axis=1, keepdims=True) + 1e-6)
    qh = q / np.sqrt((q * q).sum(axis=1, keepdims=True) + 1e-6) / math.sqrt(Dk)
    S = S0.copy()
    o = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, chunk):
        sl = slice(c0, min(T, c0 + chunk))
        K, Q, V = kh[sl], qh[sl], v[sl]
        g = np.exp(np.cumsum(gate[sl]))
        ratio = g[:, None] / g[None, :]
        n = K.shape[0]
        low = np.tril(np.ones((n, n)), -1)
        A = np.eye(n) + beta[sl][:, None] * ratio * (K @ K.T) * low
        rhs = beta[sl][:, None] * (V - g[:, None] * (K @ S.T))
        U = scipy.linalg.solve_triangular(A, rhs, lower=True, unit_diagonal=True)
        incl = np.tril(np.ones((n, n)))
        o[sl] = g[:, None] * (Q @ S.T) + ((ratio * incl) * (Q @ K.T)) @ U
        S = g[-1] * S + (U * (g[-1] / g)[:, None]).T @ K
    return o, S


def pin_gdn_chunkwise_form_agrees():
    """The token-by-token oracle equals the chunkwise (triangular-solve) form
    of the gated delta rule, for chunks of 1, 4 and 7 tokens over 23 tokens."""
    T = 23
    q, k, v, gate, beta, S0 = _gdn_case(T, Hqk=1, Hv=1, Dk=8, Dv=6)
    o, S = _gdn(q, k, v, gate, beta, S0, [0, T])
    qb, kb, vb = (M.bf16_bits_to_f64(_bits(x)) for x in (q, k, v))
    for chunk in (1, 4, 7):
        oc, Sc = _gdn_chunkwise(qb[:, 0], kb[:, 0], vb[:, 0], gate[:, 0], beta[:, 0], S0[0, 0], chunk)
        assert np.allclose(oc, o[:, 0], rtol=1e-9, atol=1e-11), chunk
        assert np.allclose(Sc, S[0, 0], rtol=1e-9, atol=1e-11), chunk


PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
