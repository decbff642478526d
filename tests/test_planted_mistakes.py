"""Plants plausible mistakes in the CPU oracle (on the CPU, by swapping one of
its functions for a mutated copy) and checks that at least one pin fails for
each: the pins are sensitive to dropped terms, wrong signs, wrong indices and
transposed operands, not only to crashes."""
import numpy as np
import pytest

import oracle.attention as A
import oracle.gated_deltanet as G
import oracle.moe as M
from tests.oracle_pins import PINS

_dequant = M.dequant
_route = M.route
_routing = M.routing_tables
_swiglu = M.swiglu_expert
_select = M.select_top_k
_logits = M.router_logits
_rms = M.rms_norm


def nibble_order_reversed(codes, scales, biases, group=64):
    c = np.asarray(codes).view(np.uint32)
    N, KW = c.shape
    sh = 4 * (7 - np.arange(8, dtype=np.uint32))
    q = ((c[:, :, None] >> sh[None, None, :]) & np.uint32(15)).reshape(N, KW * 8).astype(np.float64)
    s = np.repeat(M.bf16_bits_to_f64(scales), group, axis=1)
    b = np.repeat(M.bf16_bits_to_f64(biases), group, axis=1)
    return s * q + b


def bias_subtracted(codes, scales, biases, group=64):
    W0 = _dequant(codes, scales, np.zeros_like(np.asarray(biases)), group)
    return W0 - np.repeat(M.bf16_bits_to_f64(biases), group, axis=1)


def signed_codes(codes, scales, biases, group=64):
    W = _dequant(codes, scales, biases, group)
    q = (W - np.repeat(M.bf16_bits_to_f64(biases), group, axis=1))
    s = np.repeat(M.bf16_bits_to_f64(scales), group, axis=1)
    with np.errstate(invalid="ignore", divide="ignore"):
        qq = np.where(s != 0, np.rint(q / np.where(s != 0, s, 1)), 0)
    qq = np.where(qq >= 8, qq - 16, qq)
    return s * qq + np.repeat(M.bf16_bits_to_f64(biases), group, axis=1)


def scale_per_group_of_32(codes, scales, biases, group=64):
    return _dequant(codes, np.repeat(scales, 2, axis=1)[:, : np.asarray(scales).shape[1]], biases, group)


def ties_to_higher_index(logits, top_k):
    l32 = np.asarray(logits).astype(np.float32)
    E = l32.shape[1]
    order = np.argsort(-l32[:, ::-1], axis=1, kind="stable")
    return (E - 1 - order[:, :top_k]).astype(np.int32)


def logits_transposed_bias(x, wr, bias=None):
    l = _logits(x, wr, None)
    if bias is not None:
        l = l - np.asarray(bias, dtype=np.float64)[None, :]
    return l


def no_renormalisation(x, wr, bias, wsg, top_k, **kw):
    ids, w, g, l = _route(x, wr, bias, wsg, top_k, **kw)
    p = np.exp(l - l.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    return ids, np.take_along_axis(p, ids.astype(np.int64), axis=1), g, l


def gate_is_one_minus_sigmoid(x, wr, bias, wsg, top_k, **kw):
    ids, w, g, l = _route(x, wr, bias, wsg, top_k, **kw)
    return ids, w, (None if g is None else 1.0 - g), l


def scatter_reversed_within_expert(ids, E, block_m, shared=True):
    tab = _routing(ids, E, block_m, shared)
    off, srt = tab["offsets"], tab["sorted"].copy()
    for e in range(E):
        srt[off[e]:off[e + 1]] = srt[off[e]:off[e + 1]][::-1]
    inv = np.zeros_like(srt)
    inv[srt] = np.arange(srt.size, dtype=srt.dtype)
    return dict(tab, sorted=srt, inv=inv)


def tiles_off_by_one(ids, E, block_m, shared=True):
    tab = _routing(ids, E, block_m, shared)
    return dict(tab, tile_rows=np.minimum(tab["tile_rows"] + 1, block_m + 1))


def offsets_inclusive(ids, E, block_m, shared=True):
    tab = _routing(ids, E, block_m, shared)
    off = tab["offsets"].copy()
    off[:-1] = off[1:]
    return dict(tab, offsets=off)


def gate_up_swapped(xrows, w_gu, w_dn):
    I = w_gu.shape[0] // 2
    return _swiglu(xrows, np.concatenate([w_gu[I:], w_gu[:I]]), w_dn)


def relu_instead_of_silu(xrows, w_gu, w_dn):
    I = w_gu.shape[0] // 2
    gu = xrows @ w_gu.T
    return (np.maximum(gu[:, :I], 0) * gu[:, I:]) @ w_dn.T


def down_transposed(xrows, w_gu, w_dn):
    I = w_gu.shape[0] // 2
    gu = xrows @ w_gu.T
    h = gu[:, :I] / (1 + np.exp(-gu[:, :I])) * gu[:, I:]
    H = w_dn.shape[0]
    return h @ (w_dn if H == I else w_dn.reshape(I, H))


def rms_sum_not_mean(r_bits, eps, gain_bits=None):
    r = M.bf16_bits_to_f64(r_bits)
    x = r / np.sqrt(np.sum(r * r, axis=1, keepdims=True) + eps)
    return x if gain_bits is None else x * M.bf16_bits_to_f64(gain_bits)[None, :]


def rms_without_sqrt(r_bits, eps, gain_bits=None):
    r = M.bf16_bits_to_f64(r_bits)
    x = r / (np.mean(r * r, axis=1, keepdims=True) + eps)
    return x if gain_bits is None else x * M.bf16_bits_to_f64(gain_bits)[None, :]


def rms_eps_outside_sqrt(r_bits, eps, gain_bits=None):
    r = M.bf16_bits_to_f64(r_bits)
    x = r / (np.sqrt(np.mean(r * r, axis=1, keepdims=True)) + eps)
    return x if gain_bits is None else x * M.bf16_bits_to_f64(gain_bits)[None, :]


def rms_gain_divides(r_bits, eps, gain_bits=None):
    x = _rms(r_bits, eps)
    return x if gain_bits is None else x / M.bf16_bits_to_f64(gain_bits)[None, :]


MUTANTS = [
    ("dequant", nibble_order_reversed), ("dequant", bias_subtracted), ("dequant", signed_codes),
    ("dequant", scale_per_group_of_32), ("select_top_k", ties_to_higher_index),
    ("router_logits", logits_transposed_bias), ("route", no_renormalisation),
    ("route", gate_is_one_minus_sigmoid), ("routing_tables", scatter_reversed_within_expert),
    ("routing_tables", tiles_off_by_one), ("routing_tables", offsets_inclusive),
    ("swiglu_expert", gate_up_swapped), ("swiglu_expert", relu_instead_of_silu),
    ("swiglu_expert", down_transposed), ("rms_norm", rms_sum_not_mean), ("rms_norm", rms_without_sqrt),
    ("rms_norm", rms_eps_outside_sqrt), ("rms_norm", rms_gain_divides),
]


def _attention_variant(label, mapping="div", scale_mode="rsqrt", len_shift=0, normalise=True, v_head=None,
                       shift=True):
    """A copy of the decode-attention oracle with one plausible mistake."""
    def attn(q_bits, k_bits, v_bits, lens, scale=None):
        q, K, V = (M.bf16_bits_to_f64(t) for t in (q_bits, k_bits, v_bits))
        B, Hq, D = q.shape
        Hkv = K.shape[1]
        r = Hq // Hkv
        s = {"rsqrt": 1 / np.sqrt(D), "one": 1.0, "sqrt": np.sqrt(D)}[scale_mode] if scale is None else scale
        o = np.zeros((B, Hq, D))
        for b in range(B):
            n = int(lens[b])
            n = min(max(n + len_shift, 1), K.shape[2]) if n > 0 else 0
            for h in range(Hq if n else 0):
                g = h // r if mapping == "div" else h % Hkv
                gv = g if v_head is None else v_head(h, Hkv)
                lg = s * (K[b, g, :n] @ q[b, h])
                with np.errstate(over="ignore", invalid="ignore"):
                    w = np.exp(lg - lg.max()) if shift else np.exp(lg)
                if normalise:
                    with np.errstate(invalid="ignore"):
                        w /= w.sum()
                o[b, h] = w @ V[b, gv, :n]
        return o
    attn.__name__ = label
    return attn


ATTN_MUTANTS = [
    _attention_variant("kv_head_by_modulo", mapping="mod"),
    _attention_variant("scale_missing", scale_mode="one"),
    _attention_variant("scale_inverted", scale_mode="sqrt"),
    _attention_variant("one_position_short", len_shift=-1),
    _attention_variant("one_position_past_length", len_shift=1),
    _attention_variant("weights_not_normalised", normalise=False),
    _attention_variant("values_from_other_kv_head", v_head=lambda h, Hkv: (h + 1) % Hkv),
    _attention_variant("softmax_without_max_shift", shift=False),
]


def _caught_by_some_pin():
    caught = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    return caught


@pytest.mark.parametrize("mutant", ATTN_MUTANTS, ids=[m.__name__ for m in ATTN_MUTANTS])
def test_planted_attention_mistake_is_caught(monkeypatch, mutant):
    monkeypatch.setattr(A, "gqa_decode_attention", mutant)
    assert _caught_by_some_pin(), f"no pin caught the planted mistake {mutant.__name__}"


def test_attention_variant_without_mistake_passes(monkeypatch):
    """The mutant generator itself, with no mistake switched on, passes every
    pin (so a caught mutant is caught for its mistake)."""
    monkeypatch.setattr(A, "gqa_decode_attention", _attention_variant("faithful_copy"))
    assert not _caught_by_some_pin()


def _gdn_variant(label, order="decay_first", knorm=True, qscale=True, delta_from="decayed", mapping="div",
                 read="after"):
    """A copy of the Gated DeltaNet oracle with one plausible mistake."""
    def scan(q_bits, k_bits, v_bits, gate, beta, state0, offsets):
        q, k, v = (M.bf16_bits_to_f64(t) for t in (q_bits, k_bits, v_bits))
        S_all = np.array(state0, dtype=np.float64, copy=True)
        T, Hqk, Dk = q.shape
        Hv = v.shape[1]
        per = Hv // Hqk
        o = np.zeros((T, Hv, v.shape[2]))
        for b in range(len(offsets) - 1):
            for h in range(Hv):
                g = h // per if mapping == "div" else h % Hqk
                S = S_all[b, h]
                for t in range(int(offsets[b]), int(offsets[b + 1])):
                    kh = k[t, g] / np.sqrt((k[t, g] ** 2).sum() + 1e-6) if knorm else k[t, g]
                    qh = q[t, g] / np.sqrt((q[t, g] ** 2).sum() + 1e-6)
                    if qscale:
                        qh = qh / np.sqrt(Dk)
                    a = np.exp(gate[t, h])
                    if read == "before":
                        o[t, h] = (a * S) @ qh
                    if order == "decay_first":
                        Sk = (S @ kh) if delta_from == "undecayed" else (a * S) @ kh
                        S *= a
                        S += np.outer(beta[t, h] * (v[t, h] - Sk), kh)
                    else:
                        S += np.outer(beta[t, h] * (v[t, h] - S @ kh), kh)
                        S *= a
                    if read == "after":
                        o[t, h] = S @ qh
        return o, S_all
    scan.__name__ = label
    return scan


GDN_MUTANTS = [
    _gdn_variant("decay_after_write", order="write_first"),
    _gdn_variant("key_not_normalised", knorm=False),
    _gdn_variant("query_not_scaled", qscale=False),
    _gdn_variant("delta_against_undecayed_state", delta_from="undecayed"),
    _gdn_variant("value_head_by_modulo", mapping="mod"),
    _gdn_variant("output_read_before_write", read="before"),
]


@pytest.mark.parametrize("mutant", GDN_MUTANTS, ids=[m.__name__ for m in GDN_MUTANTS])
def test_planted_gdn_mistake_is_caught(monkeypatch, mutant):
    monkeypatch.setattr(G, "gated_delta_scan", mutant)
    assert _caught_by_some_pin(), f"no pin caught the planted mistake {mutant.__name__}"


def test_gdn_variant_without_mistake_passes(monkeypatch):
    monkeypatch.setattr(G, "gated_delta_scan", _gdn_variant("faithful_copy"))
    assert not _caught_by_some_pin()


@pytest.mark.parametrize("name,mutant", MUTANTS, ids=[m.__name__ for _, m in MUTANTS])
def test_planted_mistake_is_caught(monkeypatch, name, mutant):
    monkeypatch.setattr(M, name, mutant)
    caught = []
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake {mutant.__name__}"
