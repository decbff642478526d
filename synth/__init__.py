"""Seeded synthetic inputs for one Qwen3.6-35B-A3B-shaped MoE layer.

This module only draws random numbers. It holds none of the layer's arithmetic
(no dequantisation, routing, activation or combine), so both the CPU oracle and
the CUDA path can take their inputs from it without sharing any of the method.

Generator: a counter-based form of SplitMix64 (Steele, Lea and Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014). The i-th output of a
SplitMix64 stream started from state s is mix(s + (i + 1) * GAMMA), with
GAMMA = 0x9E3779B97F4A7C15 and `mix` the published 64-bit finaliser. Every
tensor draws from its own stream, whose starting state is output number
`stream` of the stream seeded with the run seed. Any element is therefore a pure
function of (seed, stream, index): the device can generate a whole layer while
the oracle regenerates only the experts it needs, bit for bit the same integer
draws (torch int64 arithmetic wraps modulo 2**64 on both CPU and CUDA).

Normals use the Box-Muller transform in fp64 on two consecutive draws, then
round fp64 -> fp32 -> bf16, each round-to-nearest-even.

Distributions (the router of 256 experts with top-8 plus one shared expert is
from "Model specification" on dothoosh.com; the 4-bit format with one bf16
scale and bias per 64 weights from its "Prefill optimisations"):
  x      ~ N(0, 1)                    bf16 [T, H]
  W_r    ~ N(0, 1/sqrt(H))            bf16 [E, H]
  w_sg   ~ N(0, 1/sqrt(H))            bf16 [H]
  codes  uniform 0..15 per nibble     uint32 words, 8 nibbles each
  scale  = |N(0, 0.02)|               bf16, one per 64 weights along K
  bias   = -8 * scale + N(0, 1e-3)    bf16, one per 64 weights along K
"""
from __future__ import annotations

import itertools
import math
from dataclasses import dataclass, field

import torch

GAMMA = 0x9E3779B97F4A7C15
MIX1 = 0xBF58476D1CE4E5B9
MIX2 = 0x94D049BB133111EB


def _s64(v: int) -> int:
    """Reinterpret an unsigned 64-bit constant as a signed int64."""
    v &= (1 << 64) - 1
    return v - (1 << 64) if v >= (1 << 63) else v


def _srl(z: torch.Tensor, s: int) -> torch.Tensor:
    """Logical right shift of int64 bit patterns."""
    return (z >> s) & ((1 << (64 - s)) - 1)


def _mix(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _srl(z, 30)) * _s64(MIX1)
    z = (z ^ _srl(z, 27)) * _s64(MIX2)
    return z ^ _srl(z, 31)


def _mix_int(v: int) -> int:
    m = (1 << 64) - 1
    v &= m
    v = ((v ^ (v >> 30)) * MIX1) & m
    v = ((v ^ (v >> 27)) * MIX2) & m
    return v ^ (v >> 31)


def stream_key(seed: int, stream: int) -> int:
    """Starting state of stream `stream`: output number `stream` of the
    SplitMix64 sequence seeded with `seed` (an unsigned 64-bit integer)."""
    return _mix_int(seed + (stream + 1) * GAMMA)


def draws(keys: torch.Tensor, start: int, n: int) -> torch.Tensor:
    """Raw 64-bit draws (as int64 bit patterns) number start..start+n-1 of
    every stream in `keys` (int64 [S]) -> int64 [S, n]."""
    dev = keys.device
    i = torch.arange(start + 1, start + n + 1, dtype=torch.int64, device=dev)
    ctr = i * _s64(GAMMA)
    return _mix(keys[:, None] + ctr[None, :])


def _keys(seed: int, streams, device) -> torch.Tensor:
    return torch.tensor([_s64(stream_key(seed, s)) for s in streams], dtype=torch.int64, device=device)


def uniform_words(seed: int, streams, n: int, device="cpu") -> torch.Tensor:
    """n uint32 words per stream (low 32 bits of each draw; every nibble is
    uniform on 0..15), returned as int32 bit patterns [S, n]."""
    z = draws(_keys(seed, streams, device), 0, n) & 0xFFFFFFFF
    z = torch.where(z >= (1 << 31), z - (1 << 32), z)
    return z.to(torch.int32)


def normal_f64(seed: int, streams, n: int, device="cpu") -> torch.Tensor:
    """n standard normals per stream, fp64 [S, n] (Box-Muller on draws 2i, 2i+1)."""
    z = draws(_keys(seed, streams, device), 0, 2 * n).view(-1, n, 2)
    u1 = (_srl(z[..., 0], 11) + 1).to(torch.float64) * (2.0 ** -53)
    u2 = _srl(z[..., 1], 11).to(torch.float64) * (2.0 ** -53)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)


def to_bf16(v64: torch.Tensor) -> torch.Tensor:
    """fp64 -> fp32 -> bf16, each step round-to-nearest-even."""
    return v64.to(torch.float32).to(torch.bfloat16)


# Stream numbering: kind * 2**32 + layer * 2**12 + expert.
K_X, K_WR, K_WSG = 1, 2, 3
K_GU_CODES, K_GU_SCALE, K_GU_BIAS = 10, 11, 12
K_DN_CODES, K_DN_SCALE, K_DN_BIAS = 20, 21, 22
K_ZIPF_PERM, K_HOT = 30, 31


def stream_id(kind: int, layer: int = 0, expert: int = 0) -> int:
    return (int(kind) << 32) | (int(layer) << 12) | int(expert)


def qmat(seed: int, layer: int, experts, n_rows: int, k: int, kinds, device="cpu", group: int = 64):
    """Packed 4-bit weights for the listed experts: codes int32 [X, n_rows, k/8],
    scales and biases bf16 [X, n_rows, k/64]."""
    kc, ks, kb = kinds
    experts = list(experts)
    codes = uniform_words(seed, [stream_id(kc, layer, e) for e in experts], n_rows * (k // 8), device)
    ng = n_rows * (k // group)
    scale = to_bf16(normal_f64(seed, [stream_id(ks, layer, e) for e in experts], ng, device).abs() * 0.02)
    noise = normal_f64(seed, [stream_id(kb, layer, e) for e in experts], ng, device)
    bias = to_bf16(-8.0 * scale.to(torch.float64) + 1e-3 * noise)
    X = len(experts)
    return (codes.view(X, n_rows, k // 8), scale.view(X, n_rows, k // group), bias.view(X, n_rows, k // group))


@dataclass
class LayerSpec:
    """One workload: T tokens through one MoE layer of shape (H, I, E, top_k)."""
    name: str
    T: int
    H: int
    I: int
    E: int = 256
    top_k: int = 8
    shared: bool = True
    bias: str = "none"          # "none" | "zipf" | "hot"
    zipf_s: float = 1.1
    hot_experts: int = 4
    cold_experts: int = 30
    hot_logit: float = 0.0      # logit offset of the hot experts ("hot" bias)
    seed: int = 20260001
    layers: int = 1
    chunk: int = 0              # 0: one call; else tokens per call


def router_bias(spec: LayerSpec, device="cpu"):
    """Per-expert fp32 router logit bias for the skewed workloads, or None.

    zipf: b_e = ln p_e with p_e proportional to rank**-s over a seeded
          permutation of the experts.
    hot:  `hot_experts` experts get +hot_logit, `cold_experts` get -30, the
          rest 0 (experts picked by a seeded permutation)."""
    if spec.bias == "none":
        return None
    E = spec.E
    key = uniform_words(spec.seed, [stream_id(K_ZIPF_PERM)], E, "cpu")[0].to(torch.int64) & 0xFFFFFFFF
    perm = torch.argsort(key * 1024 + torch.arange(E), stable=True)
    b = torch.zeros(E, dtype=torch.float64)
    if spec.bias == "zipf":
        rank = torch.arange(1, E + 1, dtype=torch.float64)
        p = rank ** (-spec.zipf_s)
        p = p / p.sum()
        b[perm] = torch.log(p)
    elif spec.bias == "hot":
        b[perm[: spec.hot_experts]] = spec.hot_logit
        b[perm[spec.hot_experts: spec.hot_experts + spec.cold_experts]] = -30.0
    else:
        raise ValueError(spec.bias)
    return b.to(torch.float32).to(device)


def activations(spec: LayerSpec, T: int | None = None, device="cpu", start: int = 0):
    """x bf16 [T, H] (token rows start..start+T-1 of the workload)."""
    T = spec.T if T is None else T
    z = normal_f64(spec.seed, [stream_id(K_X)], (start + T) * spec.H, device)[0]
    return to_bf16(z[start * spec.H:]).view(T, spec.H)


def router_weights(spec: LayerSpec, layer: int = 0, device="cpu"):
    """W_r bf16 [E, H] and w_sg bf16 [H] (None without a shared expert)."""
    std = 1.0 / math.sqrt(spec.H)
    wr = to_bf16(normal_f64(spec.seed, [stream_id(K_WR, layer)], spec.E * spec.H, device)[0] * std)
    wsg = None
    if spec.shared:
        wsg = to_bf16(normal_f64(spec.seed, [stream_id(K_WSG, layer)], spec.H, device)[0] * std)
    return wr.view(spec.E, spec.H), wsg


def expert_weights(spec: LayerSpec, experts, layer: int = 0, device="cpu"):
    """Packed weights of the listed experts (index E = the shared expert).

    gate_up: codes [X, 2I, H/8], scale/bias [X, 2I, H/64] (gate rows first)
    down:    codes [X, H, I/8],  scale/bias [X, H, I/64]"""
    gu = qmat(spec.seed, layer, experts, 2 * spec.I, spec.H, (K_GU_CODES, K_GU_SCALE, K_GU_BIAS), device)
    dn = qmat(spec.seed, layer, experts, spec.H, spec.I, (K_DN_CODES, K_DN_SCALE, K_DN_BIAS), device)
    return gu, dn


@dataclass
class Layer:
    """All tensors of one layer (bf16 as torch.bfloat16, codes as int32 bits)."""
    wr: torch.Tensor
    wsg: torch.Tensor | None
    bias: torch.Tensor | None
    gu: tuple
    dn: tuple
    sgu: tuple | None = None
    sdn: tuple | None = None
    extra: dict = field(default_factory=dict)


def layer(spec: LayerSpec, layer_idx: int = 0, device="cpu") -> Layer:
    wr, wsg = router_weights(spec, layer_idx, device)
    gu, dn = expert_weights(spec, range(spec.E), layer_idx, device)
    sgu = sdn = None
    if spec.shared:
        sgu, sdn = expert_weights(spec, [spec.E], layer_idx, device)
    return Layer(wr=wr, wsg=wsg, bias=router_bias(spec, device), gu=gu, dn=dn, sgu=sgu, sdn=sdn)


# The five workloads (token counts, shapes and router skew).
WORKLOADS = {
    "tiny": LayerSpec("tiny", T=64, H=512, I=128, seed=20260001),
    "decode-t1": LayerSpec("decode-t1", T=1, H=2048, I=512, seed=20260002, layers=40),
    "decode-t4": LayerSpec("decode-t4", T=4, H=2048, I=512, seed=20260002, layers=40),
    "prefill-zipf-512": LayerSpec("prefill-zipf-512", T=512, H=2048, I=512, bias="zipf", seed=20260003),
    "prefill-4096": LayerSpec("prefill-4096", T=4096, H=2048, I=512, seed=20260004),
    # 2048 tokens, unbiased router: the prompt length of the tile-height
    # ablation (rows per expert tile, 16 -> 32 and beyond)
    "prefill-2048": LayerSpec("prefill-2048", T=2048, H=2048, I=512, seed=20260006),
    "long-skew-16384": LayerSpec("long-skew-16384", T=16384, H=2048, I=512, bias="hot",
                                 hot_logit=1.65, seed=20260005, chunk=2048),
}


# ------------------------------------------------------- decode attention ---
# Streams: kind * 2**32 + layer * 2**12 + (b * Hkv + g) for the cache,
# kind * 2**32 + layer * 2**12 + b for the query.
K_ATT_Q, K_ATT_K, K_ATT_V = 40, 41, 42


@dataclass
class AttnSpec:
    """One decode-attention workload: B sequences with cache lengths `lens`,
    Hq query heads sharing Hkv KV heads of size D ("Model specification" on
    dothoosh.com: 16 query and 2 KV heads; D is not given there).

    q ~ N(0, q_std^2), K ~ N(0, 1), V ~ N(0, 1), all bf16. With the default
    scale 1/sqrt(D) the scores are then ~ N(0, q_std^2): q_std = 1 spreads the
    weights over the whole context, larger values make them peak on a few
    positions."""
    name: str
    lens: tuple
    Hq: int = 16
    Hkv: int = 2
    D: int = 256
    L_max: int = 0               # 0: max(lens)
    q_std: float = 1.0
    seed: int = 20260101
    layers: int = 1

    @property
    def B(self) -> int:
        return len(self.lens)

    @property
    def Lmax(self) -> int:
        return self.L_max or max(self.lens)


def attn_query(spec: AttnSpec, layer: int = 0, device="cpu"):
    """q bf16 [B, Hq, D]."""
    z = normal_f64(spec.seed, [stream_id(K_ATT_Q, layer, b) for b in range(spec.B)], spec.Hq * spec.D, device)
    return to_bf16(z * spec.q_std).view(spec.B, spec.Hq, spec.D)


def attn_cache(spec: AttnSpec, kind: int, layer: int = 0, device="cpu", pairs=None, rows=None):
    """K (kind K_ATT_K) or V (K_ATT_V) cache rows 0..rows-1 (default L_max) of
    the listed (b, g) pairs (default: all, in b-major order): bf16 [P, rows, D].
    Every row, including those past a sequence's length, holds finite values."""
    Hkv, D = spec.Hkv, spec.D
    rows = spec.Lmax if rows is None else rows
    if pairs is None:
        pairs = [(b, g) for b in range(spec.B) for g in range(Hkv)]
    out = torch.empty(len(pairs), rows, D, dtype=torch.bfloat16, device=device)
    for i, (b, g) in enumerate(pairs):   # one stream per pair keeps the draws per call bounded
        z = normal_f64(spec.seed, [stream_id(kind, layer, b * Hkv + g)], rows * D, device)
        out[i] = to_bf16(z).view(rows, D)
    return out


def attn_inputs(spec: AttnSpec, layer: int = 0, device="cpu"):
    """q [B, Hq, D], K and V [B, Hkv, L_max, D] (bf16) and lens int32 [B]."""
    q = attn_query(spec, layer, device)
    k = attn_cache(spec, K_ATT_K, layer, device).view(spec.B, spec.Hkv, spec.Lmax, spec.D)
    v = attn_cache(spec, K_ATT_V, layer, device).view(spec.B, spec.Hkv, spec.Lmax, spec.D)
    lens = torch.tensor(spec.lens, dtype=torch.int32, device=device)
    return q, k, v, lens


# Single-sequence decode at the context lengths the decode measurements on
# the pages use (32K, 64K, 128K), with the model's 10 full-attention layers
# per step; and a batch of ragged lengths.
ATTN_WORKLOADS = {
    "attn-decode-32k": AttnSpec("attn-decode-32k", lens=(32768,), layers=10, seed=20260111),
    "attn-decode-64k": AttnSpec("attn-decode-64k", lens=(65536,), layers=10, seed=20260112),
    "attn-decode-128k": AttnSpec("attn-decode-128k", lens=(131072,), layers=10, seed=20260113),
    "attn-decode-batch8": AttnSpec("attn-decode-batch8", lens=(4096, 32768, 1, 17000, 65536, 8191, 777, 20000),
                                   layers=10, seed=20260114),
}


# --------------------------------------------------------- Gated DeltaNet ---
# Streams: kind * 2**32 + layer * 2**12 + (0 for the token tensors, b for a
# sequence's initial state).
K_GDN_Q, K_GDN_K, K_GDN_V, K_GDN_GATE, K_GDN_BETA, K_GDN_STATE = 50, 51, 52, 53, 54, 55


@dataclass
class GdnSpec:
    """One Gated DeltaNet workload: sequences of `lens` new tokens each, packed
    end to end, through a layer of Hqk query/key heads and Hv value heads
    ("Model specification" on dothoosh.com: 30 Gated DeltaNet layers; the
    sizes are not given there).

    q, k, v ~ N(0, 1) bf16; gate = log(alpha) = -|N(0, 0.05)| (alpha in about
    0.9 .. 1); beta = sigmoid(N(0, 1)); initial state ~ N(0, 0.1^2) fp32."""
    name: str
    lens: tuple
    Hqk: int = 16
    Hv: int = 32
    Dk: int = 128
    Dv: int = 128
    seed: int = 20260201
    layers: int = 1

    @property
    def B(self) -> int:
        return len(self.lens)

    @property
    def T(self) -> int:
        return sum(self.lens)


def gdn_inputs(spec: GdnSpec, layer: int = 0, device="cpu"):
    """q, k bf16 [T, Hqk, Dk]; v bf16 [T, Hv, Dv]; gate, beta fp32 [T, Hv];
    state0 fp32 [B, Hv, Dv, Dk]; offsets int32 [B+1]."""
    T, Hqk, Hv, Dk, Dv = spec.T, spec.Hqk, spec.Hv, spec.Dk, spec.Dv
    q = to_bf16(normal_f64(spec.seed, [stream_id(K_GDN_Q, layer)], T * Hqk * Dk, device)[0]).view(T, Hqk, Dk)
    k = to_bf16(normal_f64(spec.seed, [stream_id(K_GDN_K, layer)], T * Hqk * Dk, device)[0]).view(T, Hqk, Dk)
    v = to_bf16(normal_f64(spec.seed, [stream_id(K_GDN_V, layer)], T * Hv * Dv, device)[0]).view(T, Hv, Dv)
    gate = (-0.05 * normal_f64(spec.seed, [stream_id(K_GDN_GATE, layer)], T * Hv, device)[0].abs())
    beta = torch.sigmoid(normal_f64(spec.seed, [stream_id(K_GDN_BETA, layer)], T * Hv, device)[0])
    state = torch.empty(spec.B, Hv, Dv, Dk, dtype=torch.float32, device=device)
    for b in range(spec.B):
        state[b] = (0.1 * normal_f64(spec.seed, [stream_id(K_GDN_STATE, layer, b)], Hv * Dv * Dk, device)[0]
                    ).to(torch.float32).view(Hv, Dv, Dk)
    offsets = torch.tensor([0] + list(itertools.accumulate(spec.lens)), dtype=torch.int32, device=device)
    return (q, k, v, gate.to(torch.float32).view(T, Hv), beta.to(torch.float32).view(T, Hv), state, offsets)


# Prefill of one 4096-token prompt (4 layers per step) and decode of 64
# sequences one token each through the model's 30 Gated DeltaNet layers; a
# ragged pack for the tests.
GDN_WORKLOADS = {
    "gdn-prefill-4096": GdnSpec("gdn-prefill-4096", lens=(4096,), layers=4, seed=20260211),
    "gdn-decode-b64": GdnSpec("gdn-decode-b64", lens=(1,) * 64, layers=30, seed=20260212),
}
