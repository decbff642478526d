"""The C++ oracle (oracle/moe_ref.cpp) behind the same functions as the numpy
oracle (oracle/moe.py), so that the same pins, planted mistakes and parity
tests run against either (test infrastructure: only the tests, the smoke check
and the benchmark's CPU legs use it).

This module only marshals arguments: every step of the arithmetic runs in the
compiled C++ file. `load(path)` binds another build of it (the planted-mistake
variants); the functions below use the default build, compiled on first use.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_ref.cpp")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libbgref.so")
GROUP = 64

_P = ctypes.c_void_p
_I = ctypes.c_int
_lock = threading.Lock()
_default = None


def compile_ref(out=LIB, mutant: int = 0, force: bool = False) -> str:
    """g++ -O2 build of moe_ref.cpp into `out` (BGREF_MUTANT=mutant)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SRC):
        return out
    cmd = ["g++", "-std=c++17", "-O2", "-shared", "-fPIC", f"-DBGREF_MUTANT={int(mutant)}", SRC, "-o", out + ".tmp"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"g++ failed for {SRC}:\n{r.stderr}")
    os.replace(out + ".tmp", out)
    return out


class Ref:
    """One loaded build of the C++ oracle."""

    def __init__(self, path: str):
        L = ctypes.CDLL(path)
        L.bgref_bf16_to_f64.argtypes = [ctypes.c_int64, _P, _P]
        L.bgref_dequant.argtypes = [_I, _I, _P, _P, _P, _P]
        L.bgref_router_logits.argtypes = [_I, _I, _I, _P, _P, _P, _P]
        L.bgref_select_top_k.argtypes = [_I, _I, _I, _P, _P]
        L.bgref_route.argtypes = [_I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P]
        L.bgref_routing_tables.argtypes = [_I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I]
        L.bgref_routing_tables.restype = _I
        L.bgref_swiglu.argtypes = [_I, _I, _I, _P, _P, _P, _P]
        L.bgref_moe_experts.argtypes = [_I] * 5 + [_P] * 4 + [ctypes.POINTER(_P)] * 6 + [_P]
        L.bgref_moe_experts.restype = _I
        L.bgref_rms_norm.argtypes = [_I, _I, _P, ctypes.c_double, _P, _P]
        self.L = L

    # -- marshalling helpers
    @staticmethod
    def _c(a, dtype):
        """Contiguous array of `dtype`; integer arrays of the same width are
        reinterpreted (raw bit patterns), anything else converted."""
        a = np.asarray(a)
        dt = np.dtype(dtype)
        a = a.view(dt) if a.dtype.kind in "iu" and dt.kind in "iu" and a.dtype.itemsize == dt.itemsize \
            else a.astype(dt)
        return np.ascontiguousarray(a)

    @staticmethod
    def _p(a):
        return None if a is None else a.ctypes.data_as(_P)

    def bits(self, a):
        return self._c(a, np.uint16)

    def bf16_bits_to_f64(self, bits):
        b = self.bits(bits)
        out = np.empty(b.shape, dtype=np.float64)
        self.L.bgref_bf16_to_f64(b.size, self._p(b), self._p(out))
        return out

    def dequant(self, codes, scales, biases, group: int = GROUP):
        assert group == GROUP
        c = self._c(codes, np.uint32)
        s, b = self.bits(scales), self.bits(biases)
        N, K = c.shape[0], c.shape[1] * 8
        assert s.shape == (N, K // GROUP) and b.shape == s.shape, (s.shape, N, K)
        W = np.empty((N, K), dtype=np.float64)
        self.L.bgref_dequant(N, K, self._p(c), self._p(s), self._p(b), self._p(W))
        return W

    def _x(self, x_bits=None, x_f64=None):
        return (self.bf16_bits_to_f64(x_bits) if x_f64 is None
                else np.ascontiguousarray(np.asarray(x_f64, dtype=np.float64)))

    def router_logits(self, x_bits, wr_bits, bias=None, x_f64=None):
        x = self._x(x_bits, x_f64)
        wr = self.bits(wr_bits)
        T, H = x.shape
        E = wr.shape[0]
        bb = None if bias is None else np.ascontiguousarray(np.asarray(bias, dtype=np.float32))
        l = np.empty((T, E), dtype=np.float64)
        self.L.bgref_router_logits(T, H, E, self._p(x), self._p(wr), self._p(bb), self._p(l))
        return l

    def select_top_k(self, logits, top_k: int):
        l = np.ascontiguousarray(np.asarray(logits, dtype=np.float64))
        T, E = l.shape
        ids = np.empty((T, top_k), dtype=np.int32)
        self.L.bgref_select_top_k(T, E, top_k, self._p(l), self._p(ids))
        return ids

    def route(self, x_bits, wr_bits, bias, wsg_bits, top_k: int, x_f64=None):
        x = self._x(x_bits, x_f64)
        wr = self.bits(wr_bits)
        T, H = x.shape
        E = wr.shape[0]
        bb = None if bias is None else np.ascontiguousarray(np.asarray(bias, dtype=np.float32))
        wsg = None if wsg_bits is None else self.bits(wsg_bits)
        logits = np.empty((T, E), dtype=np.float64)
        ids = np.empty((T, top_k), dtype=np.int32)
        w = np.empty((T, top_k), dtype=np.float64)
        gate = None if wsg is None else np.empty(T, dtype=np.float64)
        self.L.bgref_route(T, H, E, top_k, self._p(x), self._p(wr), self._p(bb), self._p(wsg), self._p(logits),
                           self._p(ids), self._p(w), self._p(gate))
        return ids, w, gate, logits

    def routing_tables(self, ids, E: int, block_m: int, shared: bool = True):
        ids = np.ascontiguousarray(np.asarray(ids, dtype=np.int32))
        T, K = ids.shape
        A = T * K
        cap = E + 1 + (A + T) // max(1, block_m) + 1
        counts = np.empty(E + 1, dtype=np.int32)
        offsets = np.empty(E + 2, dtype=np.int32)
        srt = np.empty(A, dtype=np.int32)
        inv = np.empty(A, dtype=np.int32)
        te, tr0, tr = (np.empty(cap, dtype=np.int32) for _ in range(3))
        n = self.L.bgref_routing_tables(T, K, E, block_m, int(bool(shared)), self._p(ids), self._p(counts),
                                        self._p(offsets), self._p(srt), self._p(inv), self._p(te), self._p(tr0),
                                        self._p(tr), cap)
        assert n >= 0
        return dict(counts=counts, offsets=offsets, sorted=srt, inv=inv, tile_expert=te[:n], tile_row0=tr0[:n],
                    tile_rows=tr[:n], num_tiles=n)

    def swiglu_expert(self, xrows, w_gu, w_dn):
        x = np.ascontiguousarray(np.asarray(xrows, dtype=np.float64))
        gu = np.ascontiguousarray(np.asarray(w_gu, dtype=np.float64))
        dn = np.ascontiguousarray(np.asarray(w_dn, dtype=np.float64))
        n, H = x.shape
        I = gu.shape[0] // 2
        assert gu.shape == (2 * I, H) and dn.shape == (H, I)
        o = np.empty((n, H), dtype=np.float64)
        self.L.bgref_swiglu(n, H, I, self._p(x), self._p(gu), self._p(dn), self._p(o))
        return o

    def moe_forward(self, x_bits, wr_bits, bias, wsg_bits, top_k: int, expert_fn, tokens=None, x_f64=None):
        """The same contract as oracle.moe.moe_forward: route the tokens, then
        fetch the experts they use through expert_fn(e) (e == E: the shared
        expert) and run the layer, all arithmetic in C++."""
        src = np.asarray(x_f64) if x_f64 is not None else np.asarray(x_bits)
        tokens = np.arange(src.shape[0]) if tokens is None else np.asarray(tokens)
        x = self._x(None if x_f64 is not None else np.asarray(x_bits)[tokens],
                    None if x_f64 is None else np.asarray(x_f64, dtype=np.float64)[tokens])
        ids, w, gate, logits = self.route(None, wr_bits, bias, wsg_bits, top_k, x_f64=x)
        n, H = x.shape
        E = self.bits(wr_bits).shape[0]
        keep = []  # keeps the fetched arrays alive for the call

        def table():
            return (_P * (E + 1))()

        tabs = [table() for _ in range(6)]
        kinds = (np.uint32, np.uint16, np.uint16, np.uint32, np.uint16, np.uint16)
        used = sorted(set(int(e) for e in np.unique(ids)))
        sh = None
        if gate is not None:
            sh = expert_fn(E)
            if sh is None:
                gate = None
        I = None
        for e in used + ([E] if gate is not None else []):
            parts = sh if e == E else expert_fn(e)
            for j, (a, dt) in enumerate(zip(parts, kinds)):
                arr = self._c(a, dt)
                keep.append(arr)
                tabs[j][e] = arr.ctypes.data
            I = self._c(parts[0], np.uint32).shape[0] // 2
        y = np.zeros((n, H), dtype=np.float64)
        if I is not None:
            rc = self.L.bgref_moe_experts(n, H, I, E, top_k, self._p(x), self._p(np.ascontiguousarray(ids)),
                                          self._p(np.ascontiguousarray(w)),
                                          self._p(None if gate is None else np.ascontiguousarray(gate)),
                                          *tabs, self._p(y))
            assert rc == 0
        return y, ids, w, gate, logits

    def rms_norm(self, r_bits, eps: float, gain_bits=None):
        r = self.bits(r_bits)
        T, H = r.shape
        g = None if gain_bits is None else self.bits(gain_bits)
        x = np.empty((T, H), dtype=np.float64)
        self.L.bgref_rms_norm(T, H, self._p(r), float(eps), self._p(g), self._p(x))
        return x

    def topk_gap(self, logits, top_k: int):
        l32 = np.sort(np.asarray(logits).astype(np.float32).astype(np.float64), axis=1)[:, ::-1]
        if top_k >= l32.shape[1]:
            return np.full(l32.shape[0], np.inf)
        return l32[:, top_k - 1] - l32[:, top_k]


def default() -> Ref:
    global _default
    with _lock:
        if _default is None:
            _default = Ref(compile_ref())
        return _default


def load(path: str) -> Ref:
    return Ref(path)


def __getattr__(name):
    # oracle.cpp.route(...) and friends: the default build's methods
    if name in ("bf16_bits_to_f64", "dequant", "router_logits", "select_top_k", "route", "routing_tables",
                "swiglu_expert", "moe_forward", "rms_norm", "topk_gap"):
        return getattr(default(), name)
    raise AttributeError(name)
