"""Helpers for the GPU parity tests: run the library through its C ABI on
seeded inputs, run the CPU oracle on the same inputs, compare.

The bar (from the layer's acceptance criteria): routing ids identical except
on near-tie tokens; routing tables bit-exact given identical ids; y within
rel-L2 <= 3e-3 and max-abs <= 1e-2 * RMS(oracle y) over the compared tokens;
tokens left out (ids differ on a near tie) at most 0.1 % of the tokens."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
from tests._util import bits16, u32

REL_L2 = 3e-3
MAX_ABS_RMS = 1e-2
NEAR_TIE = 1e-4
MAX_EXCLUDED = 1e-3


def device_layer(spec, layer_idx, device):
    return synth.layer(spec, layer_idx, device)


def layer_expert_fn(L, E):
    """expert_fn for the oracle from a (device) synth.Layer: copies only the
    experts asked for."""
    cache = {}

    def fn(e):
        if e in cache:
            return cache[e]
        if e == E:
            if L.sgu is None:
                return None
            gu, dn, i = L.sgu, L.sdn, 0
        else:
            gu, dn, i = L.gu, L.dn, e
        cache[e] = (u32(gu[0][i]), bits16(gu[1][i]), bits16(gu[2][i]),
                    u32(dn[0][i]), bits16(dn[1][i]), bits16(dn[2][i]))
        return cache[e]
    return fn


def experts_arg(L):
    routed = ((L.gu[0], L.gu[1], L.gu[2]), (L.dn[0], L.dn[1], L.dn[2]))
    shared = None if L.sgu is None else ((L.sgu[0], L.sgu[1], L.sgu[2]), (L.sdn[0], L.sdn[1], L.sdn[2]))
    return routed, shared


def gpu_forward(m, spec, L, x, block_m=16, keep_route=True, path=None):
    """One moe_forward call through the C ABI (moe_forward_timed with the
    given expert path when `path` is set). Returns (y fp32 [T,H] on CPU,
    routing outputs as CPU numpy arrays or None)."""
    T = x.shape[0]
    shape = m.make_shape(T, spec.H, spec.I, spec.E, spec.top_k, spec.shared, block_m)
    dev = x.device
    ws = m.alloc_workspace(shape, dev)
    y = torch.empty(T, spec.H, dtype=torch.float32, device=dev)
    ro = m.alloc_route_out(shape, dev) if keep_route else None
    routed, shared = experts_arg(L)
    if path is None:
        m.forward(shape, x, L.wr, L.bias, routed, shared, L.wsg, y, ws, route_out=ro)
    else:
        m.forward_timed(shape, x, L.wr, L.bias, routed, shared, L.wsg, y, ws, route_out=ro, path=path)
    torch.cuda.synchronize()
    if ro is not None:
        assert m.status_read(ro["status"]) == 0
        ro = {k: v.cpu().numpy() for k, v in ro.items()}
    return y.cpu().numpy(), ro


def oracle_forward(spec, L, x, tokens=None):
    fn = layer_expert_fn(L, spec.E)
    bias = None if L.bias is None else L.bias.cpu().numpy()
    wsg = None if L.wsg is None else bits16(L.wsg)
    return oracle.moe_forward(bits16(x), bits16(L.wr), bias, wsg, spec.top_k, fn, tokens=tokens)


def near_tie(logits, top_k):
    """Tokens with any two of their top_k + 1 largest fp32 logits closer than
    NEAR_TIE (the only tokens whose selection may differ by rounding)."""
    l32 = np.sort(np.asarray(logits).astype(np.float32).astype(np.float64), axis=1)[:, ::-1]
    k1 = min(top_k + 1, l32.shape[1])
    return np.any(np.diff(l32[:, :k1], axis=1) > -NEAR_TIE, axis=1)


def check_ids(ids_gpu, ids_ref, logits, top_k):
    """Returns the mask of excluded tokens; asserts the rest match exactly."""
    ids_gpu = np.asarray(ids_gpu).reshape(ids_ref.shape)
    mism = np.any(ids_gpu != ids_ref, axis=1)
    near = near_tie(logits, top_k)
    assert not np.any(mism & ~near), f"ids differ on {np.sum(mism & ~near)} tokens with a clear margin"
    excl = mism & near
    assert excl.sum() <= MAX_EXCLUDED * len(excl), f"{excl.sum()} near-tie tokens of {len(excl)} differ"
    return excl


def check_y(y_gpu, y_ref, excl=None):
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    keep = np.ones(len(y_ref), dtype=bool) if excl is None else ~excl
    err = y_gpu[keep] - y_ref[keep]
    ref = y_ref[keep]
    rms = np.sqrt(np.mean(ref ** 2))
    rel = np.linalg.norm(err) / np.linalg.norm(ref)
    mx = np.abs(err).max() / rms
    assert np.all(np.isfinite(y_gpu[keep]))
    assert rel <= REL_L2, f"rel-L2 {rel:.3e} > {REL_L2}"
    assert mx <= MAX_ABS_RMS, f"max-abs/RMS {mx:.3e} > {MAX_ABS_RMS}"
    return rel, mx


def check_tables(ro, ids_gpu, spec, T, block_m):
    """Routing tables bit-exact against the oracle's, given the GPU's ids."""
    K = spec.top_k
    tab = oracle.routing_tables(np.asarray(ids_gpu)[: T * K].reshape(T, K), spec.E, block_m, spec.shared)
    A = T * K
    assert np.array_equal(ro["counts"], tab["counts"])
    assert np.array_equal(ro["offsets"], tab["offsets"])
    assert np.array_equal(ro["sorted"][:A], tab["sorted"])
    assert np.array_equal(ro["inv"][:A], tab["inv"])
    n = tab["num_tiles"]
    assert int(ro["num_tiles"][0]) == n
    for k in ("tile_expert", "tile_row0", "tile_rows"):
        assert np.array_equal(ro[k][:n], tab[k]), k
    return tab
