"""Helpers for the GPU parity tests: run the library through its C ABI on
seeded inputs, run the CPU oracle on the same inputs, compare.

The bar (from the layer's acceptance criteria): each token's set of routed
experts identical except on tokens whose 8th/9th router-logit gap is below
1e-4; routing tables bit-exact given identical ids; y within rel-L2 <= 3e-3
and max-abs <= 1e-2 * RMS(oracle y) over every other token; tokens left out
(expert sets differ across a near tie) at most 0.1 % of the tokens."""
from __future__ import annotations

import numpy as np
import torch

import oracle.cpp as ORACLE  # the C++ oracle (oracle/moe_ref.cpp); the numpy one cross-checks it
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


def gpu_forward(m, spec, L, x, block_m=16, keep_route=True, path=None, check_status=True):
    """One moe_forward call through the C ABI (moe_forward_timed with the
    given expert path when `path` is set). Returns (y fp32 [T,H] on CPU,
    routing outputs as CPU numpy arrays or None); with check_status=False,
    ((y, routing outputs), the call's device status)."""
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
    status = None
    if ro is not None:
        status = m.status_read(ro["status"])
        assert not check_status or status == 0, m.status_string(status)
        ro = {k: v.cpu().numpy() for k, v in ro.items()}
    if not check_status:
        return (y.cpu().numpy(), ro), status
    return y.cpu().numpy(), ro


def oracle_forward(spec, L, x, tokens=None):
    """The C++ oracle's layer for the listed tokens (all by default):
    (y fp64 [n, H], ids, weights, gate, logits)."""
    fn = layer_expert_fn(L, spec.E)
    bias = None if L.bias is None else L.bias.cpu().numpy()
    wsg = None if L.wsg is None else bits16(L.wsg)
    return ORACLE.moe_forward(bits16(x), bits16(L.wr), bias, wsg, spec.top_k, fn, tokens=tokens)


def oracle_route(spec, L, x):
    """The C++ oracle's routing of every token: (ids, weights, gate, logits)."""
    bias = None if L.bias is None else L.bias.cpu().numpy()
    wsg = None if L.wsg is None else bits16(L.wsg)
    return ORACLE.route(bits16(x), bits16(L.wr), bias, wsg, spec.top_k)


def topk_gap(logits, top_k):
    """l_(top_k) - l_(top_k + 1) per token on the oracle's fp64 logits (inf
    when every expert is selected): the margin between the last expert chosen
    and the first one left out."""
    l = np.sort(np.asarray(logits, dtype=np.float64), axis=1)[:, ::-1]
    if top_k >= l.shape[1]:
        return np.full(l.shape[0], np.inf)
    return l[:, top_k - 1] - l[:, top_k]


def check_ids(ids_gpu, ids_ref, logits, top_k):
    """Routing ids of the GPU against the oracle's, compared as sets per token
    (an order swap inside the selection leaves y unchanged, so such tokens are
    still compared). A token may differ only if its 8th/9th logit gap (the
    top_k-th / (top_k+1)-th) is below NEAR_TIE; those tokens are left out of
    the y comparison and must number at most MAX_EXCLUDED of the tokens.
    Returns the mask of excluded tokens."""
    ids_ref = np.asarray(ids_ref)
    ids_gpu = np.asarray(ids_gpu).reshape(ids_ref.shape)
    differ = np.any(np.sort(ids_gpu, axis=1) != np.sort(ids_ref, axis=1), axis=1)
    near = topk_gap(logits, top_k) < NEAR_TIE
    assert not np.any(differ & ~near), f"expert sets differ on {np.sum(differ & ~near)} tokens with a clear 8th/9th gap"
    excl = differ & near
    assert excl.sum() <= MAX_EXCLUDED * len(excl), f"{excl.sum()} near-tie tokens of {len(excl)} differ"
    return excl


def check_weights(ids_gpu, w_gpu, ids_ref, w_ref, keep, rtol=2e-5, atol=1e-6):
    """Routing weights per (token, expert): each token's weights are put in
    expert-id order on both sides before comparing, so an order swap inside
    the selection compares like with like."""
    ids_ref = np.asarray(ids_ref)
    ids_gpu = np.asarray(ids_gpu).reshape(ids_ref.shape)
    w_gpu = np.asarray(w_gpu).reshape(ids_ref.shape)
    og, orf = np.argsort(ids_gpu, axis=1), np.argsort(ids_ref, axis=1)
    wg = np.take_along_axis(w_gpu, og, axis=1)[keep]
    wr = np.take_along_axis(np.asarray(w_ref), orf, axis=1)[keep]
    assert np.allclose(wg, wr, rtol=rtol, atol=atol), float(np.max(np.abs(wg - wr)))


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
    tab = ORACLE.routing_tables(np.asarray(ids_gpu)[: T * K].reshape(T, K), spec.E, block_m, spec.shared)
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
