"""Python binding of the GB300 MoE-layer library (libbgmoe.so).

Argument marshalling only: torch tensors become device pointers and the
current CUDA stream is passed through; every step of the layer runs in the
library's CUDA kernels. There is no fallback: if the library is not built,
importing the entry points raises.

Entry points mirror the C ABI in include/moe.h (workspace_bytes, max_tiles,
route_blocks, route, forward, forward_residual, forward_timed, route_noalloc,
status_read, status_string, test_route_stall, test_decode_stall) and
include/attention.h (attn_workspace_bytes, attn_decode, attn_decode_timed) and
include/gdn.h (gdn_scan, gdn_scan_timed).
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libbgmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED_SHAPE = 0, 1, 2
MOE_ERR_WORKSPACE_TOO_SMALL, MOE_ERR_CUDA, MOE_ERR_DEVICE_TIMEOUT, MOE_ERR_RANGE, MOE_ERR_BOUNDS = 3, 4, 5, 6, 7
PATH_AUTO, PATH_GEMV, PATH_TENSOR_CORE, PATH_FUSED_DECODE = 0, 1, 2, 3

P = ctypes.c_void_p


class Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("T", "H", "I", "I_shared", "E", "top_k", "group_size", "block_m")]


class AttnShape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("B", "Hq", "Hkv", "D", "L_max")]


class GdnShape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("B", "T", "Hqk", "Hv", "Dk", "Dv")]


class QMat(ctypes.Structure):
    _fields_ = [("codes", P), ("scales", P), ("biases", P)]


class ExpertsC(ctypes.Structure):
    _fields_ = [("gate_up", QMat), ("down", QMat)]


ROUTE_FIELDS = ("ids", "weights", "gate", "counts", "offsets", "sorted", "inv",
                "tile_expert", "tile_row0", "tile_rows", "num_tiles", "status")


class RouteOutC(ctypes.Structure):
    _fields_ = [(n, P) for n in ROUTE_FIELDS]


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} ({status}){': ' + detail if detail else ''}")


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with bit_grouped_expert_moe_gb300._build.build()")
        L = ctypes.CDLL(LIB_PATH)
        i32, sz = ctypes.c_int32, ctypes.c_size_t
        L.moe_abi_version.restype = i32
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_status_string.argtypes = [i32]
        L.moe_last_error_detail.restype = ctypes.c_char_p
        sp = ctypes.POINTER(Shape)
        L.moe_workspace_bytes.argtypes = [sp, ctypes.POINTER(sz)]
        L.moe_max_tiles.argtypes = [sp, ctypes.POINTER(i32)]
        L.moe_route_blocks.argtypes = [sp, ctypes.POINTER(i32)]
        L.moe_route.argtypes = [sp, P, P, P, P, ctypes.POINTER(RouteOutC), P, sz, P]
        L.moe_forward.argtypes = [sp, P, P, P, ctypes.POINTER(ExpertsC), ctypes.POINTER(ExpertsC), P, P,
                                  ctypes.POINTER(RouteOutC), P, sz, P]
        L.moe_forward_residual.argtypes = [sp, P, P, ctypes.c_float, P, P, ctypes.POINTER(ExpertsC),
                                           ctypes.POINTER(ExpertsC), P, P, P, ctypes.POINTER(RouteOutC), P, sz, P]
        L.moe_forward_timed.argtypes = [sp, P, P, P, ctypes.POINTER(ExpertsC), ctypes.POINTER(ExpertsC), P, P,
                                        ctypes.POINTER(RouteOutC), P, sz, ctypes.POINTER(P), i32, P]
        L.moe_route_noalloc.argtypes = [sp, P, P, P, P, ctypes.POINTER(RouteOutC), P]
        L.moe_route_noalloc.restype = i32
        L.moe_status_read.argtypes = [P, P, ctypes.POINTER(i32)]
        L.moe_test_route_stall.argtypes = [sp, P, P, P, P, ctypes.POINTER(RouteOutC), P, sz, i32, ctypes.c_int64, P]
        L.moe_test_decode_stall.argtypes = [sp, P, P, P, ctypes.POINTER(ExpertsC), ctypes.POINTER(ExpertsC), P, P,
                                            ctypes.POINTER(RouteOutC), P, sz, i32, ctypes.c_int64, P]
        ap = ctypes.POINTER(AttnShape)
        L.moe_attn_workspace_bytes.argtypes = [ap, ctypes.POINTER(sz)]
        L.moe_attn_decode.argtypes = [ap, P, P, P, P, ctypes.c_float, P, P, sz, P]
        L.moe_attn_decode_timed.argtypes = [ap, P, P, P, P, ctypes.c_float, P, P, sz, ctypes.POINTER(P), P]
        L.moe_attn_test_stall.argtypes = [ap, P, P, P, P, ctypes.c_float, P, P, sz, i32, ctypes.c_int64, P]
        for f in ("moe_attn_workspace_bytes", "moe_attn_decode", "moe_attn_decode_timed", "moe_attn_test_stall"):
            getattr(L, f).restype = i32
        gp = ctypes.POINTER(GdnShape)
        L.moe_gdn_scan.argtypes = [gp, P, P, P, P, P, P, P, P, P, P, P]
        L.moe_gdn_scan_timed.argtypes = [gp, P, P, P, P, P, P, P, P, P, P, ctypes.POINTER(P), P]
        L.moe_gdn_scan.restype = i32
        L.moe_gdn_scan_timed.restype = i32
        for f in ("moe_workspace_bytes", "moe_max_tiles", "moe_route_blocks", "moe_route", "moe_forward",
                  "moe_forward_timed", "moe_forward_residual",
                  "moe_status_read", "moe_test_route_stall", "moe_test_decode_stall"):
            getattr(L, f).restype = i32
        _lib = L
    return _lib


def status_string(s: int) -> str:
    return lib().moe_status_string(int(s)).decode()


def _check(rc: int, where: str):
    if rc != MOE_OK:
        raise MoeError(rc, where, lib().moe_last_error_detail().decode())


def make_shape(T, H, I, E=256, top_k=8, shared=True, block_m=16, group_size=64) -> Shape:
    return Shape(T, H, I, I if shared else 0, E, top_k, group_size, block_m)


def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def workspace_bytes(shape: Shape) -> int:
    n = ctypes.c_size_t()
    _check(lib().moe_workspace_bytes(ctypes.byref(shape), ctypes.byref(n)), "moe_workspace_bytes")
    return n.value


def max_tiles(shape: Shape) -> int:
    n = ctypes.c_int32()
    _check(lib().moe_max_tiles(ctypes.byref(shape), ctypes.byref(n)), "moe_max_tiles")
    return n.value


def route_blocks(shape: Shape) -> int:
    n = ctypes.c_int32()
    _check(lib().moe_route_blocks(ctypes.byref(shape), ctypes.byref(n)), "moe_route_blocks")
    return n.value


def alloc_route_out(shape: Shape, device) -> dict:
    """Device tensors for every routing output of `shape`."""
    T, K, E = shape.T, shape.top_k, shape.E
    A = T * K
    mt = max(1, max_tiles(shape))
    i32 = dict(dtype=torch.int32, device=device)
    return dict(ids=torch.empty(max(A, 1), **i32), weights=torch.empty(max(A, 1), dtype=torch.float32, device=device),
                gate=torch.empty(max(T, 1), dtype=torch.float32, device=device), counts=torch.empty(E + 1, **i32),
                offsets=torch.empty(E + 2, **i32), sorted=torch.empty(max(A, 1), **i32), inv=torch.empty(max(A, 1), **i32),
                tile_expert=torch.empty(mt, **i32), tile_row0=torch.empty(mt, **i32), tile_rows=torch.empty(mt, **i32),
                num_tiles=torch.zeros(1, **i32), status=torch.zeros(1, **i32))


def alloc_workspace(shape: Shape, device) -> torch.Tensor:
    """A workspace buffer of moe_workspace_bytes() bytes (torch allocations are
    at least 256-byte aligned)."""
    return torch.empty(max(workspace_bytes(shape), 256), dtype=torch.uint8, device=device)


def _route_c(out: dict) -> RouteOutC:
    return RouteOutC(*[_ptr(out.get(n)) for n in ROUTE_FIELDS])


def _experts_c(ex) -> ExpertsC | None:
    """ex = ((gu_codes, gu_scales, gu_biases), (dn_codes, dn_scales, dn_biases))."""
    if ex is None:
        return None
    (gc, gs, gb), (dc, ds, db) = ex
    return ExpertsC(QMat(_ptr(gc), _ptr(gs), _ptr(gb)), QMat(_ptr(dc), _ptr(ds), _ptr(db)))


def route(shape, x, w_router, router_bias, w_shared_gate, out: dict, workspace, stream=None):
    r = _route_c(out)
    _check(lib().moe_route(ctypes.byref(shape), _ptr(x), _ptr(w_router), _ptr(router_bias), _ptr(w_shared_gate),
                           ctypes.byref(r), _ptr(workspace), workspace.numel() * workspace.element_size(),
                           _stream(stream)), "moe_route")


def route_noalloc(shape, x, w_router, router_bias, w_shared_gate, out: dict, stream=None):
    """moe_route without a workspace (the library's own static device
    scratch; see include/moe.h for the size limit and the sharing rules)."""
    r = _route_c(out)
    _check(lib().moe_route_noalloc(ctypes.byref(shape), _ptr(x), _ptr(w_router), _ptr(router_bias),
                                   _ptr(w_shared_gate), ctypes.byref(r), _stream(stream)), "moe_route_noalloc")


def forward(shape, x, w_router, router_bias, experts, shared, w_shared_gate, y, workspace, route_out=None,
            stream=None):
    ec = _experts_c(experts)
    sc = _experts_c(shared)
    r = _route_c(route_out) if route_out is not None else None
    _check(lib().moe_forward(ctypes.byref(shape), _ptr(x), _ptr(w_router), _ptr(router_bias), ctypes.byref(ec),
                             ctypes.byref(sc) if sc is not None else None, _ptr(w_shared_gate), _ptr(y),
                             ctypes.byref(r) if r is not None else None, _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream(stream)), "moe_forward")


def forward_residual(shape, r, w_router, router_bias, experts, shared, w_shared_gate, y, r_next, workspace,
                     norm_weight=None, norm_eps=1e-6, route_out=None, stream=None):
    """moe_forward_residual: one pre-norm MoE block. The layer runs on
    x = RMSNorm(r) (gain norm_weight, or 1), y is its output and
    r_next = bf16(r + y) the next layer's residual row (bf16 [T, H],
    distinct from r). Fused decode shapes only."""
    ec = _experts_c(experts)
    sc = _experts_c(shared)
    rc = _route_c(route_out) if route_out is not None else None
    _check(lib().moe_forward_residual(ctypes.byref(shape), _ptr(r), _ptr(norm_weight), float(norm_eps),
                                      _ptr(w_router), _ptr(router_bias), ctypes.byref(ec),
                                      ctypes.byref(sc) if sc is not None else None, _ptr(w_shared_gate), _ptr(y),
                                      _ptr(r_next), ctypes.byref(rc) if rc is not None else None, _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _stream(stream)),
           "moe_forward_residual")


def forward_timed(shape, x, w_router, router_bias, experts, shared, w_shared_gate, y, workspace, events=None,
                  route_out=None, path=PATH_AUTO, stream=None):
    """forward() with a chosen expert path (PATH_AUTO, PATH_GEMV,
    PATH_TENSOR_CORE) that records six caller-created CUDA events (raw
    cudaEvent_t handles, e.g. torch.cuda.Event(enable_timing=True).cuda_event
    after one record()) around its kernels when `events` is given."""
    ec = _experts_c(experts)
    sc = _experts_c(shared)
    r = _route_c(route_out) if route_out is not None else None
    ev = (P * 6)(*events) if events is not None else None
    _check(lib().moe_forward_timed(ctypes.byref(shape), _ptr(x), _ptr(w_router), _ptr(router_bias), ctypes.byref(ec),
                                   ctypes.byref(sc) if sc is not None else None, _ptr(w_shared_gate), _ptr(y),
                                   ctypes.byref(r) if r is not None else None, _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), ev, int(path), _stream(stream)),
           "moe_forward_timed")


def test_decode_stall(shape, x, w_router, router_bias, experts, shared, w_shared_gate, y, workspace, route_out: dict,
                      stalled_block: int, timeout_ns: int, stream=None):
    """moe_test_decode_stall: the fused decode path with one block that never
    publishes the h of its gate/up items, and a short device timeout."""
    ec = _experts_c(experts)
    sc = _experts_c(shared)
    r = _route_c(route_out)
    _check(lib().moe_test_decode_stall(ctypes.byref(shape), _ptr(x), _ptr(w_router), _ptr(router_bias),
                                       ctypes.byref(ec), ctypes.byref(sc) if sc is not None else None,
                                       _ptr(w_shared_gate), _ptr(y), ctypes.byref(r), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), stalled_block, timeout_ns,
                                       _stream(stream)), "moe_test_decode_stall")


def status_read(status: torch.Tensor, stream=None) -> int:
    v = ctypes.c_int32()
    _check(lib().moe_status_read(_ptr(status), _stream(stream), ctypes.byref(v)), "moe_status_read")
    return v.value


def test_route_stall(shape, x, w_router, router_bias, w_shared_gate, out: dict, workspace, stalled_block: int,
                     timeout_ns: int, stream=None):
    r = _route_c(out)
    _check(lib().moe_test_route_stall(ctypes.byref(shape), _ptr(x), _ptr(w_router), _ptr(router_bias),
                                      _ptr(w_shared_gate), ctypes.byref(r), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), stalled_block, timeout_ns,
                                      _stream(stream)), "moe_test_route_stall")


# ----------------------------------------------------- decode attention ---

def attn_shape(B, Hq, Hkv, D, L_max) -> AttnShape:
    return AttnShape(B, Hq, Hkv, D, L_max)


def attn_workspace_bytes(shape: AttnShape) -> int:
    n = ctypes.c_size_t()
    _check(lib().moe_attn_workspace_bytes(ctypes.byref(shape), ctypes.byref(n)), "moe_attn_workspace_bytes")
    return n.value


def attn_alloc_workspace(shape: AttnShape, device) -> torch.Tensor:
    return torch.empty(max(attn_workspace_bytes(shape), 256), dtype=torch.uint8, device=device)


def attn_decode(shape, q, k_cache, v_cache, lens, o, workspace, scale=None, stream=None):
    """moe_attn_decode: q bf16 [B, Hq, D], caches bf16 [B, Hkv, L_max, D],
    lens int32 [B], o fp32 [B, Hq, D] (all on the device). The workspace's
    first int32 is the call's device status word."""
    s = 1.0 / (shape.D ** 0.5) if scale is None else float(scale)
    _check(lib().moe_attn_decode(ctypes.byref(shape), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(lens), s,
                                 _ptr(o), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream(stream)), "moe_attn_decode")


def attn_test_stall(shape, q, k_cache, v_cache, lens, o, workspace, stalled_block: int, timeout_ns: int,
                    scale=None, stream=None):
    """moe_attn_test_stall: attn_decode with one grid block whose producer
    issues no cache loads and a short device timeout (test only)."""
    s = 1.0 / (shape.D ** 0.5) if scale is None else float(scale)
    _check(lib().moe_attn_test_stall(ctypes.byref(shape), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(lens), s,
                                     _ptr(o), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     int(stalled_block), int(timeout_ns), _stream(stream)), "moe_attn_test_stall")


def attn_decode_timed(shape, q, k_cache, v_cache, lens, o, workspace, events, scale=None, stream=None):
    """attn_decode recording three caller-created CUDA events (raw handles)
    before the block kernel, between it and the merge kernel, and after."""
    s = 1.0 / (shape.D ** 0.5) if scale is None else float(scale)
    ev = (P * 3)(*events)
    _check(lib().moe_attn_decode_timed(ctypes.byref(shape), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(lens), s,
                                       _ptr(o), _ptr(workspace), workspace.numel() * workspace.element_size(), ev,
                                       _stream(stream)), "moe_attn_decode_timed")


# ------------------------------------------------------- Gated DeltaNet ---

def gdn_shape(B, T, Hqk, Hv, Dk=128, Dv=128) -> GdnShape:
    return GdnShape(B, T, Hqk, Hv, Dk, Dv)


def gdn_scan(shape, q, k, v, gate, beta, offsets, state_in, state_out, o, status=None, stream=None):
    """moe_gdn_scan: q, k bf16 [T, Hqk, Dk]; v bf16 [T, Hv, Dv]; gate, beta
    fp32 [T, Hv]; offsets int32 [B+1]; states fp32 [B, Hv, Dv, Dk] (state_out
    may be state_in); o fp32 [T, Hv, Dv]; status an optional int32 device word."""
    _check(lib().moe_gdn_scan(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(beta),
                              _ptr(offsets), _ptr(state_in), _ptr(state_out), _ptr(o), _ptr(status),
                              _stream(stream)), "moe_gdn_scan")


def gdn_scan_timed(shape, q, k, v, gate, beta, offsets, state_in, state_out, o, events, status=None, stream=None):
    ev = (P * 2)(*events)
    _check(lib().moe_gdn_scan_timed(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(beta),
                                    _ptr(offsets), _ptr(state_in), _ptr(state_out), _ptr(o), _ptr(status), ev,
                                    _stream(stream)), "moe_gdn_scan_timed")
