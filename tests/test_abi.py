"""The C-ABI library without a GPU: it loads, exports every entry point that
include/moe.h declares, and rejects bad arguments on the host before any
CUDA work (no compute calls here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


def test_every_declared_symbol_is_exported(moelib):
    syms = declared_symbols()
    assert len(syms) >= 10
    L = moelib.lib()
    for s in syms:
        assert hasattr(L, s), s


def test_abi_version_and_strings(moelib):
    L = moelib.lib()
    assert L.moe_abi_version() == 1
    for s in range(6):
        assert moelib.status_string(s)
    assert moelib.status_string(99) == "unknown status"


def test_workspace_bytes_grows_with_tokens(moelib):
    sizes = [moelib.workspace_bytes(moelib.make_shape(T, 2048, 512)) for T in (1, 4, 512, 4096)]
    assert all(b > a for a, b in zip(sizes, sizes[1:]))
    assert sizes[-1] % 256 == 0


@pytest.mark.parametrize("kw,code", [
    (dict(H=100), 2), (dict(I=96), 2), (dict(top_k=9), 2), (dict(E=300), 2), (dict(block_m=48), 2),
    (dict(block_m=256), 2),
    (dict(group_size=32), 2), (dict(T=-1), 1), (dict(E=4, top_k=8), 2)])
def test_shape_rejected(moelib, kw, code):
    args = dict(T=4, H=512, I=128, E=256, top_k=8, shared=True, block_m=16, group_size=64)
    args.update(kw)
    sh = moelib.make_shape(**args)
    n = ctypes.c_size_t()
    assert moelib.lib().moe_workspace_bytes(ctypes.byref(sh), ctypes.byref(n)) == code


def test_max_tiles_formula(moelib):
    for T, bm in [(1, 16), (64, 16), (4096, 128), (37, 32)]:
        sh = moelib.make_shape(T, 512, 128, block_m=bm)
        A = T * 8
        want = -(-A // bm) + min(256, A) + -(-T // bm)
        assert moelib.max_tiles(sh) == want


def _fake_route_out(moelib, shared=True):
    vals = [0x10000 * (i + 1) for i in range(len(moelib.ROUTE_FIELDS))]
    r = moelib.RouteOutC(*vals)
    if not shared:
        r.gate = None
    return r


def test_host_side_errors_before_any_cuda_call(moelib):
    """Null pointers, short or misaligned workspaces and T == 0 are settled on
    the host; the fake device addresses below are never dereferenced."""
    L = moelib.lib()
    sh = moelib.make_shape(64, 512, 128)
    need = moelib.workspace_bytes(sh)
    r = _fake_route_out(moelib)
    x, w, g, ws = 0x100000, 0x200000, 0x300000, 0x400000
    assert L.moe_route(ctypes.byref(sh), x, w, None, g, ctypes.byref(r), ws, need - 1, None) == 3
    assert L.moe_route(ctypes.byref(sh), None, w, None, g, ctypes.byref(r), ws, need, None) == 1
    assert L.moe_route(ctypes.byref(sh), x, w, None, None, ctypes.byref(r), ws, need, None) == 1
    assert L.moe_route(ctypes.byref(sh), x, w, None, g, ctypes.byref(r), ws + 16, need, None) == 1
    r2 = _fake_route_out(moelib)
    r2.sorted = None
    assert L.moe_route(ctypes.byref(sh), x, w, None, g, ctypes.byref(r2), ws, need, None) == 1
    sh0 = moelib.make_shape(0, 512, 128)
    assert L.moe_route(ctypes.byref(sh0), x, w, None, g, ctypes.byref(r), ws, 0, None) == 0
    ex = moelib.ExpertsC(moelib.QMat(1 << 20, 2 << 20, 3 << 20), moelib.QMat(4 << 20, 5 << 20, 6 << 20))
    assert L.moe_forward(ctypes.byref(sh), x, w, None, ctypes.byref(ex), None, g, 0x500000, None, ws, need,
                         None) == 1  # shared expert missing
    assert L.moe_forward(ctypes.byref(sh), x, w, None, ctypes.byref(ex), ctypes.byref(ex), g, 0x500000, None, ws,
                         need - 256, None) == 3
    assert L.moe_forward(ctypes.byref(sh0), x, w, None, ctypes.byref(ex), ctypes.byref(ex), g, 0x500000, None, ws,
                         0, None) == 0
    shn = moelib.make_shape(64, 512, 128, shared=False)
    rn = _fake_route_out(moelib, shared=False)
    assert L.moe_route(ctypes.byref(shn), x, w, None, None, ctypes.byref(rn), ws,
                       moelib.workspace_bytes(shn) - 1, None) == 3


def test_stall_hook_argument_checks(moelib):
    L = moelib.lib()
    sh = moelib.make_shape(64, 512, 128)
    r = _fake_route_out(moelib)
    nb = moelib.route_blocks(sh)
    assert nb == 4
    for blk, to in [(-1, 10**6), (nb, 10**6), (0, 0), (0, 10**10)]:
        assert L.moe_test_route_stall(ctypes.byref(sh), 0x100000, 0x200000, None, 0x300000, ctypes.byref(r),
                                      0x400000, 1 << 30, blk, to, None) == 1


@pytest.mark.parametrize("shape,code", [
    ((0, 16, 2, 256, 64), 2), ((4097, 16, 2, 256, 64), 2), ((1, 16, 3, 256, 64), 2), ((1, 18, 2, 256, 64), 2),
    ((1, 16, 2, 96, 64), 2), ((1, 16, 2, 512, 64), 2), ((1, 16, 2, 256, 0), 2), ((1, 16, 2, 256, (1 << 26) + 1), 2),
    ((2048, 64, 64, 64, 8), 2), ((1, 16, 2, 256, 1 << 26), 0), ((4096, 8, 8, 64, 1), 0)])
def test_attention_shape_checks(moelib, shape, code):
    sh = moelib.attn_shape(*shape)
    n = ctypes.c_size_t()
    assert moelib.lib().moe_attn_workspace_bytes(ctypes.byref(sh), ctypes.byref(n)) == code


def test_attention_workspace_formula(moelib):
    """256 bytes of status, 256 per-block flags, then (256 + B*Hkv) partial
    slots of 8 heads x (D + 2) floats."""
    for B, Hkv, D in [(1, 2, 256), (8, 2, 256), (37, 4, 64)]:
        sh = moelib.attn_shape(B, 4 * Hkv, Hkv, D, 1000)
        assert moelib.attn_workspace_bytes(sh) == 256 + 1024 + (256 + B * Hkv) * 8 * (D + 2) * 4


def test_attention_host_side_errors_before_any_cuda_call(moelib):
    """Null or misaligned pointers, a short workspace and a bad scale are
    rejected on the host; the fake device addresses are never dereferenced."""
    L = moelib.lib()
    sh = moelib.attn_shape(2, 16, 2, 256, 4096)
    need = moelib.attn_workspace_bytes(sh)
    q, k, v, lens, o, ws = 0x100000, 0x200000, 0x300000, 0x400000, 0x500000, 0x600000
    call = L.moe_attn_decode
    assert call(ctypes.byref(sh), q, k, v, lens, 0.0625, o, ws, need - 1, None) == 3
    assert call(ctypes.byref(sh), None, k, v, lens, 0.0625, o, ws, need, None) == 1
    assert call(ctypes.byref(sh), q, k, None, lens, 0.0625, o, ws, need, None) == 1
    assert call(ctypes.byref(sh), q, k, v, None, 0.0625, o, ws, need, None) == 1
    assert call(ctypes.byref(sh), q + 8, k, v, lens, 0.0625, o, ws, need, None) == 1
    assert call(ctypes.byref(sh), q, k + 2, v, lens, 0.0625, o, ws, need, None) == 1
    assert call(ctypes.byref(sh), q, k, v, lens, 0.0625, o + 8, ws, need, None) == 1
    assert call(ctypes.byref(sh), q, k, v, lens, 0.0625, o, ws + 16, need, None) == 1
    for bad in (0.0, -1.0, float("inf"), float("nan")):
        assert call(ctypes.byref(sh), q, k, v, lens, bad, o, ws, need, None) == 1
    assert L.moe_attn_decode_timed(ctypes.byref(sh), q, k, v, lens, 0.0625, o, ws, need, None, None) == 1
    # the stall hook: a negative block or a timeout out of (0, 1 s] is refused
    # before any CUDA call
    for blk, to in [(-1, 10**6), (0, 0), (0, -5), (0, 10**10)]:
        assert L.moe_attn_test_stall(ctypes.byref(sh), q, k, v, lens, 0.0625, o, ws, need, blk, to, None) == 1


@pytest.mark.parametrize("shape,code", [
    ((1, 1, 16, 32, 128, 128), 0), ((0, 1, 16, 32, 128, 128), 2), ((1, -1, 16, 32, 128, 128), 2),
    ((1, 1, 16, 24, 128, 128), 2), ((1, 1, 32, 16, 128, 128), 2), ((1, 1, 16, 32, 64, 128), 2),
    ((1, 1, 16, 32, 128, 64), 2), ((65536, 1, 1, 1, 128, 128), 2), ((1, 1, 1, 4097, 128, 128), 2),
    # the largest supported grid, 65535 x 4096 x 8 = 2^31 - 32768 blocks, is accepted
    ((65535, 1, 1, 4096, 128, 128), 0)])
def test_gdn_shape_checks(moelib, shape, code):
    """Shapes are checked on the host before any CUDA call (the fake device
    addresses are never dereferenced)."""
    sh = moelib.gdn_shape(*shape)
    p = 0x100000
    # offsets = NULL: a supported shape gets as far as the pointer checks (1),
    # an unsupported one stops at the shape check (2); nothing is launched
    got = moelib.lib().moe_gdn_scan(ctypes.byref(sh), p, p, p, p, p, None, p, p, p, None, None)
    assert got == (code if code else 1)


def test_gdn_host_side_errors_before_any_cuda_call(moelib):
    L = moelib.lib()
    sh = moelib.gdn_shape(2, 8, 16, 32)
    a = [0x100000 * (i + 1) for i in range(9)]   # q k v gate beta offsets state_in state_out o
    for i in range(9):
        bad = list(a)
        bad[i] = None
        assert L.moe_gdn_scan(ctypes.byref(sh), *bad, None, None) == 1, i
    for i, off in [(0, 8), (1, 4), (6, 4), (7, 8), (2, 2), (2, 8), (3, 2), (8, 2)]:
        bad = list(a)
        bad[i] += off
        assert L.moe_gdn_scan(ctypes.byref(sh), *bad, None, None) == 1, (i, off)
    ev = (ctypes.c_void_p * 2)(0x700000, None)
    assert L.moe_gdn_scan_timed(ctypes.byref(sh), *a, None, ev, None) == 1
