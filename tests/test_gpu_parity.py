"""GPU parity: the CUDA library through its C ABI against the CPU oracle on
the same seeded inputs, for every workload shape and the edge cases."""
import numpy as np
import pytest
import torch

import oracle.cpp as oracle  # the C++ oracle
import synth
from tests import parity
from tests._util import bits16, bf16_from_f64, read_golden


def bits16_to_f64(b):
    return oracle.bf16_bits_to_f64(b)
from tests.oracle_pins import check_routing_invariants

pytestmark = pytest.mark.gpu


def _run_and_check(moelib, dev, spec, block_m=16, tokens=None, layer_idx=0, path=None):
    """One call against the oracle: routing ids (as sets), weights, gate and
    the routing tables on every token; y on every token, or on `tokens` (a
    seeded sample at the largest sizes, where the oracle's plain loops would
    take minutes)."""
    L = parity.device_layer(spec, layer_idx, dev)
    x = synth.activations(spec, device=dev)
    y, ro = parity.gpu_forward(moelib, spec, L, x, block_m, path=path)
    K = spec.top_k
    ids_gpu = ro["ids"][: spec.T * K].reshape(spec.T, K)
    ids_ref, w_ref, g_ref, logits = parity.oracle_route(spec, L, x)
    excl = parity.check_ids(ids_gpu, ids_ref, logits, K)
    # The GPU logits are fp32 sums of H products (|error| < 1e-5 at H = 2048);
    # a renormalised softmax weight moves by at most 2 max|dl| relative, and
    # the gate sigmoid by at most |dl| / 4.
    parity.check_weights(ids_gpu, ro["weights"][: spec.T * K].reshape(spec.T, K), ids_ref, w_ref, ~excl)
    if spec.shared:
        assert np.allclose(ro["gate"][: spec.T], g_ref, rtol=0, atol=3e-6)
    parity.check_tables(ro, ids_gpu, spec, spec.T, block_m)
    sel = np.arange(spec.T) if tokens is None else np.asarray(tokens)
    y_ref, *_ = parity.oracle_forward(spec, L, x, tokens=sel)
    return parity.check_y(y[sel], y_ref, excl[sel])


def _sample(T, n, seed):
    """n of T token indices, seeded, always with the first and the last."""
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, T - 1], rng.choice(T, n - 2, replace=False)]))


def test_generator_is_device_independent(cuda_dev):
    spec = synth.WORKLOADS["prefill-4096"]
    xg = synth.activations(spec, T=64, device=cuda_dev).cpu()
    xc = synth.activations(spec, T=64)
    assert torch.equal(xg.view(torch.int16), xc.view(torch.int16))
    gg, dg = synth.expert_weights(spec, [3, 256], 0, cuda_dev)
    gc, dc = synth.expert_weights(spec, [3, 256], 0, "cpu")
    for a, b in zip(gg + dg, gc + dc):
        assert torch.equal(a.cpu().view(torch.int16) if a.dtype == torch.bfloat16 else a.cpu(),
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b)


def test_tiny_layer(moelib, cuda_dev):
    rel, mx = _run_and_check(moelib, cuda_dev, synth.WORKLOADS["tiny"])
    assert rel < 1e-3


@pytest.mark.parametrize("block_m", [16, 32, 64, 128])
def test_tiny_block_sizes(moelib, cuda_dev, block_m):
    _run_and_check(moelib, cuda_dev, synth.WORKLOADS["tiny"], block_m=block_m)


@pytest.mark.parametrize("T", [1, 2, 3, 17, 37, 100])
def test_ragged_token_counts(moelib, cuda_dev, T):
    spec = synth.LayerSpec("ragged", T=T, H=512, I=128, seed=20260011)
    _run_and_check(moelib, cuda_dev, spec)


@pytest.mark.parametrize("E,K,shared,H,I", [(64, 8, True, 256, 128), (16, 2, False, 128, 64),
                                             (8, 1, True, 64, 64), (256, 8, False, 512, 192),
                                             (32, 4, True, 384, 320)])
def test_other_shapes(moelib, cuda_dev, E, K, shared, H, I):
    spec = synth.LayerSpec("shape", T=45, H=H, I=I, E=E, top_k=K, shared=shared, seed=20260012)
    _run_and_check(moelib, cuda_dev, spec, block_m=32)


@pytest.mark.parametrize("T", [1, 4])
def test_decode_full_size(moelib, cuda_dev, T):
    spec = synth.WORKLOADS[f"decode-t{T}"]
    _run_and_check(moelib, cuda_dev, spec)
    _run_and_check(moelib, cuda_dev, spec, layer_idx=39)


def test_prefill_zipf_512(moelib, cuda_dev):
    spec = synth.WORKLOADS["prefill-zipf-512"]
    _run_and_check(moelib, cuda_dev, spec, block_m=64)


def test_prefill_4096(moelib, cuda_dev):
    """Routing on all 4096 tokens; y on a seeded sample of 512."""
    spec = synth.WORKLOADS["prefill-4096"]
    _run_and_check(moelib, cuda_dev, spec, block_m=128, tokens=_sample(spec.T, 512, 1))


def test_long_skew_chunks(moelib, cuda_dev):
    """16384 tokens in 2048-token calls reusing one workspace; every chunk's
    routing is checked on all its tokens, its y on a seeded sample (384
    tokens of the first chunk, 96 of each other)."""
    spec = synth.WORKLOADS["long-skew-16384"]
    L = parity.device_layer(spec, 0, cuda_dev)
    C = spec.chunk
    chunk_spec = synth.LayerSpec(spec.name, T=C, H=spec.H, I=spec.I, bias=spec.bias, hot_logit=spec.hot_logit,
                                 seed=spec.seed)
    shape = moelib.make_shape(C, spec.H, spec.I, block_m=128)
    ws = moelib.alloc_workspace(shape, cuda_dev)
    ro = moelib.alloc_route_out(shape, cuda_dev)
    routed, shared = parity.experts_arg(L)
    rng = np.random.default_rng(5)
    hot_share = []
    for c in range(spec.T // C):
        x = synth.activations(spec, T=C, device=cuda_dev, start=c * C)
        y = torch.empty(C, spec.H, dtype=torch.float32, device=cuda_dev)
        moelib.forward(shape, x, L.wr, L.bias, routed, shared, L.wsg, y, ws, route_out=ro)
        torch.cuda.synchronize()
        assert moelib.status_read(ro["status"]) == 0
        sel = np.sort(rng.choice(C, 384 if c == 0 else 96, replace=False))
        ids_ref, _, _, logits = parity.oracle_route(chunk_spec, L, x)
        ids_gpu = ro["ids"].cpu().numpy()[: C * 8].reshape(C, 8)
        excl = parity.check_ids(ids_gpu, ids_ref, logits, 8)
        y_ref, *_ = parity.oracle_forward(chunk_spec, L, x, tokens=sel)
        parity.check_y(y.cpu().numpy()[sel], y_ref, excl[sel])
        counts = ro["counts"].cpu().numpy()
        b = L.bias.cpu().numpy()
        hot_share.append(counts[:256][b > 0].sum() / (C * 8))
        assert counts[:256][b < -1].sum() == 0
    assert 0.17 < np.mean(hot_share) < 0.23


@pytest.mark.parametrize("block_m", [16, 32, 64, 128])
def test_tensor_core_tiny(moelib, cuda_dev, block_m):
    _run_and_check(moelib, cuda_dev, synth.WORKLOADS["tiny"], block_m=block_m, path=moelib.PATH_TENSOR_CORE)


@pytest.mark.parametrize("T", [1, 2, 3, 17, 37, 100, 300])
def test_tensor_core_ragged(moelib, cuda_dev, T):
    spec = synth.LayerSpec("ragged", T=T, H=512, I=128, seed=20260015)
    _run_and_check(moelib, cuda_dev, spec, block_m=32, path=moelib.PATH_TENSOR_CORE)


@pytest.mark.parametrize("E,K,shared,H,I,bm", [(64, 8, True, 1024, 256, 64), (16, 2, False, 512, 128, 16),
                                                (32, 4, True, 1536, 384, 32), (256, 8, True, 2048, 512, 128)])
def test_tensor_core_shapes(moelib, cuda_dev, E, K, shared, H, I, bm):
    spec = synth.LayerSpec("tc-shape", T=200, H=H, I=I, E=E, top_k=K, shared=shared, seed=20260016)
    _run_and_check(moelib, cuda_dev, spec, block_m=bm, path=moelib.PATH_TENSOR_CORE)


def test_gemv_path_prefill_shape(moelib, cuda_dev):
    spec = synth.LayerSpec("gemv-prefill", T=256, H=2048, I=512, bias="zipf", seed=20260017)
    _run_and_check(moelib, cuda_dev, spec, block_m=64, path=moelib.PATH_GEMV)


def test_tensor_core_unsupported_shape_is_refused(moelib, cuda_dev):
    spec = synth.LayerSpec("no-tc", T=64, H=320, I=128, E=16, seed=20260018)
    L = parity.device_layer(spec, 0, cuda_dev)
    x = synth.activations(spec, device=cuda_dev)
    with pytest.raises(moelib.MoeError) as ei:
        parity.gpu_forward(moelib, spec, L, x, 16, path=moelib.PATH_TENSOR_CORE)
    assert ei.value.status == moelib.MOE_ERR_UNSUPPORTED_SHAPE


@pytest.mark.parametrize("T,E,K,shared,H,I", [(1, 256, 8, True, 2048, 512), (4, 256, 8, True, 2048, 512),
                                               (3, 64, 8, True, 512, 128), (2, 16, 2, False, 512, 256),
                                               (4, 8, 1, True, 512, 256), (1, 32, 4, False, 1024, 384),
                                               (4, 4, 4, True, 2048, 128), (2, 256, 8, True, 1536, 640),
                                               (3, 256, 8, True, 2048, 1024)])
def test_fused_decode(moelib, cuda_dev, T, E, K, shared, H, I):
    spec = synth.LayerSpec("fused", T=T, H=H, I=I, E=E, top_k=K, shared=shared, seed=20260019)
    _run_and_check(moelib, cuda_dev, spec, path=moelib.PATH_FUSED_DECODE)


@pytest.mark.parametrize("T,gain", [(1, False), (4, True), (3, False)])
def test_prenorm_chain_of_three_layers(moelib, cuda_dev, T, gain):
    """Three pre-norm MoE blocks run back to back through moe_forward_residual,
    each call's r_next feeding the next call: every layer's y meets the bar
    against the oracle applied to that layer's residual row (x = RMSNorm(r),
    then the layer), and r_next is exactly bf16(r + y) of the kernel's own y."""
    spec = synth.LayerSpec("chain", T=T, H=2048, I=512, seed=20260041, layers=3)
    layers = [parity.device_layer(spec, li, cuda_dev) for li in range(3)]
    r0 = synth.activations(spec, device=cuda_dev)
    g = None
    if gain:  # a gain row of 0.5 .. 1.5 in bf16
        g = (0.5 + torch.arange(spec.H, device=cuda_dev, dtype=torch.float32) / spec.H).to(torch.bfloat16)
    eps = 1e-6
    shape = moelib.make_shape(T, spec.H, spec.I, spec.E, spec.top_k, spec.shared, 16)
    ws = moelib.alloc_workspace(shape, cuda_dev)
    rs = [r0] + [torch.empty_like(r0) for _ in range(3)]
    ys = [torch.empty(T, spec.H, dtype=torch.float32, device=cuda_dev) for _ in range(3)]
    ros = [moelib.alloc_route_out(shape, cuda_dev) for _ in range(3)]
    for li, L in enumerate(layers):
        routed, shared = parity.experts_arg(L)
        moelib.forward_residual(shape, rs[li], L.wr, L.bias, routed, shared, L.wsg, ys[li], rs[li + 1], ws,
                                norm_weight=g, norm_eps=eps, route_out=ros[li])
    torch.cuda.synchronize()
    for li, L in enumerate(layers):
        assert moelib.status_read(ros[li]["status"]) == 0
        y_gpu = ys[li].cpu().numpy()
        r_bits = bits16(rs[li])
        # the join: the kernel's own y added to its own input row, rounded once to bf16
        want = bf16_from_f64(bits16_to_f64(r_bits) + y_gpu.astype(np.float64))
        assert np.array_equal(bits16(rs[li + 1]), want)
        x = oracle.rms_norm(r_bits, eps, None if g is None else bits16(g))
        y_ref, ids_ref, w_ref, g_ref, logits = oracle.moe_forward(None, bits16(L.wr), None, bits16(L.wsg),
                                                                  spec.top_k, parity.layer_expert_fn(L, spec.E),
                                                                  x_f64=x)
        ids_gpu = ros[li]["ids"].cpu().numpy()[: T * spec.top_k].reshape(T, spec.top_k)
        excl = parity.check_ids(ids_gpu, ids_ref, logits, spec.top_k)
        parity.check_y(y_gpu, y_ref, excl)
    # the stream stays in range over the three layers (the reason for the norm)
    assert torch.isfinite(rs[3].float()).all()


def test_prenorm_block_needs_the_fused_path(moelib, cuda_dev):
    """moe_forward_residual runs on the fused decode kernel only: a shape the
    fused kernel refuses (H > 2048) is refused, with nothing launched."""
    spec = synth.LayerSpec("chain-big", T=2, H=2304, I=256, E=64, top_k=4, seed=20260042)
    L = parity.device_layer(spec, 0, cuda_dev)
    r = synth.activations(spec, device=cuda_dev)
    shape = moelib.make_shape(2, spec.H, spec.I, spec.E, spec.top_k, spec.shared, 16)
    ws = moelib.alloc_workspace(shape, cuda_dev)
    y = torch.empty(2, spec.H, device=cuda_dev)
    routed, shared = parity.experts_arg(L)
    with pytest.raises(moelib.MoeError) as ei:
        moelib.forward_residual(shape, r, L.wr, L.bias, routed, shared, L.wsg, y, torch.empty_like(r), ws)
    assert ei.value.status == moelib.MOE_ERR_UNSUPPORTED_SHAPE


@pytest.mark.parametrize("H,I", [(128, 64), (320, 128), (256, 128), (4096, 512), (512, 1152)])
def test_fused_decode_shape_limits(moelib, cuda_dev, H, I):
    """The fused path takes H a multiple of 512 up to 2048 (each warp a
    quarter of K in whole 128-wide blocks, 16-row output tiles on at most the
    SM count) and I a multiple of 128 up to 1024: other decode shapes are
    refused on it and served by the GEMV path under the automatic choice."""
    spec = synth.LayerSpec("fused-limits", T=2, H=H, I=I, E=16, top_k=2, seed=20260021)
    L = parity.device_layer(spec, 0, cuda_dev)
    x = synth.activations(spec, device=cuda_dev)
    with pytest.raises(moelib.MoeError) as ei:
        parity.gpu_forward(moelib, spec, L, x, 16, path=moelib.PATH_FUSED_DECODE)
    assert ei.value.status == moelib.MOE_ERR_UNSUPPORTED_SHAPE
    _run_and_check(moelib, cuda_dev, spec, path=moelib.PATH_AUTO)


@pytest.mark.parametrize("T", [1, 4])
def test_gemv_path_decode(moelib, cuda_dev, T):
    _run_and_check(moelib, cuda_dev, synth.WORKLOADS[f"decode-t{T}"], path=moelib.PATH_GEMV)


def test_fused_decode_deterministic_and_refuses_prefill(moelib, cuda_dev):
    spec = synth.WORKLOADS["decode-t4"]
    L = parity.device_layer(spec, 3, cuda_dev)
    x = synth.activations(spec, device=cuda_dev)
    y1, r1 = parity.gpu_forward(moelib, spec, L, x, 16, path=moelib.PATH_FUSED_DECODE)
    y2, r2 = parity.gpu_forward(moelib, spec, L, x, 16, path=moelib.PATH_FUSED_DECODE)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    big = synth.LayerSpec("big", T=8, H=512, I=128, seed=20260020)
    Lb = parity.device_layer(big, 0, cuda_dev)
    with pytest.raises(moelib.MoeError) as ei:
        parity.gpu_forward(moelib, big, Lb, synth.activations(big, device=cuda_dev), 16,
                           path=moelib.PATH_FUSED_DECODE)
    assert ei.value.status == moelib.MOE_ERR_UNSUPPORTED_SHAPE


def test_topk_ties_through_gpu(moelib, cuda_dev):
    """The hand-ranked tie cases of tests/golden/topk_ties.txt through
    moe_route (lowest index first among equal logits)."""
    for (k,), logits, want in read_golden("topk_ties.txt"):
        E = len(logits)
        H = 64
        x = np.zeros((1, H))
        x[0, 0] = 1.0
        wr = np.zeros((E, H))
        wr[:, 0] = [float(v) for v in logits]
        xt = torch.from_numpy(bf16_from_f64(x).view(np.int16)).view(torch.bfloat16).to(cuda_dev)
        wt = torch.from_numpy(bf16_from_f64(wr).view(np.int16)).view(torch.bfloat16).to(cuda_dev)
        shape = moelib.make_shape(1, H, 64, E=E, top_k=int(k), shared=False)
        out = moelib.alloc_route_out(shape, cuda_dev)
        ws = moelib.alloc_workspace(shape, cuda_dev)
        moelib.route(shape, xt, wt, None, None, out, ws)
        torch.cuda.synchronize()
        assert out["ids"][: int(k)].tolist() == [int(v) for v in want]


@pytest.mark.parametrize("T,bm", [(64, 16), (1000, 32), (4096, 128), (2048, 16)])
def test_routing_tables_invariants_and_bitexact(moelib, cuda_dev, T, bm):
    spec = synth.LayerSpec("route", T=T, H=256, I=64, seed=20260013)
    wr, wsg = synth.router_weights(spec, 0, cuda_dev)
    x = synth.activations(spec, device=cuda_dev)
    shape = moelib.make_shape(T, spec.H, spec.I, block_m=bm)
    out = moelib.alloc_route_out(shape, cuda_dev)
    ws = moelib.alloc_workspace(shape, cuda_dev)
    moelib.route(shape, x, wr, None, wsg, out, ws)
    torch.cuda.synchronize()
    ro = {k: v.cpu().numpy() for k, v in out.items()}
    assert ro["status"][0] == 0
    ids = ro["ids"][: T * 8].reshape(T, 8)
    tab = parity.check_tables(ro, ids, spec, T, bm)
    check_routing_invariants(ids, 256, bm, tab)
    ids_ref, w_ref, g_ref, logits = oracle.route(bits16(x), bits16(wr), None, bits16(wsg), 8)
    parity.check_ids(ids, ids_ref, logits, 8)


def test_deterministic(moelib, cuda_dev):
    spec = synth.WORKLOADS["prefill-zipf-512"]
    L = parity.device_layer(spec, 0, cuda_dev)
    x = synth.activations(spec, device=cuda_dev)
    y1, r1 = parity.gpu_forward(moelib, spec, L, x, 64)
    y2, r2 = parity.gpu_forward(moelib, spec, L, x, 64)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    for k in r1:
        assert np.array_equal(r1[k], r2[k]), k


@pytest.mark.parametrize("name,bm", [("prefill-4096", 128), ("prefill-zipf-512", 64)])
def test_tensor_core_repeatable(moelib, cuda_dev, name, bm):
    """The tensor-core path has no atomics, so repeated runs must agree bit
    for bit; a ring-slot race between the dequantisation, gather and MMA
    warps would show up as differing values (and did, in an earlier layout
    whose dequantisation ran three stages ahead of the completed MMAs; builds
    with other ring depths are checked in test_gpu_ring_depths.py)."""
    spec = synth.WORKLOADS[name]
    L = parity.device_layer(spec, 0, cuda_dev)
    x = synth.activations(spec, device=cuda_dev)
    y0, _ = parity.gpu_forward(moelib, spec, L, x, bm, path=moelib.PATH_TENSOR_CORE)
    for _ in range(5):
        y1, _ = parity.gpu_forward(moelib, spec, L, x, bm, path=moelib.PATH_TENSOR_CORE)
        assert np.array_equal(y0.view(np.uint32), y1.view(np.uint32))


def test_zero_tokens_is_noop(moelib, cuda_dev):
    spec = synth.LayerSpec("z", T=0, H=512, I=128)
    shape = moelib.make_shape(0, 512, 128)
    L = synth.layer(synth.LayerSpec("z", T=1, H=512, I=128, E=8), 0, cuda_dev)
    y = torch.full((1, 512), 7.0, device=cuda_dev)
    routed, shared = parity.experts_arg(L)
    ws = torch.empty(256, dtype=torch.uint8, device=cuda_dev)
    x = torch.zeros(1, 512, dtype=torch.bfloat16, device=cuda_dev)
    moelib.forward(shape, x, L.wr, None, routed, shared, L.wsg, y, ws)
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)


def test_device_timeout_is_reported_not_hung(moelib, cuda_dev):
    """A routing block that never publishes its histogram makes the others
    wait out a short limit and report MOE_ERR_DEVICE_TIMEOUT; the context stays
    usable and the next normal call succeeds."""
    spec = synth.LayerSpec("stall", T=64, H=256, I=64, seed=20260014)
    wr, wsg = synth.router_weights(spec, 0, cuda_dev)
    x = synth.activations(spec, device=cuda_dev)
    shape = moelib.make_shape(64, spec.H, spec.I)
    assert moelib.route_blocks(shape) >= 2
    out = moelib.alloc_route_out(shape, cuda_dev)
    ws = moelib.alloc_workspace(shape, cuda_dev)
    moelib.test_route_stall(shape, x, wr, None, wsg, out, ws, stalled_block=0, timeout_ns=20_000_000)
    assert moelib.status_read(out["status"]) == moelib.MOE_ERR_DEVICE_TIMEOUT
    moelib.route(shape, x, wr, None, wsg, out, ws)
    assert moelib.status_read(out["status"]) == 0
    ids = out["ids"].cpu().numpy()[: 64 * 8].reshape(64, 8)
    ids_ref, *_ , logits = oracle.route(bits16(x), bits16(wr), None, bits16(wsg), 8)
    parity.check_ids(ids, ids_ref, logits, 8)


def test_fused_decode_timeout_is_reported_not_hung(moelib, cuda_dev):
    """One block of the fused decode kernel never publishes the h of its
    gate/up items: the blocks that need that h give up after a 20 ms limit and
    return (every block lets its own copies land first), the call reports
    MOE_ERR_DEVICE_TIMEOUT, and the next normal call on the same context and
    workspace is correct."""
    spec = synth.WORKLOADS["decode-t1"]
    L = parity.device_layer(spec, 0, cuda_dev)
    x = synth.activations(spec, device=cuda_dev)
    shape = moelib.make_shape(spec.T, spec.H, spec.I, spec.E, spec.top_k, spec.shared, 16)
    routed, shared = parity.experts_arg(L)
    ws = moelib.alloc_workspace(shape, cuda_dev)
    y = torch.empty(spec.T, spec.H, dtype=torch.float32, device=cuda_dev)
    ro = moelib.alloc_route_out(shape, cuda_dev)
    moelib.test_decode_stall(shape, x, L.wr, L.bias, routed, shared, L.wsg, y, ws, ro, stalled_block=3,
                             timeout_ns=20_000_000)
    torch.cuda.synchronize()
    assert moelib.status_read(ro["status"]) == moelib.MOE_ERR_DEVICE_TIMEOUT
    moelib.forward_timed(shape, x, L.wr, L.bias, routed, shared, L.wsg, y, ws, route_out=ro,
                         path=moelib.PATH_FUSED_DECODE)
    torch.cuda.synchronize()
    assert moelib.status_read(ro["status"]) == 0
    y_ref, ids_ref, w_ref, g_ref, logits = parity.oracle_forward(spec, L, x)
    excl = parity.check_ids(ro["ids"][: spec.top_k].cpu().numpy().reshape(1, -1), ids_ref, logits, spec.top_k)
    parity.check_y(y.cpu().numpy(), y_ref, excl)
