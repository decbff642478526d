"""moe_route_noalloc: routing for callers that cannot allocate device memory.

Such callers (a host callback or real-time loop that must not enter the CUDA
allocator, a plugin handed only its input and output buffers, an embedder
whose device memory a host framework budgets) get the same routing outputs
as moe_route with a workspace. This file is collected last so that a run that
stops at its first failure has run every other test before it."""
import ctypes

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu


def _outputs(out, T, K):
    o = {k: v.cpu().numpy() for k, v in out.items()}
    n = int(o["num_tiles"][0])
    return o, n


@pytest.mark.parametrize("T,bias", [(64, "none"), (300, "zipf")])
def test_noalloc_route_matches_workspace_route_twice(moelib, cuda_dev, T, bias):
    spec = synth.LayerSpec("noalloc", T=T, H=2048, I=512, bias=bias, seed=20260031)
    wr, wsg = synth.router_weights(spec, 0, cuda_dev)
    b = synth.router_bias(spec, cuda_dev)
    shape = moelib.make_shape(T, spec.H, spec.I, block_m=32)
    ws = moelib.alloc_workspace(shape, cuda_dev)
    for call in range(2):  # two calls in a row reuse the static scratch
        x = synth.activations(spec, device=cuda_dev, start=call * T)
        ref = moelib.alloc_route_out(shape, cuda_dev)
        got = moelib.alloc_route_out(shape, cuda_dev)
        moelib.route(shape, x, wr, b, wsg, ref, ws)
        moelib.route_noalloc(shape, x, wr, b, wsg, got)
        torch.cuda.synchronize()
        assert moelib.status_read(got["status"]) == 0 and moelib.status_read(ref["status"]) == 0
        r, nr = _outputs(ref, T, 8)
        g, ng = _outputs(got, T, 8)
        A = T * 8
        assert nr == ng
        for k, n in [("ids", A), ("counts", 257), ("offsets", 258), ("sorted", A), ("inv", A),
                     ("tile_expert", nr), ("tile_row0", nr), ("tile_rows", nr)]:
            assert np.array_equal(g[k][:n], r[k][:n]), k
        assert np.allclose(g["weights"][:A], r["weights"][:A], rtol=2e-5, atol=1e-6)
        assert np.allclose(g["gate"][:T], r["gate"][:T], rtol=0, atol=3e-6)


def test_noalloc_refuses_shapes_beyond_its_scratch(moelib, cuda_dev):
    shape = moelib.make_shape(4096, 2048, 512)
    out = moelib.alloc_route_out(shape, cuda_dev)
    x = torch.zeros(4096, 2048, dtype=torch.bfloat16, device=cuda_dev)
    wr = torch.zeros(256, 2048, dtype=torch.bfloat16, device=cuda_dev)
    wsg = torch.zeros(2048, dtype=torch.bfloat16, device=cuda_dev)
    with pytest.raises(moelib.MoeError) as ei:
        moelib.route_noalloc(shape, x, wr, None, wsg, out)
    assert ei.value.status == moelib.MOE_ERR_UNSUPPORTED_SHAPE
    assert "static buffer holds 1048576" in str(ei.value)
