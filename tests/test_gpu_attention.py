"""Decode attention through the C ABI on the GPU against the fp64 oracle.

Tolerance, from the arithmetic: the kernel rounds each probability p_j to
bf16 (relative error <= 2^-9) and divides by the sum of the rounded values,
so each normalised weight is within 2^-8 * (1 + 2^-8) of w_j relative. Then
|o_kernel - o| <= 2^-8 * sum_j w_j |v_j| per element, which is the oracle run
on |V|. The fp32 scores (exact bf16 products, fp32 sums) move the weights by
far less; 2 % of the bound plus a small absolute term covers them and the
fp32 accumulation.
"""
import numpy as np
import pytest
import torch

import synth
from oracle.attention import gqa_decode_attention
from tests._util import bits16

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _bound(q, k, v, lens, scale=None):
    vabs = (bits16(v) & np.uint16(0x7FFF))
    o_abs = gqa_decode_attention(bits16(q), bits16(k), vabs, lens, scale)
    vmax = float(np.abs(v.float().numpy()).max()) if v.numel() else 0.0
    return 1.02 * 2.0 ** -8 * o_abs + 1e-4 * o_abs + 2e-6 * vmax + 1e-7


def _run(moelib, q, k, v, lens, scale=None):
    B, Hq, D = q.shape
    Hkv, L = k.shape[1], k.shape[2]
    sh = moelib.attn_shape(B, Hq, Hkv, D, L)
    ws = moelib.attn_alloc_workspace(sh, DEV)
    o = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device=DEV)
    moelib.attn_decode(sh, q.to(DEV), k.to(DEV), v.to(DEV), lens.to(DEV), o, ws, scale=scale)
    assert moelib.status_read(ws[:4].view(torch.int32)) == 0
    return o.cpu().numpy()


def _check(moelib, spec, poison=False, scale=None):
    q, k, v, lens = synth.attn_inputs(spec)
    if poison:   # rows past each context hold NaN: they must not reach o
        for b, n in enumerate(spec.lens):
            k[b, :, n:] = float("nan")
            v[b, :, n:] = float("nan")
    got = _run(moelib, q, k, v, lens, scale)
    kc, vc = k.clone(), v.clone()
    if poison:
        for b, n in enumerate(spec.lens):
            kc[b, :, n:] = 0
            vc[b, :, n:] = 0
    want = gqa_decode_attention(bits16(q), bits16(kc), bits16(vc), spec.lens, scale)
    tol = _bound(q, kc, vc, spec.lens, scale)
    err = np.abs(got - want)
    assert np.all(np.isfinite(got))
    bad = err > tol
    assert not bad.any(), (spec.name, int(bad.sum()), float((err / tol).max()))
    rel = np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30)
    return rel


CASES = [
    synth.AttnSpec("one-position", lens=(1,)),
    synth.AttnSpec("one-block-minus-one", lens=(63,)),
    synth.AttnSpec("one-block", lens=(64,)),
    synth.AttnSpec("one-block-plus-one", lens=(65,)),
    synth.AttnSpec("ragged-1000", lens=(1000,), q_std=3.0),
    synth.AttnSpec("with-empty", lens=(0, 130, 4097), L_max=4100),
    synth.AttnSpec("mha-d128", lens=(77, 300), Hq=8, Hkv=8, D=128),
    synth.AttnSpec("gqa4-d64", lens=(200, 5), Hq=4, Hkv=1, D=64),
    synth.AttnSpec("gqa2-d256", lens=(513, 64, 9), Hq=6, Hkv=3, D=256),
    synth.AttnSpec("peaked-5000", lens=(5000,), q_std=6.0),
    synth.AttnSpec("fewer-blocks-than-sms", lens=(100,)),
    synth.AttnSpec("many-sequences", lens=tuple(int(x) for x in
                                                np.random.default_rng(7).integers(0, 700, size=37)), L_max=720),
]


@pytest.mark.parametrize("spec", CASES, ids=[c.name for c in CASES])
def test_attention_matches_oracle(moelib, spec):
    rel = _check(moelib, spec)
    assert rel < 2e-3, rel


def test_attention_masks_rows_past_context(moelib):
    spec = synth.AttnSpec("poisoned", lens=(70, 1, 200), L_max=256)
    _check(moelib, spec, poison=True)


def test_attention_explicit_scale(moelib):
    _check(moelib, synth.AttnSpec("scale", lens=(333,), Hq=8, Hkv=2, D=128), scale=0.2)


def test_attention_repeatable(moelib):
    spec = synth.AttnSpec("repeat", lens=(20000, 3000), q_std=2.0)
    q, k, v, lens = synth.attn_inputs(spec, device=DEV)
    outs = [_run(moelib, q, k, v, lens) for _ in range(3)]
    assert all(np.array_equal(outs[0], o) for o in outs[1:])


def test_attention_full_size_32k(moelib):
    """The 32K-context workload (16 query heads, 2 KV heads, D = 256), every
    output against the oracle."""
    rel = _check(moelib, synth.ATTN_WORKLOADS["attn-decode-32k"])
    assert rel < 2e-3, rel


def test_attention_batch8_sampled(moelib):
    """The ragged 8-sequence workload at full size, run whole on the GPU;
    four of its sequences (the shortest, the longest and two others) checked
    one by one against the oracle."""
    spec = synth.ATTN_WORKLOADS["attn-decode-batch8"]
    q, k, v, lens = synth.attn_inputs(spec, device=DEV)
    got = _run(moelib, q, k, v, lens)
    for b in (2, 4, 6, 7):
        n = spec.lens[b]
        qb = q[b:b + 1].cpu()
        kb = k[b:b + 1, :, :n].cpu()
        vb = v[b:b + 1, :, :n].cpu()
        want = gqa_decode_attention(bits16(qb), bits16(kb), bits16(vb), [n])
        tol = _bound(qb, kb, vb, [n])
        assert np.all(np.abs(got[b:b + 1] - want) <= tol), b


def test_attention_invalid_length_sets_status(moelib):
    spec = synth.AttnSpec("bad-len", lens=(10, 20), Hq=4, Hkv=2, D=64)
    q, k, v, lens = synth.attn_inputs(spec, device=DEV)
    lens[1] = 21   # > L_max
    sh = moelib.attn_shape(2, 4, 2, 64, 20)
    ws = moelib.attn_alloc_workspace(sh, DEV)
    o = torch.full((2, 4, 64), 7.0, device=DEV)
    moelib.attn_decode(sh, q, k, v, lens, o, ws)
    assert moelib.status_read(ws[:4].view(torch.int32)) == moelib.MOE_ERR_INVALID_ARG
    assert torch.all(o == 7.0)


def test_attention_timeout_is_reported_not_hung(moelib):
    """One grid block issues none of its cache loads: its consumers' waits
    run out after a 20 ms limit, the block exits with nothing in flight, the
    call reports MOE_ERR_DEVICE_TIMEOUT, and the next normal call on the same
    context and workspace matches the oracle."""
    # 32768 positions = 1024 fixed blocks over 2 KV heads: every grid block has a run
    spec = synth.AttnSpec("stall", lens=(32768,), Hq=16, Hkv=2, D=128)
    q, k, v, lens = synth.attn_inputs(spec, device=DEV)
    sh = moelib.attn_shape(spec.B, spec.Hq, spec.Hkv, spec.D, spec.Lmax)
    ws = moelib.attn_alloc_workspace(sh, DEV)
    o = torch.zeros(spec.B, spec.Hq, spec.D, dtype=torch.float32, device=DEV)
    moelib.attn_test_stall(sh, q, k, v, lens, o, ws, stalled_block=3, timeout_ns=20_000_000)
    torch.cuda.synchronize()
    assert moelib.status_read(ws[:4].view(torch.int32)) == moelib.MOE_ERR_DEVICE_TIMEOUT
    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    got = _run(moelib, qc, kc, vc, lens.cpu())
    want = gqa_decode_attention(bits16(qc), bits16(kc), bits16(vc), spec.lens)
    assert np.all(np.abs(got - want) <= _bound(qc, kc, vc, spec.lens))
