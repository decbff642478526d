"""The C++ oracle (oracle/moe_ref.cpp): the MoE pins run against it, each
planted mistake compiled into it makes a pin fail, and it agrees with the
numpy oracle (two independent statements of the same definitions) on the
workloads' shapes. No GPU needed."""
import numpy as np
import pytest
import torch

import oracle.cpp as C
import oracle.moe as M
import synth
import tests.oracle_pins as P
from tests import parity
from tests._util import bits16

MOE_PINS = [p for p in P.PINS if not p.__name__.startswith(("pin_attn", "pin_gdn"))]


@pytest.mark.parametrize("pin", MOE_PINS, ids=[p.__name__ for p in MOE_PINS])
def test_pin_on_cpp_oracle(pin, monkeypatch):
    monkeypatch.setattr(P, "M", C.default())
    pin()


# BGREF_MUTANT values planted in moe_ref.cpp and what each one gets wrong.
MUTANTS = {
    1: "nibble order reversed inside a word",
    2: "bias subtracted instead of added",
    3: "ties go to the higher expert index",
    4: "silu with the sign of the exponent flipped",
    5: "gate and up swapped",
    6: "softmax normalised over all experts",
    7: "shared gate through tanh instead of the sigmoid",
    8: "shared expert added without its gate",
    9: "shared expert missing from the routing counts",
    10: "router bias dropped",
    11: "scale and bias per 32 weights instead of 64",
    12: "RMS norm without the square root",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=[f"{k}-{v}" for k, v in sorted(MUTANTS.items())])
def test_planted_mistake_in_cpp_oracle_is_caught(mutant, tmp_path, monkeypatch):
    ref = C.load(C.compile_ref(str(tmp_path / f"libbgref_m{mutant}.so"), mutant=mutant, force=True))
    monkeypatch.setattr(P, "M", ref)
    failed = []
    for pin in MOE_PINS:
        try:
            pin()
        except Exception:
            failed.append(pin.__name__)
    assert failed, f"no pin caught mutant {mutant} ({MUTANTS[mutant]})"


def _agree(spec, tokens=None, layer_idx=0):
    L = synth.layer(spec, layer_idx, "cpu")
    x = synth.activations(spec)
    fn = parity.layer_expert_fn(L, spec.E)
    bias = None if L.bias is None else L.bias.numpy()
    wsg = None if L.wsg is None else bits16(L.wsg)
    args = (bits16(x), bits16(L.wr), bias, wsg, spec.top_k, fn)
    yc, ic, wc, gc, lc = C.moe_forward(*args, tokens=tokens)
    yn, i_n, wn, gn, ln = M.moe_forward(*args, tokens=tokens)
    assert np.array_equal(ic, i_n)
    assert np.allclose(lc, ln, rtol=0, atol=1e-12)
    assert np.allclose(wc, wn, rtol=1e-12, atol=1e-15)
    if gn is not None:
        assert np.allclose(gc, gn, rtol=1e-12, atol=0)
    assert np.linalg.norm(yc - yn) <= 1e-12 * np.linalg.norm(yn)
    tc, tn = C.routing_tables(ic, spec.E, 16, spec.shared), M.routing_tables(i_n, spec.E, 16, spec.shared)
    for k in tn:
        assert np.array_equal(np.asarray(tc[k]), np.asarray(tn[k])), k


def test_agrees_with_numpy_oracle_tiny():
    _agree(synth.WORKLOADS["tiny"])


def test_agrees_with_numpy_oracle_decode():
    _agree(synth.WORKLOADS["decode-t4"], layer_idx=7)


def test_agrees_with_numpy_oracle_skewed_samples():
    _agree(synth.WORKLOADS["prefill-zipf-512"], tokens=np.array([0, 17, 300, 511]))
    spec = synth.WORKLOADS["long-skew-16384"]
    _agree(synth.LayerSpec(spec.name, T=64, H=spec.H, I=spec.I, bias=spec.bias, hot_logit=spec.hot_logit,
                           seed=spec.seed), tokens=np.array([1, 40, 63]))


def test_agrees_with_numpy_oracle_other_shapes():
    for E, K, shared, H, I in [(16, 2, False, 128, 64), (8, 1, True, 64, 64), (32, 4, True, 384, 320)]:
        _agree(synth.LayerSpec("shape", T=9, H=H, I=I, E=E, top_k=K, shared=shared, seed=20260012))


def test_rms_norm_agrees():
    rng = np.random.default_rng(3)
    r = bits16(synth.to_bf16(torch.from_numpy(rng.standard_normal((7, 320)) * 3)))
    g = bits16(synth.to_bf16(torch.from_numpy(rng.uniform(0.5, 2, 320))))
    for gain in (None, g):
        assert np.allclose(C.rms_norm(r, 1e-6, gain), M.rms_norm(r, 1e-6, gain), rtol=1e-14, atol=0)


def test_routing_tables_agree_on_random_ids():
    rng = np.random.default_rng(4)
    for T, E, K, bm, shared in [(1, 8, 8, 16, True), (37, 256, 8, 16, True), (100, 32, 4, 128, False),
                                (64, 256, 8, 64, True)]:
        ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
        tc, tn = C.routing_tables(ids, E, bm, shared), M.routing_tables(ids, E, bm, shared)
        for k in tn:
            assert np.array_equal(np.asarray(tc[k]), np.asarray(tn[k])), (T, E, k)
