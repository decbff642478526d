"""The Gated DeltaNet scan through the C ABI on the GPU against the fp64 oracle.

Tolerance, from the arithmetic: the kernel runs the recurrence in fp32
(u = 2^-24), with a few roundings per state element and token (one fused
update, 16-term partial dots, an 8-way shuffle tree, rsqrt and exp within
2 ulp). The recurrence contracts by alpha <= 1 per token (about 0.96 on these
inputs), so an error made at one token fades within ~1 / (1 - alpha) = 25
tokens: the accumulated relative error stays near 25 x 10 u = 1.5e-5. The
tests ask rel-L2 <= 1e-4 and, per element, |error| <= 1e-3 x RMS, for the
outputs and the final states.
"""
import numpy as np
import pytest
import torch

import synth
from oracle.gated_deltanet import gated_delta_scan
from tests._util import bits16

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _run(moelib, spec, inputs, inplace=False):
    q, k, v, gate, beta, state, offsets = (x.to(DEV) for x in inputs)
    sh = moelib.gdn_shape(spec.B, spec.T, spec.Hqk, spec.Hv, spec.Dk, spec.Dv)
    o = torch.full((spec.T, spec.Hv, spec.Dv), float("nan"), device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = state if inplace else torch.full_like(state, float("nan"))
    moelib.gdn_scan(sh, q, k, v, gate, beta, offsets, state, out, o, status=st)
    assert moelib.status_read(st) == 0
    return o.cpu().numpy(), out.cpu().numpy()


def _oracle(inputs, heads=None):
    q, k, v, gate, beta, state, offsets = inputs
    if heads is not None:   # value heads only (each with its own query/key head)
        Hqk, Hv = q.shape[1], v.shape[1]
        per = Hv // Hqk
        outs = [_oracle((q[:, h // per:h // per + 1], k[:, h // per:h // per + 1], v[:, h:h + 1], gate[:, h:h + 1],
                         beta[:, h:h + 1], state[:, h:h + 1], offsets)) for h in heads]
        return np.concatenate([a for a, _ in outs], axis=1), np.concatenate([b for _, b in outs], axis=1)
    return gated_delta_scan(bits16(q), bits16(k), bits16(v), gate.double().numpy(), beta.double().numpy(),
                            state.double().numpy(), offsets.numpy())


def _close(got, want, what):
    if want.size == 0:
        return
    rms = float(np.sqrt(np.mean(want ** 2))) or 1.0
    err = np.abs(got - want)
    rel = float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-30))
    assert np.all(np.isfinite(got)), what
    assert rel <= 1e-4, (what, rel)
    assert float(err.max()) <= 1e-3 * rms, (what, float(err.max()), rms)


CASES = [
    synth.GdnSpec("decode-one", lens=(1,)),
    synth.GdnSpec("ragged-pack", lens=(5, 0, 17, 1), Hqk=4, Hv=8),
    synth.GdnSpec("long-300", lens=(300,), Hqk=2, Hv=4),
    synth.GdnSpec("heads-equal", lens=(40, 9), Hqk=4, Hv=4),
    synth.GdnSpec("heads-8-per-key", lens=(33,), Hqk=1, Hv=8),
    # at most two tokens per sequence on average: the short-sequence kernel
    synth.GdnSpec("short-pack", lens=(1, 2, 0, 1, 3, 1), Hqk=4, Hv=8),
    # long enough for the staged kernel, with a tail chunk of 5 and 8 + 3 tokens
    synth.GdnSpec("chunk-tails", lens=(37, 11), Hqk=2, Hv=4),
]


@pytest.mark.parametrize("spec", CASES, ids=[c.name for c in CASES])
def test_gdn_matches_oracle(moelib, spec):
    inputs = synth.gdn_inputs(spec)
    o, S = _run(moelib, spec, inputs)
    o_ref, S_ref = _oracle(inputs)
    _close(o, o_ref, "o")
    _close(S, S_ref, "state")


def test_gdn_state_in_place_and_repeatable(moelib):
    spec = synth.GdnSpec("inplace", lens=(64, 3), Hqk=2, Hv=4)
    inputs = synth.gdn_inputs(spec)
    o1, S1 = _run(moelib, spec, inputs)
    o2, S2 = _run(moelib, spec, inputs, inplace=True)
    assert np.array_equal(o1, o2) and np.array_equal(S1, S2)


def test_gdn_two_calls_equal_one(moelib):
    """A prompt run in two calls (the state handed on) gives the same outputs
    as one call, within the tolerance (the fp32 state is stored between)."""
    spec = synth.GdnSpec("split", lens=(50,), Hqk=2, Hv=4)
    q, k, v, gate, beta, state, offsets = synth.gdn_inputs(spec)
    o, S = _run(moelib, spec, (q, k, v, gate, beta, state, offsets))
    a = synth.GdnSpec("a", lens=(20,), Hqk=2, Hv=4)
    b = synth.GdnSpec("b", lens=(30,), Hqk=2, Hv=4)
    oa, Sa = _run(moelib, a, (q[:20], k[:20], v[:20], gate[:20], beta[:20], state, torch.tensor([0, 20], dtype=torch.int32)))
    ob, Sb = _run(moelib, b, (q[20:], k[20:], v[20:], gate[20:], beta[20:], torch.from_numpy(Sa),
                              torch.tensor([0, 30], dtype=torch.int32)))
    assert np.array_equal(np.concatenate([oa, ob]), o) and np.array_equal(Sb, S)


def test_gdn_full_size_prefill_sampled_heads(moelib):
    """The 4096-token prompt through 32 value heads, run whole; three value
    heads (first, middle, last) checked against the oracle, outputs and state."""
    spec = synth.GDN_WORKLOADS["gdn-prefill-4096"]
    inputs = synth.gdn_inputs(spec)
    o, S = _run(moelib, spec, inputs)
    heads = [0, 17, 31]
    o_ref, S_ref = _oracle(inputs, heads)
    _close(o[:, heads], o_ref, "o")
    _close(S[:, heads], S_ref, "state")


def test_gdn_full_size_decode(moelib):
    """64 sequences one token each, every head, against the oracle."""
    spec = synth.GDN_WORKLOADS["gdn-decode-b64"]
    inputs = synth.gdn_inputs(spec)
    o, S = _run(moelib, spec, inputs)
    o_ref, S_ref = _oracle(inputs)
    _close(o, o_ref, "o")
    _close(S, S_ref, "state")


@pytest.mark.parametrize("lens", [(4, 4), (1, 1)], ids=["staged", "short"])
def test_gdn_bad_offsets_pass_state_through(moelib, lens):
    spec = synth.GdnSpec("bad", lens=lens, Hqk=2, Hv=4)
    q, k, v, gate, beta, state, offsets = (x.to(DEV) for x in synth.gdn_inputs(spec))
    offsets[1] = spec.T + 1   # > T for sequence 0, and sequence 1 runs backwards
    sh = moelib.gdn_shape(2, spec.T, 2, 4)
    out = torch.empty_like(state)
    o = torch.zeros(spec.T, 4, 128, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    moelib.gdn_scan(sh, q, k, v, gate, beta, offsets, state, out, o, status=st)
    assert moelib.status_read(st) == moelib.MOE_ERR_INVALID_ARG
    assert torch.equal(out, state)
