"""The seeded input generator: published SplitMix64 values and determinism."""
import torch

import synth


def test_splitmix64_published_first_output():
    # SplitMix64 seeded with 0: first output 0xE220A8397B1DCDAF (the value
    # printed with the generator's reference implementation by Vigna).
    k = synth._s64(0)
    got = synth.draws(torch.tensor([k]), 0, 1)[0, 0].item() & ((1 << 64) - 1)
    assert got == 0xE220A8397B1DCDAF


def test_counter_based_slices_agree():
    keys = torch.tensor([synth._s64(synth.stream_key(7, 3))])
    whole = synth.draws(keys, 0, 100)
    part = synth.draws(keys, 40, 20)
    assert torch.equal(whole[:, 40:60], part)


def test_expert_slices_match_whole_layer():
    spec = synth.LayerSpec("t", T=4, H=128, I=64, E=16)
    L = synth.layer(spec)
    gu, dn = synth.expert_weights(spec, [5, spec.E])
    assert torch.equal(gu[0][0], L.gu[0][5]) and torch.equal(dn[2][0], L.dn[2][5])
    assert torch.equal(gu[1][1], L.sgu[1][0])


def test_distributions():
    spec = synth.LayerSpec("t", T=256, H=512, I=128, E=16)
    x = synth.activations(spec).float()
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1) < 0.02
    gu, _ = synth.expert_weights(spec, [0])
    c = gu[0].to(torch.int64) & 0xFFFFFFFF
    nib = torch.stack([(c >> (4 * i)) & 15 for i in range(8)]).flatten().float()
    assert abs(nib.mean() - 7.5) < 0.05 and nib.min() == 0 and nib.max() == 15
    s = gu[1].float()
    b = gu[2].float()
    assert (s >= 0).all() and abs(s.mean() - 0.02 * (2 / torch.pi) ** 0.5) < 1e-3
    assert abs((b + 8 * s).std() - 1e-3) < 2e-4


def test_attention_inputs_subset_and_shape():
    """A pair regenerated alone equals its slice of the whole cache; lengths
    and shapes follow the spec."""
    spec = synth.AttnSpec("t", lens=(3, 40, 0), Hq=8, Hkv=2, D=64)
    q, k, v, lens = synth.attn_inputs(spec)
    assert q.shape == (3, 8, 64) and k.shape == (3, 2, 40, 64) and v.shape == k.shape
    assert lens.tolist() == [3, 40, 0]
    one = synth.attn_cache(spec, synth.K_ATT_V, pairs=[(1, 1)])
    assert torch.equal(one[0], v[1, 1])
    assert not torch.equal(k, v)
    assert torch.isfinite(k.float()).all() and torch.isfinite(v.float()).all()


def test_gdn_inputs_shapes_and_ranges():
    spec = synth.GdnSpec("t", lens=(3, 0, 5), Hqk=2, Hv=4, Dk=8, Dv=8)
    q, k, v, gate, beta, state, offsets = synth.gdn_inputs(spec)
    assert q.shape == (8, 2, 8) and k.shape == q.shape and v.shape == (8, 4, 8)
    assert gate.shape == (8, 4) and beta.shape == (8, 4) and state.shape == (3, 4, 8, 8)
    assert offsets.tolist() == [0, 3, 3, 8]
    assert bool((gate <= 0).all()) and bool(((beta > 0) & (beta < 1)).all())
    assert not torch.equal(q, k)
