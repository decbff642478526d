"""The fp16 operand range of the expert paths, at its edges.

The expert products take fp16 operands: weights rounded once from
scale * q + bias with scale and bias converted from bf16, x converted from
bf16, h and o stored as fp16. fp16 keeps 11 significant bits from 2^-14 up to
65504 and a fixed step of 2^-24 below. Each expert path (fused decode, tensor
cores, GEMV) is run on
  * bf16 scales spread log-uniformly over 1e-7 .. 1e-4 (fp16 subnormals below
    6.1e-5), with the bias recipe of the workloads (-8 scale + N(0, 1e-3)) and
    with a bias that follows the scale (-8 scale (1 + N(0, 0.01))), where the
    weights themselves are subnormal: the tolerance holds (the fp16 weights
    are formed as fma(q 2^-14, scale 2^14, bias), rounded once);
  * x eight times the workloads' scale, h and o still inside fp16: the
    tolerance holds;
  * one x element near 65504 (h overflows), one past it (x overflows), and x
    a hundred times the workloads' scale (h overflows): MOE_ERR_RANGE;
  * subnormal weights at the workloads' x, where o falls to ~1e-8, under the
    2^-16 floor: MOE_ERR_RANGE;
  * a scale of 4, past the fp16 weights' scale * 2^14: MOE_ERR_RANGE on the
    paths with fp16 weights, a valid result on the GEMV path (fp32 weights)."""
import numpy as np
import pytest
import torch

import synth
from tests import parity

pytestmark = pytest.mark.gpu

# (label, T, H, I, expert path): a decode token on the fused kernel, the tiny
# workload's shape on tensor cores, three decode tokens on the GEMV path.
PATHS = [("fused", 1, 2048, 512, "PATH_FUSED_DECODE"), ("tensor", 64, 512, 128, "PATH_TENSOR_CORE"),
         ("gemv", 3, 512, 128, "PATH_GEMV")]
IDS = [p[0] for p in PATHS]


def _bf16(v64):
    return v64.to(torch.float32).to(torch.bfloat16)


def _spread_scales(L, seed, bias):
    """Every expert matrix of the layer, in place: scales log-uniform in
    [1e-7, 1e-4]; biases -8 scale + N(0, 1e-3) ("workload") or
    -8 scale (1 + N(0, 0.01)) ("follows")."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    for mats in (L.gu, L.dn, L.sgu, L.sdn):
        if mats is None:
            continue
        sc, bi = mats[1], mats[2]
        u = torch.rand(sc.shape, generator=g, dtype=torch.float64)
        s = _bf16(torch.exp(np.log(1e-7) + u * (np.log(1e-4) - np.log(1e-7)))).to(torch.float64)
        z = torch.randn(sc.shape, generator=g, dtype=torch.float64)
        b = -8.0 * s + 1e-3 * z if bias == "workload" else -8.0 * s * (1.0 + 0.01 * z)
        sc.copy_(s.to(torch.float32).to(torch.bfloat16))
        bi.copy_(_bf16(b))


def _run(moelib, spec, L, x, path):
    return parity.gpu_forward(moelib, spec, L, x, 16, path=getattr(moelib, path), check_status=False)


def _check_bar(moelib, spec, L, x, path):
    (y, ro), status = _run(moelib, spec, L, x, path)
    assert status == 0, moelib.status_string(status)
    y_ref, ids_ref, w_ref, g_ref, logits = parity.oracle_forward(spec, L, x)
    ids = ro["ids"][: spec.T * spec.top_k].reshape(spec.T, spec.top_k)
    excl = parity.check_ids(ids, ids_ref, logits, spec.top_k)
    return parity.check_y(y, y_ref, excl)


# x scale per path for the workload-bias case: the weights are then ~1e-3
# (the bias noise), so h ~ H * x^2 * 1e-6 and o ~ sqrt(I) * h * 1e-3. At
# H = 2048, I = 512 the workloads' x gives h ~ 1e-3 and o ~ 2e-5 (subnormal,
# every row's largest value above 3e-5); at H = 512, I = 128 that x would put
# o near 3e-6, under the floor, so x is ten times larger there (o ~ 3e-4).
SPREAD_X = {"fused": 1, "tensor": 10, "gemv": 10}


@pytest.mark.parametrize("label,T,H,I,path", PATHS, ids=IDS)
def test_spread_scales_with_workload_bias_meet_the_bar(moelib, cuda_dev, label, T, H, I, path):
    spec = synth.LayerSpec("range-scales", T=T, H=H, I=I, seed=20260051)
    L = parity.device_layer(spec, 0, cuda_dev)
    _spread_scales(L, 7, "workload")
    x = _bf16(synth.activations(spec, device=cuda_dev).to(torch.float64) * SPREAD_X[label])
    _check_bar(moelib, spec, L, x, path)


@pytest.mark.parametrize("label,T,H,I,path", PATHS, ids=IDS)
def test_subnormal_weights_meet_the_bar(moelib, cuda_dev, label, T, H, I, path):
    """Weights ~1e-4 (scale and bias fp16 subnormals on every group below
    6.1e-5), x a hundred times the workloads' scale so that h (~0.04 to 0.2)
    and o (~5e-5 to 5e-4) stay above the floor: the weights' own rounding
    (about 1e-3 of a product) stays inside the tolerance."""
    spec = synth.LayerSpec("range-subnormal-w", T=T, H=H, I=I, seed=20260055)
    L = parity.device_layer(spec, 0, cuda_dev)
    _spread_scales(L, 8, "follows")
    x = _bf16(synth.activations(spec, device=cuda_dev).to(torch.float64) * 100)
    _check_bar(moelib, spec, L, x, path)


@pytest.mark.parametrize("label,T,H,I,path", PATHS, ids=IDS)
def test_large_x_within_range_meets_the_bar(moelib, cuda_dev, label, T, H, I, path):
    """x eight times the workloads' scale: |h| grows about 64-fold (to a few
    thousand at most) and stays inside fp16."""
    spec = synth.LayerSpec("range-x8", T=T, H=H, I=I, seed=20260052)
    L = parity.device_layer(spec, 0, cuda_dev)
    x = _bf16(synth.activations(spec, device=cuda_dev).to(torch.float64) * 8)
    _check_bar(moelib, spec, L, x, path)


@pytest.mark.parametrize("value", [6e4, 1e5], ids=["near", "past"])
@pytest.mark.parametrize("label,T,H,I,path", PATHS, ids=IDS)
def test_x_near_and_past_fp16_range_is_reported(moelib, cuda_dev, label, T, H, I, path, value):
    """One x element of 6e4 (bf16 59904: x itself fits, the products it
    enters push h far past 65504) or of 1e5 (bf16 99840: inf in fp16)."""
    spec = synth.LayerSpec("range-xbig", T=T, H=H, I=I, seed=20260053)
    L = parity.device_layer(spec, 0, cuda_dev)
    x = synth.activations(spec, device=cuda_dev)
    x[0, 5] = value
    _, status = _run(moelib, spec, L, x, path)
    assert status == moelib.MOE_ERR_RANGE, moelib.status_string(status)


@pytest.mark.parametrize("label,T,H,I,path", PATHS, ids=IDS)
def test_h_past_fp16_range_is_reported(moelib, cuda_dev, label, T, H, I, path):
    """x a hundred times the workloads' scale (|x| up to a few hundred, well
    inside fp16): gate and up reach ~10^3, so |h| passes 65504."""
    spec = synth.LayerSpec("range-h", T=T, H=H, I=I, seed=20260054)
    L = parity.device_layer(spec, 0, cuda_dev)
    x = _bf16(synth.activations(spec, device=cuda_dev).to(torch.float64) * 100)
    assert float(x.float().abs().max()) < 65504
    _, status = _run(moelib, spec, L, x, path)
    assert status == moelib.MOE_ERR_RANGE, moelib.status_string(status)


@pytest.mark.parametrize("label,T,H,I,path", PATHS, ids=IDS)
def test_values_under_the_fp16_floor_are_reported(moelib, cuda_dev, label, T, H, I, path):
    """Subnormal weights (~1e-4) at the workloads' x: h ~ 5e-6 to 2e-5 and
    o ~ 1e-8, under the 2^-16 floor where fp16's fixed step costs more than
    2^-9."""
    spec = synth.LayerSpec("range-floor", T=T, H=H, I=I, seed=20260056)
    L = parity.device_layer(spec, 0, cuda_dev)
    _spread_scales(L, 9, "follows")
    _, status = _run(moelib, spec, L, synth.activations(spec, device=cuda_dev), path)
    assert status == moelib.MOE_ERR_RANGE, moelib.status_string(status)


@pytest.mark.parametrize("label,T,H,I,path", PATHS, ids=IDS)
def test_zero_input_is_not_a_range_error(moelib, cuda_dev, label, T, H, I, path):
    """x = 0: h and o are exactly zero, which fp16 holds exactly; y = 0."""
    spec = synth.LayerSpec("range-zero", T=T, H=H, I=I, seed=20260057)
    L = parity.device_layer(spec, 0, cuda_dev)
    x = torch.zeros(T, H, dtype=torch.bfloat16, device=cuda_dev)
    (y, _), status = _run(moelib, spec, L, x, path)
    assert status == 0, moelib.status_string(status)
    assert not np.any(y)


@pytest.mark.parametrize("label,T,H,I,path", PATHS, ids=IDS)
def test_scale_of_four_is_reported_on_fp16_weights(moelib, cuda_dev, label, T, H, I, path):
    """Group 0 of gate row 0 in every expert gets scale 4 (bf16 exact):
    scale * 2^14 = 65536 is past fp16, so the fused and tensor-core paths
    report MOE_ERR_RANGE; the GEMV path, which dequantises in fp32, meets the
    tolerance."""
    spec = synth.LayerSpec("range-scale4", T=T, H=H, I=I, seed=20260058)
    L = parity.device_layer(spec, 0, cuda_dev)
    for mats in (L.gu, L.sgu):
        mats[1][:, 0, 0] = 4.0
        mats[2][:, 0, 0] = -32.0
    x = synth.activations(spec, device=cuda_dev)
    if label == "gemv":
        _check_bar(moelib, spec, L, x, path)
    else:
        _, status = _run(moelib, spec, L, x, path)
        assert status == moelib.MOE_ERR_RANGE, moelib.status_string(status)
