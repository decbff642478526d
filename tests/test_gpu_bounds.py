"""The bounds-checking debug build (BGMOE_BOUNDS_CHECK, libbgmoe_bounds.so):
every index the kernels read from a device-written table is checked before
use and an out-of-range one is reported as MOE_ERR_BOUNDS instead of being
followed. Parity cases at tiny shapes (T = 1..3, 64, odd group counts, every
expert path) run through it in a separate process and must report no error
and match the oracle, routing tables (an invertible permutation) included."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RUN = r"""
import torch
import bit_grouped_expert_moe_gb300 as m
from bit_grouped_expert_moe_gb300 import _build
m.LIB_PATH = _build.DEBUG_LIB
import synth
from tests.test_gpu_parity import _run_and_check
dev = torch.device("cuda:0")
m.lib()
_run_and_check(m, dev, synth.WORKLOADS["tiny"])
for T in (1, 2, 3):
    spec = synth.LayerSpec("bounds-ragged", T=T, H=512, I=128, seed=20260061)
    for path in (m.PATH_GEMV, m.PATH_TENSOR_CORE):
        _run_and_check(m, dev, spec, path=path)
_run_and_check(m, dev, synth.LayerSpec("bounds-odd", T=45, H=1536, I=384, E=32, top_k=4, seed=20260062),
               block_m=32, path=m.PATH_TENSOR_CORE)
_run_and_check(m, dev, synth.LayerSpec("bounds-odd", T=45, H=384, I=320, E=32, top_k=4, seed=20260062),
               block_m=16, path=m.PATH_GEMV)
for T in (1, 4):
    spec = synth.LayerSpec("bounds-fused", T=T, H=2048, I=512, seed=20260063)
    _run_and_check(m, dev, spec, path=m.PATH_FUSED_DECODE)
print("bounds build ok")
"""


def test_bounds_checked_build_reports_nothing_and_matches_the_oracle():
    from bit_grouped_expert_moe_gb300 import _build
    _build.build_bounds_checked()
    r = subprocess.run([sys.executable, "-c", RUN], cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0 and "bounds build ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]
