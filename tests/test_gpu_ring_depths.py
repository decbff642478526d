"""Results of the tensor-core expert GEMM do not depend on its ring depths.

The MMAs of an item accumulate its 64-K stages in the same order whatever the
depths of the code, A and B rings, so a build with other depths must give the
same bits. A race between the dequantisation, gather and MMA warps over a
ring slot (a slot rewritten before the MMAs that read it were done) would
show up as differing values, most readily with deeper rings, where the
dequantisation runs further ahead of the completed MMAs. The default build
has a 3-deep A ring in the gate/up GEMM and a 4-deep one in the down GEMM;
builds with 4 and 3 (libbgmoe_a4d3b4.so) and with 5 and 5 and shallower code
and B rings (libbgmoe_a5d5b3c2.so) run the 4096-token and the Zipf-skewed
512-token layers three times each in their own processes, and every output
must equal the default build's bit for bit."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RUN = r"""
import hashlib, sys
import numpy as np, torch
import bit_grouped_expert_moe_gb300 as m
if sys.argv[1] != "default":
    m.LIB_PATH = sys.argv[1]
import synth
from tests import parity
dev = torch.device("cuda:0")
m.lib()
for name, bm in (("prefill-4096", 128), ("prefill-zipf-512", 64)):
    spec = synth.WORKLOADS[name]
    L = parity.device_layer(spec, 0, dev)
    x = synth.activations(spec, device=dev)
    for rep in range(3):
        y, _ = parity.gpu_forward(m, spec, L, x, bm, path=m.PATH_TENSOR_CORE)
        print("HASH", name, hashlib.sha256(np.ascontiguousarray(y).view(np.uint32).tobytes()).hexdigest())
"""


def _hashes(lib):
    r = subprocess.run([sys.executable, "-c", RUN, lib], cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    out = {}
    for line in r.stdout.splitlines():
        if line.startswith("HASH "):
            _, name, h = line.split()
            out.setdefault(name, []).append(h)
    assert set(out) == {"prefill-4096", "prefill-zipf-512"}, r.stdout[-2000:]
    return out


def test_ring_depths_give_identical_results():
    from bit_grouped_expert_moe_gb300 import _build
    want = _hashes("default")
    for name, hs in want.items():
        assert len(set(hs)) == 1, (name, "the default build is not repeatable")
    for variant in _build.RING_VARIANTS:
        lib = _build.build_ring_variant(variant)
        got = _hashes(lib)
        for name in want:
            assert got[name] == want[name], (variant, name)
