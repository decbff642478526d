"""CPU oracle for one bit-grouped-expert MoE layer (test infrastructure only).

This package is the plain, slow, fp64 statement of what the layer computes. It
exists to check the CUDA library and to serve as the timed CPU baseline; only
the tests, the smoke check and the benchmark's CPU legs may import it. The
product path never calls it and shares no code with it.

The MoE layer is stated twice, independently: in plain C++ (`moe_ref.cpp`,
reached through `cpp.py`, which only marshals arguments), the oracle the GPU
parity tests, the smoke check and the benchmark's CPU legs use; and in numpy
(`moe.py`), which the C++ one is cross-checked against. The same pins run on
both, and planted mistakes in either make a pin fail. The attention and
Gated DeltaNet oracles are numpy.

Sources (three web pages on Perplexity's Lily engine for Qwen3.6-35B-A3B):
  [dothoosh]  "Perplexity Lily: 1.35x faster decode for Qwen3.6 on Apple
              silicon", dothoosh.com
  [aikraft]   "Perplexity open-sources Lily, a Rust/Metal inference engine for
              Qwen3.6", aikraft.ru
  [droneth]   Lily inference engine article, droneth.or.th

Every function in `moe.py` names the section it follows. Where the pages are
silent (affine formula, nibble order, softmax/top-k order, shared-expert gate,
activation), the reading taken is stated in that function's docstring.
"""
from .moe import (  # noqa: F401
    bf16_bits_to_f64,
    dequant,
    router_logits,
    select_top_k,
    route,
    routing_tables,
    swiglu_expert,
    moe_forward,
    topk_gap,
    rms_norm,
)
from .attention import gqa_decode_attention  # noqa: F401,E402
from .gated_deltanet import gated_delta_scan  # noqa: F401,E402
