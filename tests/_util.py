"""Marshalling between the seeded torch inputs and the oracle's numpy arrays
(raw bf16 bit patterns as uint16, packed codes as uint32)."""
from __future__ import annotations

import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def bits16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def u32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy().view(np.uint32)


def f32(t):
    return None if t is None else t.detach().cpu().float().numpy()


def bf16_from_f64(v) -> np.ndarray:
    """Round fp64 values to bf16 bit patterns (via fp32, RNE both times)."""
    t = torch.as_tensor(np.asarray(v, dtype=np.float64)).to(torch.float32).to(torch.bfloat16)
    return bits16(t)


def expert_fn_from_layer(L, E):
    """expert_fn(e) for oracle.moe_forward from a synth.Layer."""
    def fn(e):
        if e == E:
            if L.sgu is None:
                return None
            gu, dn = L.sgu, L.sdn
            i = 0
        else:
            gu, dn = L.gu, L.dn
            i = e
        return (u32(gu[0][i]), bits16(gu[1][i]), bits16(gu[2][i]),
                u32(dn[0][i]), bits16(dn[1][i]), bits16(dn[2][i]))
    return fn


def expert_fn_lazy(spec, layer_idx=0):
    """expert_fn(e) that regenerates expert e's weights on the CPU on demand."""
    import synth

    def fn(e):
        if e == spec.E and not spec.shared:
            return None
        gu, dn = synth.expert_weights(spec, [e], layer_idx, "cpu")
        return (u32(gu[0][0]), bits16(gu[1][0]), bits16(gu[2][0]),
                u32(dn[0][0]), bits16(dn[1][0]), bits16(dn[2][0]))
    return fn


def read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([part.split() for part in line.split(":")])
    return rows
