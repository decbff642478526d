#!/usr/bin/env python3
"""Benchmark of the GB300 MoE layer (one JSON line on stdout).

Default workload: decode, T = 1 token through 40 chained MoE layers with
distinct weights (H = 2048, I = 512, E = 256 top-8 + shared, 4-bit group-64
weights, 18.2 GB of weights, far larger than L2; layer l+1 reads layer l's
x + y), one step = one pass over the 40 layers; the metric is microseconds
per layer. The same run adds a prefill-4096 record (tokens/s). --workload picks another
shape (prefill-zipf-512, prefill-4096, long-skew-16384, decode-t4, tiny),
or decode attention over a bf16 KV cache (attn-decode-32k, -64k, -128k,
attn-decode-batch8: 16 query heads on 2 KV heads, D = 256, 10 layers), or
the Gated DeltaNet scan (gdn-prefill-4096, gdn-decode-b64).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (tests' fp64 reference) on the host
cores, on a bounded sample of the same workload. Under torchrun (N > 1)
every rank runs an independent replica (the layer has no exchange step) and
rank 0 prints the line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "MoE-layer tokens/s (prefill) & µs/layer (decode); % of BF16 TC / HBM roofline"

# DRAM bytes per launch of the dominant kernel (dram__bytes_read.sum +
# dram__bytes_write.sum from one ncu capture), with the SHA-256 of the
# kernel's sources at capture time: the figure is reported only while the
# sources are unchanged, null otherwise.
CSRC = os.path.join(os.path.dirname(os.path.abspath(__file__)), "bit_grouped_expert_moe_gb300", "csrc")
PROFILED_TRAFFIC = {
    ("fused_decode_layer", "decode-t1"): dict(
        bytes=17084416 + 2048,
        sources={"decode.cu": "8a228a712d37d2c49389418197e855d6786da04591294aecee6811eff5f4dbf7",
                 "tc_ptx.cuh": "91cf5c0848386f35a604cc2a0ae91ff9fe4fb195eb7e41d989b49257ac65cd7d",
                 "common.cuh": "50bd4e54a129b106017f859e988153a6e556e0b58fca272f8d3712d8150c02c4"}),
    ("expert_gate_up", "prefill-zipf-512"): dict(
        bytes=132567040 + 4606720,
        sources={"gemm_tc.cu": "23068ea0388ed111f7d85c44483b2fe8cac112c3d26632fee35e3ee16cb1b6cc",
                 "tc_ptx.cuh": "91cf5c0848386f35a604cc2a0ae91ff9fe4fb195eb7e41d989b49257ac65cd7d",
                 "common.cuh": "50bd4e54a129b106017f859e988153a6e556e0b58fca272f8d3712d8150c02c4"}),
    ("expert_gate_up", "prefill-4096"): dict(
        bytes=415157504 + 28314880,
        sources={"gemm_tc.cu": "23068ea0388ed111f7d85c44483b2fe8cac112c3d26632fee35e3ee16cb1b6cc",
                 "tc_ptx.cuh": "91cf5c0848386f35a604cc2a0ae91ff9fe4fb195eb7e41d989b49257ac65cd7d",
                 "common.cuh": "50bd4e54a129b106017f859e988153a6e556e0b58fca272f8d3712d8150c02c4"}),
    ("attn_block_kernel", "attn-decode-32k"): dict(
        bytes=67168768 + 154112,
        sources={"attention.cu": "67f37e5399b9ed695e74164575c004b001aab86a4e69cf8343d4638d21e0a4c6",
                 "tc_ptx.cuh": "91cf5c0848386f35a604cc2a0ae91ff9fe4fb195eb7e41d989b49257ac65cd7d",
                 "common.cuh": "50bd4e54a129b106017f859e988153a6e556e0b58fca272f8d3712d8150c02c4"}),
    ("gdn_scan_kernel", "gdn-prefill-4096"): dict(
        bytes=70283776 + 24791040,
        sources={"gdn.cu": "0e6cd58b752512d1bf7c2fc631398474c866923587ccd2ea93e0e780e54f56c4",
                 "common.cuh": "50bd4e54a129b106017f859e988153a6e556e0b58fca272f8d3712d8150c02c4"}),
    ("gdn_short_kernel", "gdn-decode-b64"): dict(
        bytes=135301376 + 81671424,
        sources={"gdn.cu": "0e6cd58b752512d1bf7c2fc631398474c866923587ccd2ea93e0e780e54f56c4",
                 "common.cuh": "50bd4e54a129b106017f859e988153a6e556e0b58fca272f8d3712d8150c02c4"}),
    ("expert_gate_up", "long-skew-16384"): dict(
        bytes=328094976 + 14594048,
        sources={"gemm_tc.cu": "23068ea0388ed111f7d85c44483b2fe8cac112c3d26632fee35e3ee16cb1b6cc",
                 "tc_ptx.cuh": "91cf5c0848386f35a604cc2a0ae91ff9fe4fb195eb7e41d989b49257ac65cd7d",
                 "common.cuh": "50bd4e54a129b106017f859e988153a6e556e0b58fca272f8d3712d8150c02c4"}),
}


def profiled_traffic(kernel, workload):
    import hashlib
    rec = PROFILED_TRAFFIC.get((kernel, workload))
    if rec is None:
        return None
    for name, sha in rec["sources"].items():
        with open(os.path.join(CSRC, name), "rb") as f:
            if hashlib.sha256(f.read()).hexdigest() != sha:
                return None
    return rec["bytes"]
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
BYTES_PER_WEIGHT = 0.5 + 4.0 / 64.0  # 4-bit code + bf16 scale + bf16 bias per 64


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


# ------------------------------------------------------------ distributed --

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest of every rank's value (the job's time is its slowest rank)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": float(rows[0][2]) if rows[0][2].replace(".", "").isdigit() else None,
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------- workload --

class Workload:
    """Device-resident inputs of one workload and the per-step launch list."""

    def __init__(self, m, spec, device, block_m, rank=0):
        self.m, self.spec, self.dev = m, spec, device
        self.layers = spec.layers
        self.T = spec.chunk if spec.chunk else spec.T
        self.calls = (spec.T // spec.chunk) if spec.chunk else 1
        self.shape = m.make_shape(self.T, spec.H, spec.I, spec.E, spec.top_k, spec.shared, block_m)
        self.L = [synth.layer(spec, li, device) for li in range(self.layers)]
        self.experts = []
        for L in self.L:
            routed = ((L.gu[0], L.gu[1], L.gu[2]), (L.dn[0], L.dn[1], L.dn[2]))
            shared = None if L.sgu is None else ((L.sgu[0], L.sgu[1], L.sgu[2]), (L.sdn[0], L.sdn[1], L.sdn[2]))
            self.experts.append((routed, shared))
        # token rows (replica r of a multi-rank job takes its own rows)
        self.x = synth.activations(spec, device=device, start=rank * spec.T).view(self.calls, self.T, spec.H)
        self.ws = m.alloc_workspace(self.shape, device)
        self.y = torch.empty(self.layers, self.calls, self.T, spec.H, dtype=torch.float32, device=device)
        self.route = [m.alloc_route_out(self.shape, device) for _ in range(self.layers)]
        # Decode chains its layers as pre-norm blocks (moe_forward_residual):
        # layer l reads the residual row r_l that layer l-1 wrote
        # (r_l = bf16(r_{l-1} + y_{l-1})) and runs on RMSNorm(r_l), as a
        # model's stack of layers does; x is layer 0's residual row.
        self.chain = torch.empty(self.layers, self.T, spec.H, dtype=torch.bfloat16, device=device) \
            if self.fused() else None

    def fused(self):
        return self.T <= 4  # the library runs decode-sized calls as a prelude + the fused decode kernel

    def launches_per_step(self):
        return (2 if self.fused() else 5) * self.layers * self.calls

    def layer_input(self, li, c):
        return self.x[c] if (self.chain is None or li == 0) else self.chain[li - 1]

    def call(self, li, c, events=None):
        L = self.L[li]
        routed, shared = self.experts[li]
        if events is None and self.chain is not None:
            self.m.forward_residual(self.shape, self.layer_input(li, c), L.wr, L.bias, routed, shared, L.wsg,
                                    self.y[li, c], self.chain[li], self.ws, route_out=self.route[li])
        elif events is None:
            self.m.forward(self.shape, self.x[c], L.wr, L.bias, routed, shared, L.wsg, self.y[li, c], self.ws,
                           route_out=self.route[li])
        else:
            # the diagnostic event pass runs every layer on the workload's own
            # input (plain moe_forward semantics)
            self.m.forward_timed(self.shape, self.x[c], L.wr, L.bias, routed, shared, L.wsg,
                                 self.y[li, c], self.ws, events=events, route_out=self.route[li])

    def step(self):
        for c in range(self.calls):
            for li in range(self.layers):
                self.call(li, c)

    # -- algorithmic work (counted from the routing of the last call) --
    def work(self):
        s = self.spec
        H, I, E = s.H, s.I, s.E
        wbytes_expert = 3 * H * I * BYTES_PER_WEIGHT
        router_bytes = (E + (1 if s.shared else 0)) * H * 2
        tot_bytes = gu_bytes = fused_bytes = gu_flops = 0.0
        distinct = []
        for li in range(self.layers):
            counts = self.route[li]["counts"].cpu()
            d = int((counts[:E] > 0).sum())
            distinct.append(d)
            n_exp = d + (1 if s.shared else 0)
            per_call = n_exp * wbytes_expert + router_bytes + self.T * H * 2 + self.T * H * 4
            tot_bytes += per_call * self.calls
            gu_bytes += n_exp * (2 * I * H * BYTES_PER_WEIGHT) * self.calls
            gu_flops += (s.top_k + (1 if s.shared else 0)) * self.T * 2 * (2 * I) * H * self.calls
            # the fused kernel also reads the router weights (it computes the logits itself)
            fused_bytes += (n_exp * wbytes_expert + router_bytes + self.T * H * 6 + self.T * (E + 1) * 8) * self.calls
        flops_tok = 2 * H * E + s.top_k * 6 * H * I + (6 * H * I if s.shared else 0) + (2 * H if s.shared else 0)
        return dict(bytes_per_step=tot_bytes, gate_up_bytes_per_step=gu_bytes, fused_bytes_per_step=fused_bytes,
                    gate_up_flops_per_step=gu_flops,
                    flops_per_step=flops_tok * self.T * self.calls * self.layers,
                    distinct_experts_mean=sum(distinct) / len(distinct))


def time_region(fn, steps, stream):
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end)


def capture(fn):
    """One CUDA graph of everything fn() enqueues (the library's launches are
    captured from the current stream)."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm the launch path (attribute setup) outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def stage_times(W, steps):
    """Per-kernel averages (ms) from events recorded between the kernels of
    every call (event nodes inside a graph of one step)."""
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(W.layers * W.calls)]
    for e6 in ev:           # torch creates the CUDA event at its first record
        for e in e6:
            e.record()
    torch.cuda.synchronize()

    def timed_step():
        k = 0
        for c in range(W.calls):
            for li in range(W.layers):
                W.call(li, c, events=[e.cuda_event for e in ev[k]])
                k += 1
    g = capture(timed_step)
    sums = [0.0] * 5
    n = 0
    for _ in range(steps):
        g.replay()
        torch.cuda.synchronize()
        for e6 in ev:
            for i in range(5):
                sums[i] += e6[i].elapsed_time(e6[i + 1])
            n += 1
    return [s_ / n for s_ in sums]


def measure_moe(m, spec, args, dev, rank, world, block_m, steps, with_cpu_baseline):
    """Times one MoE workload on this rank's GPU: the device-timed step, the
    end-to-end step through the C ABI with host buffers, the per-kernel event
    split and the roofline of the dominant kernel. Returns the record."""
    W = Workload(m, spec, dev, block_m, rank)
    stream = torch.cuda.current_stream()
    graph = capture(W.step)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    for li in range(W.layers):
        assert m.status_read(W.route[li]["status"]) == 0
    work = W.work()

    barrier(world)
    with ClockSampler(dev.index or 0) as clk:
        ms = time_region(graph.replay, steps, stream)
    ms = max_over_ranks(ms, world, dev)
    ms_step = ms / steps
    clocks = clk.summary()

    # per-kernel breakdown (events between the kernels of every call: event
    # nodes serialise the launches, so programmatic-dependent-launch overlap
    # between the fused decode layers is lost in this pass)
    prof_steps = max(1, min(steps, 20))
    st = stage_times(W, prof_steps)
    names = ["router", "routing", "expert_gate_up", "expert_down", "combine"]
    per_call_ms = dict(zip(names, st))

    # End to end through the same C ABI with host buffers: every step copies
    # its x in from pinned memory and reads every layer's y back. The copies
    # run on their own streams with two device buffer sets, so step i's
    # compute overlaps step i+1's input copy and step i-1's output copy (the
    # compute steps themselves stay in order on one stream: they share the
    # workspace and routing tables).
    x_host = W.x.cpu().pin_memory()
    y_host = [torch.empty(W.y.shape, dtype=W.y.dtype).pin_memory() for _ in range(2)]
    xb, yb = [W.x, torch.empty_like(W.x)], [W.y, torch.empty_like(W.y)]
    g_cmp = []
    for b in range(2):
        W.x, W.y = xb[b], yb[b]
        g_cmp.append(capture(W.step))
    W.x, W.y = xb[0], yb[0]
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_steps(n):
        for i in range(n):
            b = i & 1
            s_in.wait_event(ev_cmp[b])    # step i-2 has read xb[b]
            with torch.cuda.stream(s_in):
                xb[b].copy_(x_host, non_blocking=True)
            ev_in[b].record(s_in)
            s_cmp.wait_event(ev_in[b])
            s_cmp.wait_event(ev_out[b])   # step i-2's yb[b] has been read back
            with torch.cuda.stream(s_cmp):
                g_cmp[b].replay()
            ev_cmp[b].record(s_cmp)
            s_out.wait_event(ev_cmp[b])
            with torch.cuda.stream(s_out):
                y_host[b].copy_(yb[b], non_blocking=True)
            ev_out[b].record(s_out)

    e2e_steps(2)
    torch.cuda.synchronize()
    n_e2e = max(2, steps // 2)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    e2e_steps(n_e2e)
    s_in.wait_stream(s_out)
    t1.record(s_in)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(t0.elapsed_time(t1), world, dev) / n_e2e
    for li in range(W.layers):
        assert m.status_read(W.route[li]["status"]) == 0

    pk, pk_src = peaks()
    layers_calls = W.layers * W.calls
    tokens_step = spec.T * W.layers
    if spec.T <= 4:
        unit = "us/layer"
        value = ms_step * 1000.0 / W.layers
        e2e_value = e2e_ms * 1000.0 / W.layers
        higher = False
    else:
        unit = "tokens/s"
        value = world * tokens_step / (ms_step / 1000.0)
        e2e_value = world * tokens_step / (e2e_ms / 1000.0)
        higher = True
    layer_bytes = work["bytes_per_step"] / layers_calls
    layer_ms = ms_step / layers_calls
    # A kernel timed inside a long step takes the sustained tensor peak; the
    # fp16 operands run at the bf16 rate.
    tensor_peak = pk.get("bf16_tflops_sustained", pk["bf16_tflops"])
    if W.fused():
        # A decode layer is the prelude plus the fused decode kernel, chained
        # to the next layer by programmatic dependent launch: its time is the
        # timed step's share per layer, and every byte of the layer moves in
        # the fused kernel.
        names = ["router", "routing", "fused_decode_layer", "-", "-"]
        per_call_ms = {k: v for k, v in zip(names, st) if k != "-"}
        dom, dom_bytes = "fused_decode_layer", work["fused_bytes_per_step"] / layers_calls
        achieved = dom_bytes / (layer_ms / 1000.0) / 1e9
        peak = pk["hbm_gbs"]
        roofline = {"kernel": "decode_layer_kernel + prelude (one layer of the timed step)", "bound": "hbm",
                    "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                    "traffic": profiled_traffic(dom, spec.name), "peak_source": pk_src,
                    "algorithmic_bytes_per_launch": int(dom_bytes),
                    "time_per_launch_us": round(layer_ms * 1000.0, 3),
                    "time_source": "ms_per_step / layers (the timed graph, launches overlapped as in the step)"}
    else:
        dom, dom_bytes = "expert_gate_up", work["gate_up_bytes_per_step"] / layers_calls
        gu_ms = per_call_ms[dom]
        gu_flops_launch = work["gate_up_flops_per_step"] / layers_calls
        tensor_bound = gu_flops_launch / dom_bytes > tensor_peak * 1e12 / (pk["hbm_gbs"] * 1e9)
        if tensor_bound:
            achieved = gu_flops_launch / (gu_ms / 1000.0) / 1e12
            roofline = {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 1), "peak": tensor_peak,
                        "unit": "TFLOP/s", "frac": round(achieved / tensor_peak, 4),
                        "traffic": profiled_traffic(dom, spec.name), "peak_source": pk_src + " (sustained bf16)",
                        "algorithmic_flops_per_launch": int(gu_flops_launch),
                        "algorithmic_bytes_per_launch": int(dom_bytes),
                        "time_per_launch_us": round(gu_ms * 1000.0, 3),
                        "time_source": "CUDA events around the launch inside the graph (no overlap to lose)"}
        else:
            achieved = dom_bytes / (gu_ms / 1000.0) / 1e9
            peak = pk["hbm_gbs"]
            roofline = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                        "unit": "GB/s", "frac": round(achieved / peak, 4),
                        "traffic": profiled_traffic(dom, spec.name), "peak_source": pk_src,
                        "algorithmic_bytes_per_launch": int(dom_bytes),
                        "time_per_launch_us": round(gu_ms * 1000.0, 3),
                        "time_source": "CUDA events around the launch inside the graph (no overlap to lose)"}
    out = {
        "metric": METRIC, "value": round(value, 3), "unit": unit, "n_gpus": world, "steps": steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": higher, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "accumulate": "f32", "data": "synthetic",
        "config": {"workload": spec.name, "T": spec.T, "H": spec.H, "I": spec.I, "E": spec.E, "top_k": spec.top_k,
                   "shared_expert": spec.shared, "layers": W.layers, "tokens_per_call": W.T, "block_m": block_m,
                   "router_bias": spec.bias, "seed": spec.seed,
                   "layer_chain": "pre-norm residual blocks: x = RMSNorm(r) (eps 1e-6, gain 1), "
                                  "r_next = bf16(r + y) feeds the next layer" if W.fused() else "independent calls",
                   "l2": f"inputs larger than L2: {W.layers} layers x {layer_bytes / 1e6:.0f} MB touched per step"
                   if W.layers > 1 else "weights 455.8 MB per layer, larger than the 129 MB L2",
                   "parallelism": "replicas" if world > 1 else "1 GPU"},
        "roofline": roofline,
        "layer": {"us_per_layer": round(layer_ms * 1000.0, 3),
                  "algorithmic_bytes_per_layer": int(layer_bytes),
                  "hbm_frac_per_layer": round(layer_bytes / (layer_ms / 1000.0) / 1e9 / pk["hbm_gbs"], 4),
                  "distinct_experts_mean": work["distinct_experts_mean"],
                  "tflops": round(work["flops_per_step"] / (ms_step / 1000.0) / 1e12, 3)},
        "kernels_us_per_call": {k: round(v * 1000.0, 3) for k, v in per_call_ms.items()},
        "kernels_timing": "CUDA events between the kernels of every call in a second graph pass; the event nodes "
                          "break programmatic-dependent-launch overlap, so these are diagnostics, not the step",
        "e2e": {"value": round(e2e_value, 3), "unit": unit, "h2d_bytes_per_step": x_host.numel() * 2,
                "d2h_bytes_per_step": y_host[0].numel() * 4,
                "pipeline": "input copy, compute and output copy on three streams with two buffer sets"},
        "gpu_launches": W.launches_per_step() * steps,
        "launch": "one CUDA graph per step",
        "clocks": clocks,
    }
    if not W.fused():
        gu_ms = per_call_ms["expert_gate_up"]
        gu_tflops = work["gate_up_flops_per_step"] / layers_calls / (gu_ms / 1000.0) / 1e12
        out["gate_up"] = {"us_per_launch": round(gu_ms * 1000.0, 3), "tflops": round(gu_tflops, 1),
                          "frac_of_sustained_bf16": round(gu_tflops / tensor_peak, 4),
                          "frac_of_burst_bf16": round(gu_tflops / pk["bf16_tflops"], 4),
                          "hbm_gbs": round(dom_bytes / (gu_ms / 1000.0) / 1e9, 1)}
    if with_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(spec, args.cpu_seconds)
    del W, graph, g_cmp, xb, yb
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


# The prefill half of the metric, measured in the same run as a decode line.
PREFILL_COMPANION = "prefill-4096"


def run_ours(args, spec, rank, world, local_rank):
    import bit_grouped_expert_moe_gb300 as m
    from bit_grouped_expert_moe_gb300 import _build
    _build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    block_m = args.block_m or (16 if spec.T <= 64 else 64 if spec.T <= 1024 else 128)
    cpu = rank == 0 and world == 1 and not args.no_cpu_baseline
    out = measure_moe(m, spec, args, dev, rank, world, block_m, args.steps, cpu)
    if spec.T <= 4 and not args.no_prefill:
        # Prefill record of the same run: tokens/s on the device and end to
        # end, the gate/up GEMM's tensor rate and fraction of the bf16 peak.
        ps = synth.WORKLOADS[PREFILL_COMPANION]
        rec = measure_moe(m, ps, args, dev, rank, world, 128, max(10, min(args.steps, 50)), False)
        out["prefill"] = {k: rec[k] for k in ("value", "unit", "ms_per_step", "steps", "e2e", "gate_up", "roofline",
                                               "layer", "kernels_us_per_call", "clocks", "gpu_launches")}
        out["prefill"]["workload"] = ps.name
        out["prefill"]["block_m"] = 128
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return out


# ------------------------------------------------------ decode attention --

METRIC_ATTN = "decode-attention µs/layer (GQA, bf16 KV cache); % of HBM roofline"


class AttnWorkload:
    """Device-resident inputs of a decode-attention workload: one layer per
    full-attention layer of the model, each with its own KV cache."""

    def __init__(self, m, spec, device):
        self.m, self.spec, self.dev = m, spec, device
        self.layers = spec.layers
        self.shape = m.attn_shape(spec.B, spec.Hq, spec.Hkv, spec.D, spec.Lmax)
        self.q = torch.empty(self.layers, spec.B, spec.Hq, spec.D, dtype=torch.bfloat16, device=device)
        self.kv = []
        for li in range(self.layers):
            q, k, v, lens = synth.attn_inputs(spec, layer=li, device=device)
            self.q[li].copy_(q)
            self.kv.append((k, v))
            del q
        self.lens = torch.tensor(spec.lens, dtype=torch.int32, device=device)
        self.o = torch.empty(self.layers, spec.B, spec.Hq, spec.D, dtype=torch.float32, device=device)
        self.ws = m.attn_alloc_workspace(self.shape, device)

    def call(self, li, events=None):
        k, v = self.kv[li]
        if events is None:
            self.m.attn_decode(self.shape, self.q[li], k, v, self.lens, self.o[li], self.ws)
        else:
            self.m.attn_decode_timed(self.shape, self.q[li], k, v, self.lens, self.o[li], self.ws, events)

    def step(self):
        for li in range(self.layers):
            self.call(li)

    def kv_bytes_per_layer(self):
        s = self.spec
        return sum(s.lens) * s.Hkv * s.D * 2 * 2


def attn_stage_times(W, steps):
    """Average block-kernel and merge-kernel times (ms) from event nodes
    between the two kernels of every layer, in a graph of one step."""
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(W.layers)]
    for e3 in ev:
        for e in e3:
            e.record()
    torch.cuda.synchronize()

    def timed_step():
        for li in range(W.layers):
            W.call(li, events=[e.cuda_event for e in ev[li]])
    g = capture(timed_step)
    blk = mrg = 0.0
    for _ in range(steps):
        g.replay()
        torch.cuda.synchronize()
        for e3 in ev:
            blk += e3[0].elapsed_time(e3[1])
            mrg += e3[1].elapsed_time(e3[2])
    n = steps * W.layers
    return blk / n, mrg / n


def run_attention(args, spec, rank, world, local_rank):
    import bit_grouped_expert_moe_gb300 as m
    from bit_grouped_expert_moe_gb300 import _build
    _build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    W = AttnWorkload(m, spec, dev)
    stream = torch.cuda.current_stream()
    graph = capture(W.step)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    assert m.status_read(W.ws[:4].view(torch.int32)) == 0

    barrier(world)
    with ClockSampler(local_rank) as clk:
        ms = time_region(graph.replay, args.steps, stream)
    ms = max_over_ranks(ms, world, dev)
    ms_step = ms / args.steps
    clocks = clk.summary()
    blk_ms, mrg_ms = attn_stage_times(W, max(1, min(args.steps, 20)))

    # End to end through the same C ABI with host buffers: every step copies
    # each layer's query in from pinned memory and reads every output back.
    q_host = W.q.cpu().pin_memory()
    o_host = torch.empty(W.o.shape, dtype=W.o.dtype).pin_memory()

    def e2e_step():
        W.q.copy_(q_host, non_blocking=True)
        graph.replay()
        o_host.copy_(W.o, non_blocking=True)
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    n_e2e = max(2, args.steps // 2)
    e2e_ms = max_over_ranks(time_region(e2e_step, n_e2e, stream), world, dev) / n_e2e
    assert m.status_read(W.ws[:4].view(torch.int32)) == 0

    pk, pk_src = peaks()
    peak = pk["hbm_gbs"]
    kv = W.kv_bytes_per_layer()
    blk_bytes = kv + spec.B * spec.Hq * spec.D * 2 + spec.B * 4
    achieved = blk_bytes / (blk_ms / 1000.0) / 1e9
    value = ms_step * 1000.0 / W.layers
    out = {
        "metric": METRIC_ATTN, "value": round(value, 3), "unit": "us/layer", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "accumulate": "f32", "data": "synthetic",
        "config": {"workload": spec.name, "B": spec.B, "lens": list(spec.lens), "Hq": spec.Hq, "Hkv": spec.Hkv,
                   "D": spec.D, "L_max": spec.Lmax, "layers": W.layers, "seed": spec.seed,
                   "l2": f"inputs larger than L2: {W.layers} layers x {kv / 1e6:.0f} MB of KV cache per step",
                   "parallelism": "replicas" if world > 1 else "1 GPU"},
        "roofline": {"kernel": "attn_block_kernel", "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": profiled_traffic("attn_block_kernel", spec.name), "peak_source": pk_src,
                     "algorithmic_bytes_per_launch": int(blk_bytes)},
        "layer": {"us_per_layer": round(value, 3), "kv_bytes_per_layer": int(kv),
                  "hbm_frac_per_layer": round(kv / (value / 1e6) / 1e9 / peak, 4)},
        "kernels_us_per_call": {"attn_block_kernel": round(blk_ms * 1000.0, 3),
                                "attn_merge_kernel": round(mrg_ms * 1000.0, 3)},
        "e2e": {"value": round(e2e_ms * 1000.0 / W.layers, 3), "unit": "us/layer",
                "h2d_bytes_per_step": q_host.numel() * 2, "d2h_bytes_per_step": o_host.numel() * 4},
        "gpu_launches": 2 * W.layers * args.steps,
        "launch": "one CUDA graph per step",
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = attn_cpu_baseline(spec, args.cpu_seconds)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return out


def _attn_oracle_inputs(spec):
    from tests._util import bits16
    q, k, v, lens = synth.attn_inputs(spec, layer=0)
    return bits16(q), bits16(k), bits16(v), list(spec.lens)


def attn_cpu_baseline(spec, seconds):
    """The attention oracle, as it stands, timed on this host's cores on
    layer 0 of the workload (inputs generated before the clock starts)."""
    import oracle
    args = _attn_oracle_inputs(spec)
    spent, calls = 0.0, 0
    while spent < seconds and calls < 50:
        t0 = time.perf_counter()
        oracle.gqa_decode_attention(*args)
        spent += time.perf_counter() - t0
        calls += 1
    return {"value": round(spent / calls * 1e6, 3), "unit": "us/layer", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{calls} calls on layer 0 of the workload (numpy fp64, BLAS multithreaded)",
            "seconds": round(spent, 2)}


def run_attention_reference(args, spec, rank, world):
    """The reference arm for attention workloads: the CPU oracle (rank 0)."""
    if rank != 0:
        return None
    import oracle
    a = _attn_oracle_inputs(spec)
    times = []
    t_start = time.perf_counter()
    for i in range(args.warmup + args.steps):
        if time.perf_counter() - t_start > 150.0 and times:
            break
        t0 = time.perf_counter()
        oracle.gqa_decode_attention(*a)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    if not times:
        times.append(dt)
    value = sum(times) / len(times) * 1e6
    return {"impl": "reference", "metric": METRIC_ATTN, "value": round(value, 3), "unit": "us/layer",
            "n_gpus": world, "steps": len(times), "steps_requested": args.steps, "warmup": args.warmup,
            "ms_per_step": round(value / 1000.0, 3), "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": spec.name, "B": spec.B, "lens": list(spec.lens), "Hq": spec.Hq,
                       "Hkv": spec.Hkv, "D": spec.D, "layers": spec.layers},
            "cpu_baseline": {"value": round(value, 3), "unit": "us/layer", "cores": os.cpu_count(),
                             "kind": "oracle", "sample": "one oracle call on layer 0 per step; capped at 150 s"},
            "e2e": {"value": round(value, 3), "unit": "us/layer", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# -------------------------------------------------------- Gated DeltaNet --

METRIC_GDN = "Gated DeltaNet scan µs/layer (fp32 state in registers); % of ALU (prefill) / HBM (decode) roofline"
# fp32 FMA peak: 152 SMs x 128 FP32 lanes x 2 flops x the SM clock (2070 MHz at most)
FP32_LANES_PER_SM = 128


class GdnWorkload:
    """Device-resident inputs of a Gated DeltaNet workload: one set per layer,
    each layer with its own initial state (read) and final state (written)."""

    def __init__(self, m, spec, device):
        self.m, self.spec, self.dev = m, spec, device
        self.layers = spec.layers
        self.shape = m.gdn_shape(spec.B, spec.T, spec.Hqk, spec.Hv, spec.Dk, spec.Dv)
        self.inp = [list(synth.gdn_inputs(spec, layer=li, device=device)) for li in range(self.layers)]
        self.state_out = [torch.empty_like(x[5]) for x in self.inp]
        self.o = torch.empty(self.layers, spec.T, spec.Hv, spec.Dv, dtype=torch.float32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)

    def call(self, li, events=None):
        q, k, v, gate, beta, state, offsets = self.inp[li]
        if events is None:
            self.m.gdn_scan(self.shape, q, k, v, gate, beta, offsets, state, self.state_out[li], self.o[li],
                            status=self.status)
        else:
            self.m.gdn_scan_timed(self.shape, q, k, v, gate, beta, offsets, state, self.state_out[li], self.o[li],
                                  events, status=self.status)

    def step(self):
        for li in range(self.layers):
            self.call(li)

    def bytes_per_layer(self):
        s = self.spec
        state = s.B * s.Hv * s.Dv * s.Dk * 4 * 2
        tok = s.T * (2 * s.Hqk * s.Dk * 2 + s.Hv * s.Dv * 2 + 2 * s.Hv * 4 + s.Hv * s.Dv * 4)
        return state + tok + (s.B + 1) * 4

    def flops_per_layer(self):
        s = self.spec   # per token and state element: the two dot products and the update (3 FMAs)
        return s.T * s.Hv * s.Dv * s.Dk * 6


def gdn_kernel_time(W, steps):
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(W.layers)]
    for e2 in ev:
        for e in e2:
            e.record()
    torch.cuda.synchronize()

    def timed_step():
        for li in range(W.layers):
            W.call(li, events=[e.cuda_event for e in ev[li]])
    g = capture(timed_step)
    t = 0.0
    for _ in range(steps):
        g.replay()
        torch.cuda.synchronize()
        for e2 in ev:
            t += e2[0].elapsed_time(e2[1])
    return t / (steps * W.layers)


def run_gdn(args, spec, rank, world, local_rank):
    import bit_grouped_expert_moe_gb300 as m
    from bit_grouped_expert_moe_gb300 import _build
    _build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    W = GdnWorkload(m, spec, dev)
    stream = torch.cuda.current_stream()
    graph = capture(W.step)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    assert m.status_read(W.status) == 0

    barrier(world)
    with ClockSampler(local_rank) as clk:
        ms = time_region(graph.replay, args.steps, stream)
    ms = max_over_ranks(ms, world, dev)
    ms_step = ms / args.steps
    clocks = clk.summary()
    k_ms = gdn_kernel_time(W, max(1, min(args.steps, 20)))

    # End to end with host buffers: every step copies each layer's token
    # inputs (q, k, v, gate, beta) in from pinned memory and reads every
    # layer's output back; the recurrent state stays on the device.
    host_in = [[x.cpu().pin_memory() for x in W.inp[li][:5]] for li in range(W.layers)]
    o_host = torch.empty(W.o.shape, dtype=W.o.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for xs in host_in for x in xs)

    def e2e_step():
        for li in range(W.layers):
            for dst, src in zip(W.inp[li][:5], host_in[li]):
                dst.copy_(src, non_blocking=True)
        graph.replay()
        o_host.copy_(W.o, non_blocking=True)
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    n_e2e = max(2, args.steps // 2)
    e2e_ms = max_over_ranks(time_region(e2e_step, n_e2e, stream), world, dev) / n_e2e
    assert m.status_read(W.status) == 0

    pk, pk_src = peaks()
    value = ms_step * 1000.0 / W.layers
    decode = spec.T <= 2 * spec.B   # the library runs these on its short-sequence kernel
    kname = "gdn_short_kernel" if decode else "gdn_scan_kernel"
    if decode:
        by = W.bytes_per_layer()
        ach = by / (k_ms / 1000.0) / 1e9
        roof = {"kernel": kname, "bound": "hbm", "achieved": round(ach, 1), "peak": pk["hbm_gbs"],
                "unit": "GB/s", "frac": round(ach / pk["hbm_gbs"], 4), "traffic": profiled_traffic(kname, spec.name),
                "peak_source": pk_src, "algorithmic_bytes_per_launch": int(by)}
    else:
        fl = W.flops_per_layer()
        sm_mhz = pk.get("sm_max_mhz", 2070.0)
        peak = 152 * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12
        ach = fl / (k_ms / 1000.0) / 1e12
        roof = {"kernel": kname, "bound": "alu", "achieved": round(ach, 2), "peak": round(peak, 1),
                "unit": "TFLOP/s", "frac": round(ach / peak, 4), "traffic": profiled_traffic(kname, spec.name),
                "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 flops x max SM clock",
                "algorithmic_flops_per_launch": int(fl)}
    out = {
        "metric": METRIC_GDN, "value": round(value, 3), "unit": "us/layer", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 5), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "inputs": "bf16 q, k, v; fp32 gate, beta, state", "data": "synthetic",
        "config": {"workload": spec.name, "B": spec.B, "T": spec.T, "Hqk": spec.Hqk, "Hv": spec.Hv, "Dk": spec.Dk,
                   "Dv": spec.Dv, "layers": W.layers, "seed": spec.seed,
                   "l2": f"{W.layers} layers x {W.bytes_per_layer() / 1e6:.0f} MB per step"
                         + (" (larger than L2)" if W.layers * W.bytes_per_layer() > 129e6 else ""),
                   "parallelism": "replicas" if world > 1 else "1 GPU"},
        "roofline": roof,
        "kernels_us_per_call": {kname: round(k_ms * 1000.0, 3)},
        "e2e": {"value": round(e2e_ms * 1000.0 / W.layers, 3), "unit": "us/layer", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": o_host.numel() * 4},
        "gpu_launches": W.layers * args.steps,
        "launch": "one CUDA graph per step",
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = gdn_cpu_baseline(spec, args.cpu_seconds)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return out


def _gdn_oracle_sample(spec, heads):
    """One oracle call on layer 0 restricted to `heads` value heads (inputs
    generated before the clock starts); returns seconds."""
    import numpy as np
    import oracle
    from tests._util import bits16
    q, k, v, gate, beta, state, offsets = synth.gdn_inputs(spec, layer=0)
    per = spec.Hv // spec.Hqk
    args = []
    for h in heads:
        g = h // per
        args.append((bits16(q[:, g:g + 1]), bits16(k[:, g:g + 1]), bits16(v[:, h:h + 1]),
                     gate[:, h:h + 1].double().numpy(), beta[:, h:h + 1].double().numpy(),
                     state[:, h:h + 1].double().numpy(), offsets.numpy()))
    t0 = time.perf_counter()
    for a in args:
        oracle.gated_delta_scan(*a)
    return time.perf_counter() - t0


def gdn_cpu_baseline(spec, seconds):
    """The oracle, as it stands, on this host's cores: value heads of layer 0
    timed one at a time until about `seconds`, scaled to a whole layer."""
    spent, heads = 0.0, 0
    while spent < seconds and heads < spec.Hv:
        spent += _gdn_oracle_sample(spec, [heads])
        heads += 1
    per_layer = spent / heads * spec.Hv
    return {"value": round(per_layer * 1e6, 3), "unit": "us/layer", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{heads} of the {spec.Hv} value heads of layer 0, scaled to the layer (numpy fp64)",
            "seconds": round(spent, 2)}


def run_gdn_reference(args, spec, rank, world):
    if rank != 0:
        return None
    times = []
    t_start = time.perf_counter()
    for i in range(args.warmup + args.steps):
        if time.perf_counter() - t_start > 150.0 and times:
            break
        dt = _gdn_oracle_sample(spec, [i % spec.Hv]) * spec.Hv
        if i >= args.warmup:
            times.append(dt)
    if not times:
        times.append(dt)
    value = sum(times) / len(times) * 1e6
    return {"impl": "reference", "metric": METRIC_GDN, "value": round(value, 3), "unit": "us/layer",
            "n_gpus": world, "steps": len(times), "steps_requested": args.steps, "warmup": args.warmup,
            "ms_per_step": round(value / 1000.0, 3), "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": spec.name, "B": spec.B, "T": spec.T, "Hqk": spec.Hqk, "Hv": spec.Hv,
                       "layers": spec.layers},
            "cpu_baseline": {"value": round(value, 3), "unit": "us/layer", "cores": os.cpu_count(),
                             "kind": "oracle",
                             "sample": "one value head of layer 0 per step, scaled to the layer; capped at 150 s"},
            "e2e": {"value": round(value, 3), "unit": "us/layer", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ----------------------------------------------------------- CPU oracle --

ORACLE_THREADS = 1  # the C++ oracle (oracle/moe_ref.cpp) runs on the calling thread

def _oracle_layer_sample(spec, layer_idx, tokens):
    """One oracle call of the workload on `tokens` of a layer; weights are
    regenerated on the CPU (not timed) and the oracle's own work (routing,
    dequantisation of every used expert, the products) is timed."""
    import numpy as np
    import oracle.cpp as oracle  # the C++ oracle, one thread
    from tests._util import bits16, expert_fn_lazy
    x = synth.activations(spec, T=max(tokens) + 1)
    wr, wsg = synth.router_weights(spec, layer_idx)
    b = synth.router_bias(spec)
    xb = bits16(x)
    wrb = bits16(wr)
    wsgb = None if wsg is None else bits16(wsg)
    bias = None if b is None else b.numpy()
    # regenerate the experts these tokens use before the clock starts
    ids, *_ = oracle.route(xb[tokens], wrb, bias, wsgb, spec.top_k)
    fn = expert_fn_lazy(spec, layer_idx)
    cache = {e: fn(int(e)) for e in list(np.unique(ids)) + ([spec.E] if spec.shared else [])}
    t0 = time.perf_counter()
    oracle.moe_forward(xb, wrb, bias, wsgb, spec.top_k, lambda e: cache[e], tokens=np.asarray(tokens))
    return time.perf_counter() - t0


def cpu_baseline(spec, seconds):
    """The oracle, as it stands, timed on this host's cores on a bounded
    sample of the workload, in the workload's unit."""
    import numpy as np
    spent, calls, toks = 0.0, 0, 0
    if spec.T <= 4:
        li = 0
        while spent < seconds and li < spec.layers:
            spent += _oracle_layer_sample(spec, li, list(range(spec.T)))
            calls += 1
            li += 1
        value, unit = spent / calls * 1e6, "us/layer"
        sample = f"{calls} of the {spec.layers} layers at T={spec.T}"
    else:
        n = min(spec.chunk or spec.T, 256)
        rng = np.random.default_rng(1)
        while spent < seconds and calls < 8:
            tokens = sorted(rng.choice(spec.chunk or spec.T, n, replace=False).tolist())
            spent += _oracle_layer_sample(spec, 0, tokens)
            calls += 1
            toks += n
        value, unit = toks / spent, "tokens/s"
        sample = f"{calls} calls of {n} sampled tokens of layer 0"
    return {"value": round(value, 3), "unit": unit, "cores": ORACLE_THREADS, "kind": "oracle",
            "sample": sample + " (the C++ oracle: plain fp64 loops on one thread)",
            "seconds": round(spent, 2)}


def run_reference(args, spec, rank, world):
    """The reference arm: the CPU oracle on the host cores (rank 0 only)."""
    if rank != 0:
        return None
    budget = 150.0
    times = []
    t_start = time.perf_counter()
    for i in range(args.warmup + args.steps):
        if time.perf_counter() - t_start > budget and len(times) >= 1:
            break
        if spec.T <= 4:
            dt = _oracle_layer_sample(spec, i % spec.layers, list(range(spec.T)))
        else:
            import numpy as np
            rng = np.random.default_rng(i)
            n = min(spec.chunk or spec.T, 64)
            dt = _oracle_layer_sample(spec, 0, sorted(rng.choice(spec.chunk or spec.T, n, replace=False).tolist()))
        if i >= args.warmup:
            times.append(dt)
    if not times:
        times.append(dt)
    mean = sum(times) / len(times)
    if spec.T <= 4:
        value, unit, higher = mean * 1e6, "us/layer", False
        sample = f"one layer at T={spec.T} per step"
    else:
        n = min(spec.chunk or spec.T, 64)
        value, unit, higher = n / mean, "tokens/s", True
        sample = f"{n} sampled tokens of layer 0 per step"
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": unit, "n_gpus": world,
           "steps": len(times), "steps_requested": args.steps, "warmup": args.warmup,
           "ms_per_step": round(mean * 1000, 3), "higher_is_better": higher, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": spec.name, "T": spec.T, "H": spec.H, "I": spec.I, "E": spec.E,
                      "top_k": spec.top_k, "layers": spec.layers},
           "cpu_baseline": {"value": round(value, 3), "unit": unit, "cores": ORACLE_THREADS, "kind": "oracle",
                            "sample": sample + f" (the C++ oracle: plain fp64 loops on one thread); capped at "
                                      f"{budget:.0f} s of oracle work"},
           "e2e": {"value": round(value, 3), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode-t1",
                    choices=sorted(synth.WORKLOADS) + sorted(synth.ATTN_WORKLOADS) + sorted(synth.GDN_WORKLOADS))
    ap.add_argument("--block-m", type=int, default=0)
    ap.add_argument("--layers", type=int, default=0, help="override the workload's layer count (profiling only)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="decode workloads: skip the prefill-4096 record measured in the same run")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local_rank = dist_env()
    if args.workload in synth.GDN_WORKLOADS:
        spec = synth.GDN_WORKLOADS[args.workload]
        if args.layers:
            import dataclasses
            spec = dataclasses.replace(spec, layers=args.layers)
        out = run_gdn_reference(args, spec, rank, world) if args.impl == "reference" else \
            run_gdn(args, spec, rank, world, local_rank)
        if rank == 0 and out is not None:
            print(json.dumps(out), flush=True)
        return
    if args.workload in synth.ATTN_WORKLOADS:
        spec = synth.ATTN_WORKLOADS[args.workload]
        if args.layers:
            import dataclasses
            spec = dataclasses.replace(spec, layers=args.layers)
        if args.impl == "reference":
            out = run_attention_reference(args, spec, rank, world)
        else:
            out = run_attention(args, spec, rank, world, local_rank)
        if rank == 0 and out is not None:
            print(json.dumps(out), flush=True)
        return
    spec = synth.WORKLOADS[args.workload]
    if args.layers:
        import dataclasses
        spec = dataclasses.replace(spec, layers=args.layers)
    if args.impl == "reference":
        out = run_reference(args, spec, rank, world)
    else:
        out = run_ours(args, spec, rank, world, local_rank)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
