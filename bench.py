#!/usr/bin/env python3
"""Benchmark of the GB300 small-batch decode hot path.

One "step" is one pass of every hot-path operation of a Kimi-K3-shaped decode layer,
at every decode batch B in {1,2,4,8,16,32,64}, on synthetic bf16 inputs:

    input projection   Y = X . W^T            K=7168  -> N=8192       (batch switch)
    output projection  Y = X . W^T + R        K=16384 -> N=7168       (split-K + residual)
    MoE front end      router 384 + latent 512 rows in one product, softmax, top-8
    MoE experts        384 routed experts (gate/up 2x2048x7168, down 7168x2048) grouped
                       GEMV + the shared expert of the same shape, one launch, + combine
    (--prefetch adds an L2 prefetch of the shared expert's weights during the front end)

`value` is the whole step's algorithmic HBM bytes (weights read once + activations in
and out, using the actual number of distinct experts each batch routes to) divided by
the device time of the step, replayed as one CUDA graph: GB/s. Every weight tensor is
re-read only after more than 3x the L2 size of other weight traffic, so every read is
cold. `sweep` gives the same figures per operation and batch (CUDA graph of R calls
over a rotating pool of weight copies >= 3x L2). `e2e` runs the step eagerly through
the public API with the step's activations copied from pinned host memory and its
outputs copied back inside the timed region. `cpu_baseline` times the fp64 oracle on a
bounded sample of the same step on the host cores.

Multi-GPU: the path has no exchange step on one GPU, so N ranks run N independent
replicas (weak scaling); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import threading
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "achieved HBM GB/s (fraction of GB300 roofline) and µs/call per decode batch 1–64"
BATCHES = [1, 2, 4, 8, 16, 32, 64]
H, N_IN, K_O, E, L, I, TOPK = 7168, 8192, 16384, 384, 512, 2048, 8
N_SK, K_SK = 2048, 1024  # the single skinny GEMM (B = 1), timed in the sweep
PREFETCH_BYTES = 24 << 20
WORKLOAD = ("Kimi-K3-shaped decode layer hot path, B in {1,2,4,8,16,32,64}: input projection "
            "7168->8192 (batch-size kernel switch), output projection 16384->7168 + residual, "
            "MoE front end 7168->384 router + 512 latent with softmax/top-8, 384 routed experts "
            "(gate/up 2x2048x7168, down 7168x2048) + shared expert overlapping them (its "
            "tiles in the routed experts' launch)")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--batches", default=",".join(map(str, BATCHES)))
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target host time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--ops", default="in,o,front,experts",
                    help="operations of the sweep (profiling subsets: in,o,front,experts; "
                         "pfscen = output projection behind a simulated communication phase; "
                         "spec = projections at speculative verification row counts; "
                         "skinny = the single B=1 1024->2048 GEMM)")
    ap.add_argument("--sweep-only", action="store_true",
                    help="only the per-operation sweep (for profiler captures)")
    ap.add_argument("--num-experts", type=int, default=E,
                    help="routed experts in the bank (smaller for profiler captures)")
    ap.add_argument("--reps", type=int, default=7, help="graph replays per sweep entry")
    ap.add_argument("--step-only", action="store_true",
                    help="only the step graph (no sweep, e2e or CPU baseline), for profiler captures")
    ap.add_argument("--layer", action="store_true",
                    help="step: moe_layer (shared expert overlapping the front end) instead of "
                         "moe_front + moe_experts")
    ap.add_argument("--prefetch", action="store_true",
                    help="step: L2 prefetch of the shared expert's weights during the front end")
    ap.add_argument("--row-major", action="store_true",
                    help="projection weights row-major [N,K] instead of tile-packed")
    return ap.parse_args()


# ------------------------------------------------------------ byte accounting --

def bytes_linear(B, N, K, residual):
    return N * K * 2 + B * K * 2 + B * N * 2 + (B * N * 2 if residual else 0)


def bytes_front(B, n_experts=E):
    return (n_experts + L) * H * 2 + B * H * 2 + B * L * 2 + B * TOPK * 8


def bytes_experts(B, U):
    per_expert = 3 * I * H * 2
    return (U + 1) * per_expert + 2 * B * H * 2 + B * TOPK * 8


# ------------------------------------------------------------------- clocks ----

class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        """Start sampling every 20 ms and return once the first sample has arrived (or
        after 5 s), so the timed region that follows is covered from its start."""
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        first = threading.Event()

        def reader():
            for line in self.proc.stdout:
                self.lines.append(line)
                first.set()

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()
        first.wait(timeout=5.0)
        self.lines.clear()  # keep only samples taken during the timed region

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        out = "".join(self.lines)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        self.thread.join(timeout=5)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "samples": len(sm),
                "reasons": sorted(reasons)}


# ----------------------------------------------------------------- workload ----

class Workload:
    """All tensors of the step on one GPU, plus the per-call launch counts."""

    def __init__(self, torch, ssd, inputs, dev, batches, seed=0, num_experts=E, experts=True,
                 packed=True):
        self.torch, self.ssd, self.dev, self.batches = torch, ssd, dev, batches
        # projection weights tile-packed once here, at load time (dec_pack_weight), and
        # read by the packed projections; row-major [N,K] with packed=False
        self.packed = packed
        self.lin = ssd.dec_linear_packed if packed else ssd.dec_linear
        self.E = num_experts
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.l2 = l2
        bf = torch.bfloat16
        W_in = inputs.weight(N_IN, H, dev, seed, "w_in")
        W_o = inputs.weight(H, K_O, dev, seed, "w_o")
        W_cat = inputs.weight(num_experts + L, H, dev, seed, "w_cat")
        # rotating copies for the per-operation sweep: >= 3x L2 per pool
        def pool(w):
            n = max(1, math.ceil(3 * l2 / (w.numel() * 2)))
            return [w] + [w.clone() for _ in range(n - 1)]
        if packed:
            W_in, W_o = ssd.dec_pack_weight(W_in), ssd.dec_pack_weight(W_o)
        self.W_in, self.W_o, self.W_cat = pool(W_in), pool(W_o), pool(W_cat)
        if experts:
            self.Wgu, self.Wd = inputs.expert_bank(num_experts, H, I, dev, seed, "bank")
        self.Wgs, self.Wds = inputs.shared_expert(H, I, dev, seed, "bank_shared")
        if packed:  # expert banks tile-packed once here as well; the row-major bank is freed
            if experts:
                self.Wgu, self.Wd = ssd.dec_pack_expert_weights(self.Wgu, self.Wd)
            gs, ds = ssd.dec_pack_expert_weights(self.Wgs[None], self.Wds[None])
            self.Wgs, self.Wds = gs[0], ds[0]
            torch.cuda.synchronize()
            torch.cuda.empty_cache()
        self.side = torch.cuda.Stream(device=dev)
        self.fork = torch.cuda.Event()
        self.join = torch.cuda.Event()
        self.t = {}
        for B in batches:
            d = {}
            d["x_in"] = inputs.activations(B, H, dev, seed, "x_in")
            d["x_o"] = inputs.activations(B, K_O, dev, seed, "x_o")
            d["r_o"] = inputs.residual(B, H, dev, seed, "r_o")
            d["x_moe"] = [inputs.activations(B, H, dev, seed + v, "x_moe") for v in range(3)]
            d["y_in"] = torch.empty(B, N_IN, dtype=bf, device=dev)
            d["y_o"] = torch.empty(B, H, dtype=bf, device=dev)
            d["lat"] = [torch.empty(B, L, dtype=bf, device=dev) for _ in range(3)]
            d["idx"] = [torch.empty(B, TOPK, dtype=torch.int32, device=dev) for _ in range(3)]
            d["w"] = [torch.empty(B, TOPK, dtype=torch.float32, device=dev) for _ in range(3)]
            d["rm"] = [torch.empty(ssd.moe_route_map_ints(B, self.E, TOPK), dtype=torch.int32,
                                   device=dev) for _ in range(3)]
            d["y_moe"] = torch.empty(B, H, dtype=bf, device=dev)
            d["ws_in"] = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N_IN, H), dev)
            d["ws_o"] = ssd.workspace(ssd.dec_linear_workspace_bytes(B, H, K_O), dev)
            d["ws_f"] = ssd.workspace(ssd.moe_front_workspace_bytes(B, self.E, L, H), dev)
            d["ws_e"] = ssd.workspace(ssd.moe_experts_workspace_bytes(B, self.E, TOPK, H, I), dev)
            if experts:
                d["ws_l"] = ssd.workspace(ssd.moe_layer_workspace_bytes(B, self.E, L, H, I, TOPK),
                                          dev)
            self.t[B] = d
        self.launches = 0
        self.prefetch = False
        self.layer = False
        torch.cuda.synchronize()

    # -- operations (each adds the kernels it launches to self.launches) --
    def op_in(self, B, rot=0):
        d = self.t[B]
        self.lin(d["x_in"], self.W_in[rot % len(self.W_in)], None, d["y_in"], d["ws_in"])
        self.launches += 1

    def op_o(self, B, rot=0):
        d = self.t[B]
        self.lin(d["x_o"], self.W_o[rot % len(self.W_o)], d["r_o"], d["y_o"], d["ws_o"])
        # from B = 32 the K = 16384 projection defers its reduction to a finishing kernel
        self.launches += 2 if B >= 32 else 1

    def op_front(self, B, rot=0, v=0, prefetch=True, with_map=True):
        """moe_front, building the route map the experts' launches read (measured: the
        whole layer is 1-11 us faster than leaving the map to moe_experts' gather)."""
        torch, ssd, d = self.torch, self.ssd, self.t[B]
        if prefetch:
            main = torch.cuda.current_stream()
            self.fork.record(main)
            self.side.wait_event(self.fork)
            ssd.l2_prefetch(self.Wgs, nbytes=PREFETCH_BYTES, max_ctas=8, stream=self.side)
            self.launches += 1
        ssd.moe_front(d["x_moe"][v], self.W_cat[rot % len(self.W_cat)], self.E, L, TOPK, d["lat"][v],
                      d["idx"][v], d["w"][v], d["ws_f"],
                      route_map=d["rm"][v] if with_map else None)
        self.launches += 1

    def op_experts(self, B, v=0):
        d = self.t[B]
        self.ssd.moe_experts(d["x_moe"][v], d["idx"][v], d["w"][v], d["rm"][v], self.Wgu, self.Wd,
                             self.Wgs, self.Wds, d["y_moe"], d["ws_e"], side_stream=self.side,
                             packed=self.packed)
        self.launches += expert_launches()

    def op_layer(self, B, v=0):
        """moe_layer: the front end and the experts in one call (on the side-stream path the
        shared expert streams its weights during the front end)."""
        d = self.t[B]
        self.ssd.moe_layer(d["x_moe"][v], self.W_cat[0], self.E, L, TOPK, self.Wgu, self.Wd,
                           self.Wgs, self.Wds, d["lat"][v], d["idx"][v], d["w"][v], d["y_moe"],
                           d["ws_l"], route_map=d["rm"][v], side_stream=self.side,
                           packed=self.packed)
        self.launches += 1 + expert_launches()  # the one-launch front end, then the experts

    def op_moe(self, B):
        if self.layer:
            self.op_layer(B)
        else:
            self.op_front(B, prefetch=self.prefetch)
            self.op_experts(B)

    def step(self):
        for B in self.batches:
            self.op_in(B)
            self.op_o(B)
            self.op_moe(B)

    def used_experts(self, B, v=0):
        rm = self.t[B]["rm"][v]
        P = B * TOPK
        return int(rm[2 * self.E + 1 + 2 * P].item())

    def step_bytes(self):
        tot = 0
        for B in self.batches:
            tot += bytes_linear(B, N_IN, H, False) + bytes_linear(B, H, K_O, True)
            tot += bytes_front(B, self.E) + bytes_experts(B, self.used_experts(B))
        return tot


def capture(torch, fn):
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # one eager pass on the capture stream (function attributes, lazy init)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_graph(torch, g, reps):
    st = torch.cuda.current_stream()
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        g.replay()
        b.record(st)
        b.synchronize()
        ts.append(a.elapsed_time(b) * 1e3)  # us
    return ts


def expert_launches():
    """Kernel launches of one moe_experts call with a route map, as the library's switches
    pick them: the gather, the routed gate/up and down (one launch, or two), the shared
    expert's gate/up and down (inside the routed launch, or two launches on the side
    stream), the combine."""
    one = os.environ.get("DEC_EXPERT_ONE_LAUNCH", "1") != "0"
    inside = (one and os.environ.get("DEC_SHARED_IN_ROUTED", "1") != "0"
              and os.environ.get("DEC_FUSED_COMBINE", "0") == "0")
    fused = os.environ.get("DEC_FUSED_COMBINE", "0") != "0"
    return 1 + (1 if one else 2) + (0 if inside else 2) + (0 if fused else 1)


# ------------------------------------------------------- prefetch scenario ----

PF_WAIT_US = 20.0
# DRAM bytes / algorithmic bytes of one expert-layer call (ncu, 32-expert bank, B = 64,
# routed and shared experts in one launch), with tile-packed banks and with row-major ones
EXPERTS_TRAFFIC_RATIO = {True: 1.0096, False: 1.0093}


def prefetch_scenario(torch, ssd, wl, batches, reps):
    """The output projection behind a communication phase, without and with a side-stream
    L2 prefetch of its weights during that phase ("Part 1 / 4. Prefetching upcoming
    weights into cache"). The phase is dec_sim_comm_wait (the stream busy, HBM idle);
    the prefetch pulls the last `prefetch_bytes` of the weight copy read next. Each mode
    is a graph of R (phase, projection) pairs over the rotating weight copies; the
    projection's time is the pair's minus the phase's."""
    ns = int(PF_WAIT_US * 1000)
    pf_bytes = min(int(PF_WAIT_US * 1e-6 * 5.0e12), int(0.6 * wl.l2)) // 16 * 16
    R = 12
    out = {"wait_us": PF_WAIT_US, "prefetch_bytes": pf_bytes, "prefetch_ctas": 64,
           "weights_bytes": wl.W_o[0].numel() * 2, "per_batch": {}}

    def seq(B, mode):
        d = wl.t[B]
        main = torch.cuda.current_stream()
        for r in range(R):
            W = wl.W_o[r % len(wl.W_o)]
            if mode == "prefetch":
                wl.fork.record(main)
                wl.side.wait_event(wl.fork)
                flat = W.view(-1)
                ssd.l2_prefetch(flat[flat.numel() - pf_bytes // 2:], max_ctas=64, stream=wl.side)
                wl.join.record(wl.side)
            ssd.dec_sim_comm_wait(ns)
            if mode == "prefetch":
                main.wait_event(wl.join)
            if mode != "wait":
                wl.lin(d["x_o"], W, d["r_o"], d["y_o"], d["ws_o"])

    for B in batches:
        t = {}
        for mode in ("wait", "none", "prefetch"):
            g = capture(torch, lambda: seq(B, mode))
            t[mode] = statistics.median(time_graph(torch, g, reps)) / R
            del g
        nb = bytes_linear(B, H, K_O, True)
        o_none, o_pf = t["none"] - t["wait"], t["prefetch"] - t["wait"]
        out["per_batch"][str(B)] = {
            "phase_us": t["wait"], "o_proj_us_after_phase": o_none,
            "o_proj_us_with_prefetch": o_pf, "GBps_after_phase": nb / o_none / 1e3,
            "GBps_with_prefetch": nb / o_pf / 1e3, "speedup": o_none / o_pf}
    return out


# ------------------------------------------- speculative verification rows ----

SPEC_ROWS = (64, 128, 256, 384, 512)


def spec_sweep(torch, ssd, inputs, wl, dev, reps):
    """The decode projections at speculative-decoding verification row counts
    (sequences x (draft length + 1) tokens, up to 512 rows per call; "Part 3: Performance
    Deep Dive", decode with DSpark): wide tensor-core tiles, CUDA graph of R calls over
    the rotating weight copies. Reports HBM GB/s and tensor TFLOP/s (2*M*N*K)."""
    R = 12
    out = {}
    for M in SPEC_ROWS:
        row = {}
        for name, N, K, pool, res in (("input_projection", N_IN, H, wl.W_in, False),
                                      ("output_projection", H, K_O, wl.W_o, True)):
            X = inputs.activations(M, K, dev, 0, "spec_x")
            Rr = inputs.residual(M, N, dev, 0, "spec_r") if res else None
            Y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            ws = ssd.workspace(ssd.dec_linear_workspace_bytes(M, N, K), dev)
            g = capture(torch, lambda: [wl.lin(X, pool[r % len(pool)], Rr, Y, ws)
                                        for r in range(R)])
            us = statistics.median(time_graph(torch, g, reps)) / R
            del g
            nb = bytes_linear(M, N, K, res)
            row[name] = {"us_per_call": us, "GBps": nb / us / 1e3,
                         "TFLOPs": 2.0 * M * N * K / us / 1e6, "tok_per_s": M * 1e6 / us,
                         "variant": ssd.dec_variant_name(ssd.dec_last_variant())}
        out[str(M)] = row
    return out


# --------------------------------------------------------- single skinny GEMM ----

def skinny_sweep(torch, ssd, inputs, dev, l2, reps, packed=False):
    """The single skinny GEMM Y = X . W^T at B = 1, K = 1024, N = 2048 through the batch
    switch (the tiny-matrix kernel: "Part 1 / 1. Tune shapes for the workload", small
    matrices at batch 1-2). Its 4.2 MB of weights fit in L2, so the graph makes one call
    per copy of a pool >= 3x L2: every copy is read again only after the whole pool."""
    B = 1
    W0 = inputs.weight(N_SK, K_SK, dev, 0, "w_skinny")
    if packed:
        W0 = ssd.dec_pack_weight(W0)
    lin = ssd.dec_linear_packed if packed else ssd.dec_linear
    n = max(2, math.ceil(3 * l2 / (W0.numel() * 2)))
    pool = [W0] + [W0.clone() for _ in range(n - 1)]
    X = inputs.activations(B, K_SK, dev, 0, "x_skinny")
    Y = torch.empty(B, N_SK, dtype=torch.bfloat16, device=dev)
    ws = ssd.workspace(ssd.dec_linear_workspace_bytes(B, N_SK, K_SK), dev)
    g = capture(torch, lambda: [lin(X, w, None, Y, ws) for w in pool])
    us = statistics.median(time_graph(torch, g, reps)) / len(pool)
    del g
    nb = bytes_linear(B, N_SK, K_SK, False)
    return {"B": B, "K": K_SK, "N": N_SK, "us_per_call": us, "GBps": nb / us / 1e3,
            "tok_per_s": B * 1e6 / us, "calls_per_graph": len(pool),
            "variant": ssd.dec_variant_name(ssd.dec_last_variant())}


def compact_table(sweep, skinny, batches):
    """Per-(operation, B) figures as flat strings (one value per batch, in the order of
    `batches`), so that a consumer keeping only scalar fields still has them."""
    out = {}
    names = (("input_projection", "in"), ("output_projection", "o"), ("moe_front", "front"),
             ("moe_experts", "experts"))
    for name, short in names:
        rows = [sweep.get(str(B), {}).get(name) for B in batches]
        if not any(rows):
            continue
        fmt = lambda key, f: "/".join("-" if r is None else f(r[key]) for r in rows)
        out[f"{short}_us"] = fmt("us_per_call", lambda v: f"{v:.2f}")
        out[f"{short}_frac"] = fmt("frac", lambda v: f"{v:.3f}")
        out[f"{short}_tok_s"] = fmt("tok_per_s", lambda v: f"{v:.0f}")
    if skinny:
        out["skinny_B1_K1024_N2048"] = (f"us {skinny['us_per_call']:.2f} GBps "
                                        f"{skinny['GBps']:.0f} frac {skinny['frac']:.3f} "
                                        f"tok_s {skinny['tok_per_s']:.0f}")
    out["table_batches"] = "/".join(map(str, batches))
    return out


# -------------------------------------------------------------- CPU baseline ----

def cpu_sample_fn(batches, seed=0):
    """A bounded slice of the step for the fp64 oracle: per batch, 64 rows of the input
    projection, 32 rows of the output projection, the whole front end, and the full
    expert layer (8 routed + shared) for one token. Returns (run(), bytes)."""
    import numpy as np
    import oracle
    rng = np.random.default_rng(seed)

    def bf(shape, std):
        v = (rng.standard_normal(shape) * std).astype(np.float32)
        return (v.view(np.uint32) >> 16).astype(np.uint16)

    w_in = bf((64, H), 0.02)
    w_o = bf((32, K_O), 0.02)
    w_cat = bf((E + L, H), 0.02)
    w_gu = [bf((2 * I, H), 0.02) for _ in range(TOPK + 1)]
    w_d = [bf((H, I), 0.02) for _ in range(TOPK + 1)]
    xs = {B: (bf((B, H), 1.0), bf((B, K_O), 1.0), bf((B, 32), 1.0)) for B in batches}
    nbytes = 0
    for B in batches:
        nbytes += bytes_linear(B, 64, H, False) + bytes_linear(B, 32, K_O, True)
        nbytes += bytes_front(B) + (TOPK + 1) * 3 * I * H * 2 + 2 * H * 2

    def run():
        for B in batches:
            x, xo, r = xs[B]
            oracle.linear(x, w_in)
            oracle.linear(xo, w_o, r)
            f = oracle.moe_front(x, w_cat, E, L, TOPK)
            yp = np.empty((1, TOPK, H))
            for j in range(TOPK):
                _, yp[0, j] = oracle.expert_mlp(x[0], w_gu[j], w_d[j])
            _, s = oracle.expert_mlp(x[0], w_gu[TOPK], w_d[TOPK])
            oracle.combine(f["w"][:1], yp, s[None, :])

    return run, nbytes


SAMPLE_DESC = ("per batch B in {%s}: 64 rows of the input projection, 32 rows of the output "
               "projection (+residual), the whole MoE front end, and one token through 8 routed "
               "experts + the shared expert; fp64 C oracle, OpenMP over output rows")


def cpu_baseline(batches, target_s):
    import oracle
    run, nbytes = cpu_sample_fn(batches)
    t0 = time.perf_counter()
    run()
    one = time.perf_counter() - t0
    reps = max(1, int(target_s / max(one, 1e-3)) - 1)
    t0 = time.perf_counter()
    for _ in range(reps):
        run()
    dt = (time.perf_counter() - t0) / reps
    return {"value": nbytes / dt / 1e9, "unit": "GB/s", "cores": oracle.num_threads(),
            "kind": "oracle", "seconds_per_sample": dt,
            "sample": SAMPLE_DESC % ",".join(map(str, batches))}


# ------------------------------------------------------------------- main ----

def dist_setup(torch):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(torch, world, x, dev):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_replicas(torch, world, ms_local, bytes_local, dev):
    """Whole-job figures of N independent replicas: the step time is the slowest rank's,
    the bytes are every rank's. Returns (ms_max, total_bytes, GB/s)."""
    ms = max_over_ranks(torch, world, ms_local, dev)
    total = bytes_local
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([float(bytes_local)], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        total = float(t.item())
    return ms, total, total / (ms * 1e-3) / 1e9


def barrier(torch, world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    oracle.build()
    batches = [int(b) for b in args.batches.split(",")]
    run, nbytes = cpu_sample_fn(batches)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = (time.perf_counter() - t0) / args.steps
    v = nbytes / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "batches": batches,
                       "sample": "bounded host sample of the step (see cpu_baseline.sample)"},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": oracle.num_threads(),
                             "kind": "oracle",
                             "sample": SAMPLE_DESC % ",".join(map(str, batches))},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    import torch
    world, rank, local = dist_setup(torch)
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    import split_switched_decode_gb300 as ssd
    from split_switched_decode_gb300 import inputs
    ssd.build()
    batches = [int(b) for b in args.batches.split(",")]
    ops = set(args.ops.split(","))
    if not args.sweep_only:
        ops = {"in", "o", "front", "experts", "pfscen", "spec", "skinny"}
    wl = Workload(torch, ssd, inputs, dev, batches, num_experts=args.num_experts,
                  experts="experts" in ops, packed=not args.row_major)
    # Measured (graphs of 3 layers, B = 1/4/16/64): front end + experts as separate calls
    # 147.0 / 441.3 / 1437.7 / 3615.5 us; with the L2 prefetch of the shared expert's
    # weights during the front end 152.1 / 443.1 / 1440.6 / 3623.9; as moe_layer 149.2 /
    # 443.3 / 1441.8 / 3621.9. The front end is latency-bound and on the critical path:
    # any traffic next to it slows it more than it saves later. The prefetch is measured
    # where it pays, behind a communication phase (prefetch_scenario).
    wl.prefetch = args.prefetch
    wl.layer = args.layer

    # routing of every X set (fixed inputs -> fixed routing -> fixed bytes); not needed
    # when only projections are swept (profiler captures of those see only their kernels)
    if ops & {"front", "experts"}:
        for B in batches:
            for v in range(3):
                wl.op_front(B, v=v, prefetch=False, with_map=True)
    torch.cuda.synchronize()

    # ---- per-operation sweep: graphs of R calls over rotating weight copies
    sweep = {}
    R_SMALL = 12
    for B in ([] if args.step_only else batches):
        row = {}
        for key, name, fn, nb in (
                ("in", "input_projection", lambda B=B: [wl.op_in(B, r) for r in range(R_SMALL)],
                 bytes_linear(B, N_IN, H, False)),
                ("o", "output_projection", lambda B=B: [wl.op_o(B, r) for r in range(R_SMALL)],
                 bytes_linear(B, H, K_O, True)),
                ("front", "moe_front", lambda B=B: [wl.op_front(B, r, v=0, prefetch=False)
                                                    for r in range(R_SMALL)],
                 bytes_front(B, wl.E))):
            if key not in ops:
                continue
            g = capture(torch, fn)
            ts = time_graph(torch, g, args.reps)
            us = statistics.median(ts) / R_SMALL
            row[name] = {"us_per_call": us, "GBps": nb / us / 1e3, "tok_per_s": B * 1e6 / us,
                         "variant": ssd.dec_variant_name(ssd.dec_last_variant())}
            del g
        if "experts" in ops:
            g = capture(torch, lambda B=B: [wl.op_experts(B, v) for v in range(3)])
            ts = time_graph(torch, g, max(3, args.reps - 2))
            nb_e = sum(bytes_experts(B, wl.used_experts(B, v)) for v in range(3)) / 3
            us = statistics.median(ts) / 3
            row["moe_experts"] = {"us_per_call": us, "GBps": nb_e / us / 1e3,
                                  "tok_per_s": B * 1e6 / us,
                                  "distinct_experts": [wl.used_experts(B, v) for v in range(3)]}
            del g
        sweep[str(B)] = row
    torch.cuda.synchronize()
    skinny = None
    if "skinny" in ops and not args.step_only:
        # config 1 is the tiny kernel's own case: its row-major weights as given
        skinny = skinny_sweep(torch, ssd, inputs, dev, wl.l2, args.reps, packed=False)
    spec = None
    if "spec" in ops and not args.step_only:
        spec = spec_sweep(torch, ssd, inputs, wl, dev, args.reps)
    pfscen = None
    if "pfscen" in ops and not args.step_only:
        pfscen = prefetch_scenario(torch, ssd, wl, [b for b in (1, 64) if b in batches],
                                   max(3, args.reps))
    if args.sweep_only:
        if rank == 0:
            print(json.dumps({"sweep_only": True, "batches": batches, "ops": sorted(ops),
                              "num_experts": wl.E, "sweep": sweep, "skinny_gemm": skinny,
                              "prefetch_scenario": pfscen, "spec_rows": spec}), flush=True)
        return 0

    # ---- the step as one CUDA graph
    launches0 = wl.launches
    g_step = capture(torch, wl.step)
    per_step_launches = (wl.launches - launches0) // 2
    step_bytes = wl.step_bytes()
    for _ in range(args.warmup):
        g_step.replay()
    torch.cuda.synchronize()
    clk = ClockSampler(local)
    clk.start()
    barrier(torch, world)
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    for _ in range(args.steps):
        g_step.replay()
    b.record(st)
    torch.cuda.synchronize()
    barrier(torch, world)
    clocks = clk.stop()
    ms = a.elapsed_time(b) / args.steps
    ms, _, value = aggregate_replicas(torch, world, ms, step_bytes, dev)
    assert ssd.dec_sync_status() == ssd.DEC_OK
    if args.step_only:
        if rank == 0:
            print(json.dumps({"step_only": True, "value": value, "unit": "GB/s", "ms_per_step": ms,
                              "batches": batches, "num_experts": wl.E,
                              "moe_call": "moe_layer" if wl.layer else "moe_front + moe_experts",
                              "l2_prefetch": wl.prefetch and not wl.layer}), flush=True)
        return 0

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        host_in = {B: {k: wl.t[B][k].cpu().pin_memory() for k in ("x_in", "x_o", "r_o")}
                   for B in batches}
        for B in batches:
            host_in[B]["x_moe"] = wl.t[B]["x_moe"][0].cpu().pin_memory()
        host_out = {B: {k: torch.empty(wl.t[B][k].shape, dtype=wl.t[B][k].dtype).pin_memory()
                        for k in ("y_in", "y_o", "y_moe")} for B in batches}
        h2d = sum(t.numel() * t.element_size() for d in host_in.values() for t in d.values())
        d2h = sum(t.numel() * t.element_size() for d in host_out.values() for t in d.values())

        def e2e_step():
            for B in batches:
                d, hi, ho = wl.t[B], host_in[B], host_out[B]
                d["x_in"].copy_(hi["x_in"], non_blocking=True)
                d["x_o"].copy_(hi["x_o"], non_blocking=True)
                d["r_o"].copy_(hi["r_o"], non_blocking=True)
                d["x_moe"][0].copy_(hi["x_moe"], non_blocking=True)
                wl.op_in(B)
                wl.op_o(B)
                wl.op_moe(B)
                ho["y_in"].copy_(d["y_in"], non_blocking=True)
                ho["y_o"].copy_(d["y_o"], non_blocking=True)
                ho["y_moe"].copy_(d["y_moe"], non_blocking=True)

        for _ in range(max(1, args.warmup)):
            e2e_step()
        torch.cuda.synchronize()
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ea.record(st)
        for _ in range(args.steps):
            e2e_step()
        eb.record(st)
        torch.cuda.synchronize()
        ems, _, evalue = aggregate_replicas(torch, world, ea.elapsed_time(eb) / args.steps,
                                            step_bytes, dev)
        e2e = {"value": evalue, "unit": "GB/s",
               "ms_per_step": ems, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "path": "eager public-API calls, pinned host inputs/outputs copied every step"}

    # ---- roofline of the dominant operation (routed + shared expert GEMV at the largest B)
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except OSError:
        pass
    peak = peaks.get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    peak = peak or 6800.0
    Bmax = str(max(batches))
    dom = sweep[Bmax]["moe_experts"]
    # DRAM bytes per call / algorithmic bytes, from one ncu capture of the same kernels
    # on a 32-expert bank (profiles/moe_experts_traffic_B64_E32.md), scaled to the call
    nb_dom = statistics.mean(bytes_experts(int(Bmax), u) for u in dom["distinct_experts"])
    roofline = {"bound": "hbm", "kernel": f"moe_experts grouped expert GEMV, B={Bmax}",
                "achieved": dom["GBps"], "peak": peak, "peak_source": peak_src, "unit": "GB/s",
                "frac": dom["GBps"] / peak, "traffic": EXPERTS_TRAFFIC_RATIO[wl.packed] * nb_dom,
                "traffic_unit": "bytes per call"}
    # context for `frac`: the read-only HBM rate (every SM streaming a contiguous share
    # of 4 GiB in 16 KB bulk copies; the copy peak above counts read and written bytes)
    rs_buf = torch.empty(4 << 30, dtype=torch.uint8, device=dev)
    ssd.dec_read_stream(rs_buf)
    torch.cuda.synchronize()
    rs_t = []
    for _ in range(5):
        ra, rb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ra.record()
        rs_n = ssd.dec_read_stream(rs_buf)
        rb.record()
        torch.cuda.synchronize()
        rs_t.append(ra.elapsed_time(rb))
    del rs_buf
    roofline["read_stream_gbs"] = rs_n / (min(rs_t) * 1e-3) / 1e9
    roofline["frac_of_read_stream"] = dom["GBps"] / roofline["read_stream_gbs"]
    for Bk, row in sweep.items():
        for op in row.values():
            op["frac"] = op["GBps"] / peak
    if skinny:
        skinny["frac"] = skinny["GBps"] / peak
    tc_peak = peaks.get("bf16_tflops") or 1900.0
    for Mk, row in (spec or {}).items():
        for op in row.values():
            op["frac_hbm"] = op["GBps"] / peak
            op["frac_tensor"] = op["TFLOPs"] / tc_peak

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        cpu = cpu_baseline(batches, args.cpu_seconds)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16", "data": "synthetic",
                "config": {"workload": WORKLOAD, "batches": batches, "step_bytes": step_bytes,
                           "l2": "cold: every weight tensor is re-read only after >3x L2 of "
                                 "other weight traffic (step), rotating copies >=3x L2 (sweep)",
                           "timing": "CUDA graph replay, CUDA events on the replay stream",
                           "moe_call": ("moe_layer (shared expert overlapping the front end)"
                                        if wl.layer else
                                        "moe_front + l2_prefetch + moe_experts" if wl.prefetch
                                        else "moe_front + moe_experts"),
                           "l2_prefetch_in_step": wl.prefetch and not wl.layer,
                           "parallelism": f"replicas x{world}",
                           "weights": ("row-major" if not wl.packed else
                                       "projection weights and expert banks tile-packed once "
                                       "at load (dec_pack_weight, dec_pack_expert_weights): "
                                       "16 KB blocks of 128 rows x 64 k; front-end W_cat "
                                       "row-major"),
                           **compact_table(sweep, skinny, batches)},
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": per_step_launches * args.steps, "clocks": clocks,
                "sweep": sweep, "skinny_gemm": skinny, "prefetch_scenario": pfscen,
                "spec_rows": spec}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
