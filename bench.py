#!/usr/bin/env python3
"""Decode-step benchmark of the affine group-quantized projection path.

Workload (one step): a 48-layer dense projection stack at M=1 token, u4
codes, group 64, bf16 scales/biases.  Each layer runs four library calls:
  fused QKV   5120 -> 5120+1024+1024  (gwa_qmv_fused_sections, Q/K/V buffers)
  o_proj      5120 -> 5120            (gwa_qmv_affine, reads Q)
  gate+up     5120 -> 2x13824, SiLU   (gwa_qmv_gate_up_silu, reads o)
  down        13824 -> 5120           (gwa_qmv_affine, reads h)
so 192 launches and 7.43 GB of packed weights per step, far above the 129 MB
L2: every step streams its weights from HBM.  Each layer's QKV reads the step
input x; every other call reads the output of the call just before it, as in
a decode step.  A step is one CUDA graph of the 192 launches in layer order
(QKV, o, gate+up, down of layer 0, then layer 1, ...), so consecutive
kernels overlap through programmatic dependent launch exactly as they would
in a model.  The per-kernel breakdown comes from a second timed region that
replays one graph per projection type (48 launches each) with CUDA events
between the graphs.

Metric: achieved HBM GB/s of algorithmic bytes (packed codes + scales +
biases + activations) and the equivalent 48-layer decode steps/s.

--impl reference times the CPU oracle (fp64, all host cores) on a bounded
sample of the same workload: one layer's four projections per step.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HIDDEN, QOUT, KVOUT, INTER, LAYERS = 5120, 5120, 1024, 13824, 48
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gwa", choices=["gwa", "reference"])
    ap.add_argument("--bits", type=int, default=4, choices=[4, 8])
    ap.add_argument("--tokens", type=int, default=1)
    ap.add_argument("--layers", type=int, default=LAYERS)
    ap.add_argument("--inputs", default="normal", choices=["chain", "normal"],
                    help="normal: every projection reads its own fixed "
                         "N(0,1) activations (the workload's x ~ N(0,1)); "
                         "chain: each projection reads the previous one's "
                         "output (q -> o -> gate+up -> down)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the secondary workloads (M=4, M=512, MoE)")
    ap.add_argument("--only-extra", default=None,
                    choices=["attention", "quantize", "moe", "formats"],
                    help="run one standalone secondary workload for --steps "
                         "after --warmup replays, print its figures and exit "
                         "(for profiling; not the bench line)")
    ap.add_argument("--lengths", default=None,
                    help="--only-extra attention: comma-separated cache lengths")
    return ap.parse_args()


# ---------------------------------------------------------------- workload
def proj_bytes(rows: int, K: int, bits: int, M: int) -> int:
    """Algorithmic bytes of one projection call: packed codes + scales +
    biases + activations (outputs excluded)."""
    return rows * K * bits // 8 + 2 * 2 * rows * (K // 64) + 2 * M * K


def layer_shapes():
    return [("qkv", QOUT + 2 * KVOUT, HIDDEN), ("o", HIDDEN, QOUT),
            ("gate_up", 2 * INTER, HIDDEN), ("down", HIDDEN, INTER)]


def layer_bytes(bits: int, M: int) -> dict:
    return {n: proj_bytes(r, k, bits, M) for n, r, k in layer_shapes()}


def workload_config(args) -> dict:
    return {
        "workload": (f"{args.layers}-layer dense decode projection stack, "
                     f"M={args.tokens}, u{args.bits} group 64 bf16 scale/bias:"
                     " fused QKV 5120->5120+1024+1024, o_proj 5120->5120, "
                     "fused gate+up 5120->2x13824 with SiLU(gate)*up, "
                     "down 13824->5120; 4 calls per layer"),
        "layers": args.layers, "M": args.tokens, "bits": args.bits,
        "group": 64, "hidden": HIDDEN, "intermediate": INTER,
        "l2": "inputs larger than L2: every step streams "
              f"{sum(layer_bytes(args.bits, args.tokens).values()) * args.layers / 1e9:.2f}"
              " GB of distinct weights (L2 is 129 MB)",
        "parallelism": f"replicas x{args.gpus}" if args.gpus > 1 else "single",
        "inputs": ("chained: o reads q, gate+up reads o, down reads h = "
                   "SiLU(gate) * up" if args.inputs == "chain"
                   else "each projection reads fixed N(0,1) activations"),
    }


def kernel_sources_sha256() -> str:
    """Hash of the decode kernel's sources; a recorded ncu traffic figure is
    only reported while the sources it was taken on are unchanged."""
    import hashlib
    h = hashlib.sha256()
    for f in ("qmv_group.cu", "group_dot.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "group_wise_affine_gb300", "csrc", f),
                  "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def recorded_traffic(kernel: str):
    """DRAM bytes per launch (read + write) recorded from one ncu capture in
    profiles/, or None when absent or taken on other kernel sources."""
    path = os.path.join(ROOT, "profiles", "qmv_group_gate_up_27648x5120_m1.md")
    if kernel != "gate_up" or not os.path.exists(path):
        return None
    traffic = sha = None
    with open(path) as f:
        for ln in f:
            if ln.startswith("traffic per launch (bytes):"):
                traffic = int(ln.split(":")[1].strip())
            if ln.startswith("kernel sources sha256:"):
                sha = ln.split(":")[1].strip()
    if traffic is None or sha != kernel_sources_sha256():
        return None
    return traffic


def _measured_tflops():
    """Dense fp16/bf16 tensor peak for a kernel timed inside a long step
    (the sustained figure; fp16 and bf16 share the nominal rate)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained"]), "measured sustained bf16"
    except Exception:
        return 1700.0, "fallback sustained"


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def mark(self, start: bool):
        if start:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "note": "nvidia-smi unavailable"}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        rows = [r.split(",") for r in out.strip().splitlines() if r.strip()]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- GPU arm
def run_gwa(args, rank: int, world: int, local_rank: int):
    import torch
    import group_wise_affine_gb300 as gwa
    import gwa_synth as synth

    gwa.load()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    M, bits, L = args.tokens, args.bits, args.layers

    W = stack_weights(bits, L, dev)
    g = torch.Generator(device=dev)
    g.manual_seed(12345 + rank)
    x = torch.randn((M, HIDDEN), generator=g, device=dev).to(torch.bfloat16)
    bufs = []
    for l in range(L):
        bufs.append(dict(
            q=torch.empty((M, QOUT), dtype=torch.bfloat16, device=dev),
            k=torch.empty((M, KVOUT), dtype=torch.bfloat16, device=dev),
            v=torch.empty((M, KVOUT), dtype=torch.bfloat16, device=dev),
            o=torch.empty((M, HIDDEN), dtype=torch.bfloat16, device=dev),
            h=torch.empty((M, INTER), dtype=torch.bfloat16, device=dev),
            y=torch.empty((M, HIDDEN), dtype=torch.bfloat16, device=dev)))
    ws = gwa.make_workspace(M, INTER, dev)   # None at decode sizes
    fixed = None
    if args.inputs == "normal":
        fixed = {k: torch.randn((M, n), generator=g, device=dev).to(torch.bfloat16)
                 for k, n in (("o", QOUT), ("gate_up", HIDDEN), ("down", INTER))}

    def src(kind, b):
        if fixed is not None:
            return fixed[kind]
        return {"o": b["q"], "gate_up": b["o"], "down": b["h"]}[kind]

    def call(kind, l, stream=None):
        w, b = W[l], bufs[l]
        if kind == "qkv":
            gwa.qmv_fused_sections(x, w["qkv"], (QOUT, KVOUT, KVOUT),
                                   outs=[b["q"], b["k"], b["v"]],
                                   workspace=ws, stream=stream)
        elif kind == "o":
            gwa.qmv_affine(src("o", b), w["o"], y=b["o"], workspace=ws,
                           stream=stream)
        elif kind == "gate_up":
            gwa.qmv_gate_up_silu(src("gate_up", b), w["gate_up"], h=b["h"],
                                 workspace=ws, stream=stream)
        else:
            gwa.qmv_affine(src("down", b), w["down"], y=b["y"], workspace=ws,
                           stream=stream)

    kinds = ["qkv", "o", "gate_up", "down"]
    for k in kinds:                       # eager warm-up (sets up the library)
        call(k, 0)
    torch.cuda.synchronize()

    side = torch.cuda.Stream(device=dev)
    gstep = torch.cuda.CUDAGraph()           # one step, layer order
    with torch.cuda.graph(gstep, stream=side):
        for l in range(L):
            for k in kinds:
                call(k, l)
    graphs = {}                              # per projection type
    for k in kinds:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr, stream=side):
            for l in range(L):
                call(k, l)
        graphs[k] = gr
    torch.cuda.synchronize()

    def step():
        gstep.replay()

    st = torch.cuda.current_stream()
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()

    clocks = ClockSampler(local_rank if world == 1 else
                          int(os.environ.get("LOCAL_RANK", 0)))
    clocks.start()
    time.sleep(0.3)
    K = args.steps
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.mark(True)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(st)
    for i in range(K):
        step()
    end.record(st)
    torch.cuda.synchronize()
    clocks.mark(False)
    total_ms = start.elapsed_time(end)
    if world > 1:
        torch.distributed.barrier()
    clk = clocks.stop()

    # per-kernel breakdown: the four per-type graphs with events between
    KB = max(3, min(K, 100))
    for _ in range(3):
        for k in kinds:
            graphs[k].replay()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)]
          for _ in range(KB)]
    torch.cuda.synchronize()
    for i in range(KB):
        ev[i][0].record(st)
        for j, k in enumerate(kinds):
            graphs[k].replay()
            ev[i][j + 1].record(st)
    torch.cuda.synchronize()
    per_kind_ms = {k: sum(ev[i][j].elapsed_time(ev[i][j + 1])
                          for i in range(KB)) / KB for j, k in enumerate(kinds)}

    # end to end: pinned host input in, step, result back out
    x_host = torch.empty((M, HIDDEN), dtype=torch.bfloat16).pin_memory()
    x_host.copy_(x.cpu())
    y_host = torch.empty((M, HIDDEN), dtype=torch.bfloat16).pin_memory()
    KE = max(3, min(K, 50))
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t_wall = time.perf_counter()
    e0.record(st)
    for _ in range(KE):
        x.copy_(x_host, non_blocking=True)
        step()
        y_host.copy_(bufs[-1]["y"], non_blocking=True)
    e1.record(st)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    e2e_ms = e0.elapsed_time(e1) / KE
    # the same with the 192 calls issued eagerly each step (no graph): the
    # host-side cost of the binding and the C ABI included
    KG = max(3, min(K, 20))
    for _ in range(2):
        for l in range(L):
            for k in kinds:
                call(k, l, stream=st)
    torch.cuda.synchronize()
    t_eager = time.perf_counter()
    e0.record(st)
    for _ in range(KG):
        x.copy_(x_host, non_blocking=True)
        for l in range(L):
            for k in kinds:
                call(k, l, stream=st)
        y_host.copy_(bufs[-1]["y"], non_blocking=True)
    e1.record(st)
    torch.cuda.synchronize()
    t_eager = time.perf_counter() - t_eager
    eager_ms = e0.elapsed_time(e1) / KG
    extras = {}
    if not args.no_extras and bits == 4 and L == LAYERS and M == 1:
        # chained activations: down reads h = SiLU(gate) * up, whose spread
        # marks most of its groups (the exact two-plane path)
        extras["stack_M1_chained"] = run_stack_extra(W, 1, dev, 50, 3, "chain")
        extras["stack_M2"] = run_stack_extra(W, 2, dev, 50, 3)
        extras["stack_M4"] = run_stack_extra(W, 4, dev, 50, 3)
        extras["stack_M8"] = run_stack_extra(W, 8, dev, 30, 3)
        extras["qkv_rope"] = run_rope_extra(W, dev, 20, 3)
        extras["prefill_stack_M512"] = run_stack_extra(W, 512, dev, 5, 2)
        # the same stack with u8 codes (its own 14 GB of weights)
        W8 = stack_weights(8, L, dev)
        extras["stack_u8_M1"] = run_stack_extra(W8, 1, dev, 50, 3)
        extras["stack_u8_M4"] = run_stack_extra(W8, 4, dev, 30, 3)
        extras["stack_u8_M8"] = run_stack_extra(W8, 8, dev, 30, 3)
        extras["prefill_stack_u8_M512"] = run_stack_extra(W8, 512, dev, 5, 2)
        del W8
        torch.cuda.empty_cache()
        extras["moe"] = run_moe_extra(dev, 50, 3)
        extras["quantize"] = run_quantize_extra(dev, 20, 3)
        extras["formats"] = run_formats_extra(dev, 10, 2)
        extras["attention"] = run_attention_extra(dev, 20, 3)
    return dict(total_ms=total_ms, per_kind_ms=per_kind_ms, clocks=clk,
                e2e_ms=e2e_ms, e2e_wall_ms=1e3 * t_wall / KE,
                eager_ms=eager_ms, eager_wall_ms=1e3 * t_eager / KG,
                h2d=M * HIDDEN * 2, d2h=M * HIDDEN * 2,
                launches=K * 4 * L, extras=extras)


# ---------------------------------------------------------------- extras
def time_graphs(graphs, steps, warmup):
    """Replays the graphs in order `steps` times; returns (total ms, per-graph
    ms summed over steps), timed with CUDA events on the current stream."""
    import torch
    st = torch.cuda.current_stream()
    for _ in range(warmup):
        for g in graphs:
            g.replay()
    torch.cuda.synchronize()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(graphs) + 1)]
          for _ in range(steps)]
    for i in range(steps):
        ev[i][0].record(st)
        for j, g in enumerate(graphs):
            g.replay()
            ev[i][j + 1].record(st)
    torch.cuda.synchronize()
    per = [sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(steps))
           for j in range(len(graphs))]
    return sum(per), per


def capture(fn):
    import torch
    side = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        fn()
    return g


def stack_weights(bits: int, L: int, dev):
    """The stack's weights: one seeded draw per layer and projection, made
    on the device."""
    import group_wise_affine_gb300 as gwa
    import gwa_synth as synth
    W = []
    for l in range(L):
        layer = {}
        for p, (name, rows, K) in enumerate(layer_shapes()):
            wq, s, b = synth.device_qweight(synth.stack_seed(l, p, bits), rows,
                                            K, bits, device=dev)
            layer[name] = gwa.QWeight(wq, s, b, rows, K, bits, 64)
        W.append(layer)
    return W


def run_stack_extra(W, M, dev, steps, warmup, inputs="normal"):
    """The same 48-layer stack (same weights) at M tokens per call; inputs
    as the --inputs option."""
    import torch
    import group_wise_affine_gb300 as gwa
    L = len(W)
    g = torch.Generator(device=dev)
    g.manual_seed(777 + M)
    x = torch.randn((M, HIDDEN), generator=g, device=dev).to(torch.bfloat16)
    mk = lambda n: torch.empty((M, n), dtype=torch.bfloat16, device=dev)
    bufs = [dict(q=mk(QOUT), k=mk(KVOUT), v=mk(KVOUT), o=mk(HIDDEN),
                 h=mk(INTER), y=mk(HIDDEN)) for _ in range(L)]
    ws = gwa.make_workspace(M, INTER, dev)
    fixed = None
    if inputs == "normal":
        fixed = {k: torch.randn((M, n), generator=g, device=dev).to(torch.bfloat16)
                 for k, n in (("o", QOUT), ("gate_up", HIDDEN), ("down", INTER))}

    def src(kind, b):
        if fixed is not None:
            return fixed[kind]
        return {"o": b["q"], "gate_up": b["o"], "down": b["h"]}[kind]

    def call(kind, l):
        w, b = W[l], bufs[l]
        if kind == "qkv":
            gwa.qmv_fused_sections(x, w["qkv"], (QOUT, KVOUT, KVOUT),
                                   outs=[b["q"], b["k"], b["v"]], workspace=ws)
        elif kind == "o":
            gwa.qmv_affine(src("o", b), w["o"], y=b["o"], workspace=ws)
        elif kind == "gate_up":
            gwa.qmv_gate_up_silu(src("gate_up", b), w["gate_up"], h=b["h"],
                                 workspace=ws)
        else:
            gwa.qmv_affine(src("down", b), w["down"], y=b["y"], workspace=ws)

    kinds = ["qkv", "o", "gate_up", "down"]
    for k in kinds:
        call(k, 0)
    torch.cuda.synchronize()
    graphs = [capture(lambda k=k: [call(k, l) for l in range(L)]) for k in kinds]
    total, per = time_graphs(graphs, steps, warmup)
    ms = total / steps
    shapes = {n: (r, k) for n, r, k in layer_shapes()}
    out = {"M": M, "inputs": inputs, "ms_per_step": round(ms, 4),
           "steps_per_s": round(1e3 / ms, 2), "kernels": {}}
    flops = 0
    bytes_ = 0
    for (kind, t) in zip(kinds, per):
        rows, K = shapes[kind]
        us = 1e3 * t / (steps * L)
        f = 2.0 * M * rows * K
        b = proj_bytes(rows, K, W[0][kind].bits, M)
        flops += f * L
        bytes_ += b * L
        out["kernels"][kind] = {"us_per_launch": round(us, 3),
                                "TFLOP/s": round(f / us / 1e6, 1),
                                "GB/s": round(b / us / 1e3, 1)}
    out["TFLOP/s"] = round(flops / (ms * 1e-3) / 1e12, 1)
    out["GB/s"] = round(bytes_ / (ms * 1e-3) / 1e9, 1)
    out["bits"] = W[0]["qkv"].bits
    out["frac_of_measured_hbm"] = round(out["GB/s"] / measured_peak()[0], 4)
    out["timing"] = "per projection type: one graph of its 48 launches"
    return out


def run_moe_extra(dev, steps, warmup, layers=16, E=256, H=2048, I=512,
                  topk=8, tokens=(1, 8)):
    """MoE expert GEMV: per layer one gate+up SiLU call and one down+combine
    call over that layer's own stacked experts (16 layers x 256 experts, so
    replays do not find the touched experts still in L2)."""
    import torch
    import group_wise_affine_gb300 as gwa
    import gwa_synth as synth
    pools = []
    for l in range(layers):
        gu = gwa.QWeight(*synth.device_qweight(50000 + 2 * l, E * 2 * I, H, 4,
                                               device=dev), E * 2 * I, H, 4, 64)
        dn = gwa.QWeight(*synth.device_qweight(50001 + 2 * l, E * H, I, 4,
                                               device=dev), E * H, I, 4, 64)
        pools.append((gwa.expert_view(gu, E), gwa.expert_view(dn, E)))
    res = {}
    per_expert = proj_bytes(2 * I, H, 4, 0) + proj_bytes(H, I, 4, 0)
    for M in tokens:
        ids_l, rw_l, bufs = [], [], []
        distinct = 0
        for l in range(layers):
            ids, rw = synth.routing(60000 + 100 * M + l, M, topk, E)
            distinct += len(set(ids.reshape(-1).tolist()))
            ids_l.append(torch.from_numpy(ids).to(dev))
            rw_l.append(torch.from_numpy(rw).to(dev))
            bufs.append(dict(
                x=torch.randn((M, H), device=dev).to(torch.bfloat16),
                h=torch.empty((M, topk, I), dtype=torch.bfloat16, device=dev),
                y=torch.empty((M, H), dtype=torch.bfloat16, device=dev)))

        def step():
            for l in range(layers):
                gu, dn = pools[l]
                b = bufs[l]
                gwa.moe_qmv_gather(b["x"], ids_l[l], gu, E, 0, out=b["h"])
                gwa.moe_qmv_gather(b["h"], ids_l[l], dn, E, 1,
                                   route_w=rw_l[l], out=b["y"])
        step()
        torch.cuda.synchronize()
        total, _ = time_graphs([capture(step)], steps, warmup)
        ms = total / steps
        act = layers * (M * H * 2 + M * topk * I * 2)
        byt = distinct * per_expert + act
        res[f"M{M}"] = {"us_per_layer": round(1e3 * ms / layers, 3),
                        "distinct_experts_per_layer": round(distinct / layers, 2),
                        "GB/s": round(byt / (ms * 1e-3) / 1e9, 1)}
    return res


def run_rope_extra(W, dev, steps, warmup, tokens=(1, 4, 512),
                   head_dim=128, base=1e6):
    """The 48 layers' fused QKV projections with the rotary embedding of Q
    and K (heads of 128, base 1e6, positions 1000 + m), against the same
    projections without it: per-launch time of each and the difference."""
    import torch
    import group_wise_affine_gb300 as gwa
    L = len(W)
    res = {}
    for M in tokens:
        g = torch.Generator(device=dev).manual_seed(4000 + M)
        x = torch.randn((M, HIDDEN), generator=g, device=dev).to(torch.bfloat16)
        pos = torch.arange(1000, 1000 + M, dtype=torch.int32, device=dev)
        mk = lambda n: torch.empty((M, n), dtype=torch.bfloat16, device=dev)
        outs = [[mk(QOUT), mk(KVOUT), mk(KVOUT)] for _ in range(L)]
        ws = gwa.make_workspace(M, HIDDEN, dev)
        rws = torch.empty(max(int(gwa.load().gwa_qkv_rope_workspace_bytes(
            M, HIDDEN, head_dim)), 256), dtype=torch.uint8, device=dev)

        def plain():
            for l in range(L):
                gwa.qmv_fused_sections(x, W[l]["qkv"], (QOUT, KVOUT, KVOUT),
                                       outs=outs[l], workspace=ws)

        def rope():
            for l in range(L):
                gwa.qmv_qkv_rope(x, W[l]["qkv"], QOUT, KVOUT, head_dim, base,
                                 pos, outs=outs[l], workspace=rws)
        plain()
        rope()
        torch.cuda.synchronize()
        total, per = time_graphs([capture(plain), capture(rope)], steps, warmup)
        us = [1e3 * t / (steps * L) for t in per]
        byt = proj_bytes(QOUT + 2 * KVOUT, HIDDEN, W[0]["qkv"].bits, M)
        res[f"M{M}"] = {"us_per_launch_rope": round(us[1], 3),
                        "us_per_launch_plain": round(us[0], 3),
                        "rope_extra_us": round(us[1] - us[0], 3),
                        "GB/s_rope": round(byt / (us[1] * 1e-6) / 1e9, 1)}
    return res


def run_formats_extra(dev, steps, warmup, N=27648, K=5120,
                      formats=((2, 64), (3, 64), (6, 64), (4, 32), (4, 128),
                               (0x108, 64))):
    """The gate+up shape (27648 x 5120, one token, SiLU epilogue) in code
    widths and group sizes outside group 64: u2, u3 and u6 on the
    general-format decode kernel, u4 in groups of 32 and 128 on the
    one-token chunk kernel, fp8 (e4m3, bits 0x108) on the general kernel's
    fp32 form; eight back-to-back launches over distinct weights so the
    timed bytes stream from HBM."""
    import torch
    import group_wise_affine_gb300 as gwa
    import gwa_synth as synth
    peak, _ = measured_peak()
    g = torch.Generator(device=dev).manual_seed(55)
    x = torch.randn((1, K), generator=g, device=dev).to(torch.bfloat16)
    h = torch.empty((1, N // 2), dtype=torch.bfloat16, device=dev)
    res = {}
    for bits, group in formats:
        ws = [gwa.QWeight(*synth.device_qweight(7000 + 10 * bits + group + c, N,
                                                K, bits, group, device=dev),
                          N, K, bits, group) for c in range(8)]
        graph = capture(lambda: [gwa.qmv_gate_up_silu(x, w, h=h) for w in ws])
        total, _ = time_graphs([graph], steps, warmup)
        us = 1e3 * total / (steps * len(ws))
        width = 8 if bits == 0x108 else bits
        byt = proj_bytes(N, K, width, 1) if group == 64 else (
            N * K * width // 8 + N * (K // group) * 4 + K * 2)
        gbs = byt / (us * 1e-6) / 1e9
        name = f"fp8_g{group}" if bits == 0x108 else f"u{bits}_g{group}"
        res[name] = {"us_per_launch": round(us, 2),
                                     "GB/s": round(gbs, 1),
                                     "frac_of_measured_hbm": round(gbs / peak, 4)}
        del ws
    return res


def run_attention_extra(dev, steps, warmup, lengths=(4096, 32768, 131072),
                        Hq=40, Hkv=8, D=128, bits=4):
    """Decode attention over a u4 value cache (one query per head, 40 query
    heads over 8 KV heads of 128): bytes = bf16 K + packed V + scales and
    biases + q + out; distinct caches per launch (more bytes than L2 across
    one pass) so they stream from HBM.  Short caches show the per-call
    latency (two dependent kernels), long ones the streaming rate."""
    import torch
    import group_wise_affine_gb300 as gwa
    peak, _ = measured_peak()
    res = {}
    for T in lengths:
        ncache = max(2, int(512e6 // (Hkv * T * (2 * D + D * bits // 8 + 4))))
        ncache = min(ncache, 16)
        g = torch.Generator(device=dev).manual_seed(9000 + T)
        q = torch.randn((1, Hq, 1, D), generator=g, device=dev).to(torch.bfloat16)
        caches = []
        for c in range(ncache):
            k = torch.randn((1, Hkv, T, D), generator=g, device=dev).to(torch.bfloat16)
            vq = torch.randint(-2**31, 2**31 - 1, (1, Hkv, T, D * bits // 32),
                               generator=g, device=dev, dtype=torch.int32)
            vs = (torch.rand((1, Hkv, T, D // 64), generator=g, device=dev) * 0.04
                  + 0.01).to(torch.bfloat16)
            vb = (-vs.float() * 7.5).to(torch.bfloat16)
            caches.append((k, vq, vs, vb))
        out = torch.empty((1, Hq, 1, D), dtype=torch.bfloat16, device=dev)
        ws = torch.empty(int(gwa.load().gwa_sdpa_workspace_bytes(1, Hq, Hkv, 1, T, D)),
                         dtype=torch.uint8, device=dev)
        graph = capture(lambda: [gwa.sdpa_dequant_v(q, *c, bits=bits, out=out,
                                                    workspace=ws) for c in caches])
        total, _ = time_graphs([graph], steps, warmup)
        us = 1e3 * total / (steps * ncache)
        byt = Hkv * T * (2 * D + D * bits // 8 + 4) + 2 * 2 * Hq * D
        gbs = byt / (us * 1e-6) / 1e9
        res[f"T{T}"] = {"us_per_call": round(us, 2), "GB/s": round(gbs, 1),
                        "frac_of_measured_hbm": round(gbs / peak, 4),
                        "bytes_per_call": byt}
        del caches
    return res


def run_quantize_extra(dev, steps, warmup, N=27648, K=5120):
    """Affine quantization (the requantize step of a LoRA merge) of the
    gate+up weight, bf16 [N, K] -> u4 and u8: bandwidth-bound, bytes = the
    bf16 input read plus codes, scales and biases written.  The input (283
    MB) exceeds L2, so back-to-back launches stream from HBM."""
    import torch
    import group_wise_affine_gb300 as gwa
    g = torch.Generator(device=dev).manual_seed(4242)
    w = (torch.randn((N, K), generator=g, device=dev) * 0.05).to(torch.bfloat16)
    peak, _ = measured_peak()
    res = {}
    for bits in (4, 8):
        out = gwa.quantize_affine(w, bits=bits)
        graph = capture(lambda: gwa.quantize_affine(w, bits=bits, out=out))
        total, _ = time_graphs([graph], steps, warmup)
        us = 1e3 * total / steps
        byt = N * K * 2 + N * K * bits // 8 + N * (K // 64) * 4
        gbs = byt / (us * 1e-6) / 1e9
        res[f"u{bits}"] = {"shape": [N, K], "us_per_launch": round(us, 2),
                           "bytes_per_launch": byt, "GB/s": round(gbs, 1),
                           "frac_of_measured_hbm": round(gbs / peak, 4)}
    del w
    return res


# ---------------------------------------------------------------- CPU oracle
def oracle_layer_prep(bits: int, M: int):
    """Host copies of layer 0's four projections (same seeded recipe, drawn
    on the host) and activations, for the CPU oracle."""
    import gwa_synth as synth
    shapes = layer_shapes()
    ws = [synth.qweight(synth.stack_seed(0, p, bits), rows, K, bits)
          for p, (_, rows, K) in enumerate(shapes)]
    xs = {K: synth.activations(777 + K, M, K) for _, _, K in shapes}
    return shapes, ws, xs


def oracle_layer_pass(prep, bits: int, nthreads: int = 0):
    import oracle
    shapes, ws, xs = prep
    for (name, rows, K), w in zip(shapes, ws):
        if name == "gate_up":
            oracle.gate_up_silu(xs[K], w.wq, w.scales, w.biases, rows, K, bits,
                                nthreads=nthreads)
        else:
            oracle.qmv(xs[K], w.wq, w.scales, w.biases, rows, K, bits,
                       nthreads=nthreads)


def oracle_layer_sample(bits: int, M: int, seconds: float, max_reps: int,
                        prep=None, nthreads: int = 0):
    """Times the oracle on layer 0's four projections, repeated until
    `seconds` have passed or `max_reps` passes ran (`nthreads` 0: all of
    the oracle's OpenMP threads)."""
    import oracle
    oracle.build()
    prep = prep or oracle_layer_prep(bits, M)
    nthreads = nthreads or oracle.max_threads()
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle_layer_pass(prep, bits, nthreads)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds or reps >= max_reps:
            break
    return reps, el, nthreads


def cpu_baseline(args):
    prep = oracle_layer_prep(args.bits, args.tokens)
    reps, el, nthreads = oracle_layer_sample(args.bits, args.tokens, 10.0, 48,
                                             prep)
    reps1, el1, _ = oracle_layer_sample(args.bits, args.tokens, 4.0, 16, prep,
                                        nthreads=1)
    lb = sum(layer_bytes(args.bits, args.tokens).values())
    return {"value": round(reps * lb / el / 1e9, 4), "unit": "GB/s",
            "cores": nthreads, "kind": "oracle",
            "steps_per_s": round(reps / el / args.layers, 6),
            "one_thread": {"value": round(reps1 * lb / el1 / 1e9, 4),
                           "unit": "GB/s", "cores": 1,
                           "sample": f"{reps1} pass(es), {el1:.1f} s"},
            "sample": (f"{reps} pass(es) of layer 0's four projections "
                       f"(fp64 C oracle, {nthreads} OpenMP threads), "
                       f"{el:.1f} s; GB/s of the same algorithmic bytes; "
                       f"one_thread: the same on one thread")}


def run_reference(args, rank: int):
    if rank != 0:
        return
    import oracle
    oracle.build()
    lb = sum(layer_bytes(args.bits, args.tokens).values())
    prep = oracle_layer_prep(args.bits, args.tokens)
    for _ in range(args.warmup):
        oracle_layer_pass(prep, args.bits)
    reps, el, nthreads = oracle_layer_sample(args.bits, args.tokens,
                                             math.inf, args.steps, prep)
    gbs = reps * lb / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4),
        "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1e3 * el / reps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "config": workload_config(args),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s",
                         "cores": nthreads, "kind": "oracle",
                         "sample": "each step: layer 0's four projections, "
                                   "fp64 C oracle (same seeded recipe)"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "steps_per_s": round(reps / el / args.layers, 6),
    }
    print(json.dumps(line), flush=True)


def max_over_ranks(ms: float, device) -> float:
    """The slowest rank's time: every rank passes its own measurement and
    all get the maximum (the whole job is done when the last rank is)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, bytes_per_rank: float, ms: float) -> float:
    """Aggregate GB/s of `world` replicas that each move `bytes_per_rank`
    in `ms` (the max over ranks)."""
    return world * bytes_per_rank / (ms * 1e-3) / 1e9


METRIC = ("quantized GEMV achieved HBM GB/s (% of GB300 peak); "
          "48-layer decode steps/s")


def main():
    args = parse()
    if args.only_extra:
        import torch
        dev = torch.device("cuda")
        fn = {"attention": run_attention_extra, "quantize": run_quantize_extra,
              "moe": run_moe_extra, "formats": run_formats_extra}[args.only_extra]
        kw = {}
        if args.only_extra == "attention" and args.lengths:
            kw["lengths"] = tuple(int(v) for v in args.lengths.split(","))
        print(json.dumps({args.only_extra: fn(dev, args.steps, args.warmup, **kw)}))
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if args.impl == "gwa" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        dist.init_process_group(backend)
    if args.impl == "reference":
        run_reference(args, rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    r = run_gwa(args, rank, world, local_rank)
    import torch
    total_ms, e2e_ms = r["total_ms"], r["e2e_ms"]
    if world > 1:
        total_ms = max_over_ranks(total_ms, "cuda")
        e2e_ms = max_over_ranks(e2e_ms, "cuda")
        r["eager_ms"] = max_over_ranks(r["eager_ms"], "cuda")
    K, L, M, bits = args.steps, args.layers, args.tokens, args.bits
    lb = layer_bytes(bits, M)
    step_bytes = sum(lb.values()) * L
    ms_step = total_ms / K
    gbs = whole_job_gbs(world, step_bytes, ms_step)
    peak, peak_kind = measured_peak()
    kernels = {}
    for kind, ms in r["per_kind_ms"].items():
        per_launch_us = 1e3 * ms / L
        a = lb[kind] / (per_launch_us * 1e-6) / 1e9
        kernels[kind] = {"us_per_launch": round(per_launch_us, 3),
                         "bytes_per_launch": lb[kind],
                         "GB/s": round(a, 1),
                         "frac_of_measured": round(a / peak, 4)}
    dom = max(r["per_kind_ms"], key=lambda k: r["per_kind_ms"][k])
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(gbs, 1), "unit": "GB/s",
        "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": workload_config(args),
        "steps_per_s": round(world * 1e3 / ms_step, 2),
        "pct_of_8tbs": round(100 * gbs / world / NOMINAL_HBM_GBS, 2),
        "pct_of_measured_hbm": round(100 * gbs / world / peak, 2),
        "roofline": {"bound": "hbm", "kernel": dom,
                     "achieved": kernels[dom]["GB/s"], "peak": peak,
                     "unit": "GB/s",
                     "frac": round(kernels[dom]["GB/s"] / peak, 4),
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "traffic": recorded_traffic(dom),
                     "traffic_source": "dram__bytes_read.sum + "
                     "dram__bytes_write.sum per launch from the ncu capture "
                     "recorded in profiles/qmv_group_gate_up_27648x5120_m1.md "
                     "(not measured by this run); null when absent or when "
                     "the kernel's sources changed since the capture",
                     "algorithmic_bytes": lb[dom]},
        "kernels": kernels,
        "kernels_timing": "per projection type: one graph of its 48 launches "
                          "replayed with CUDA events around it (a second timed "
                          "region; the step itself is timed in layer order)",
        "e2e": {"value": round(whole_job_gbs(world, step_bytes, e2e_ms), 1),
                "unit": "GB/s", "h2d_bytes_per_step": r["h2d"],
                "d2h_bytes_per_step": r["d2h"],
                "ms_per_step": round(e2e_ms, 4),
                "how": "pinned x in, one graph replay of the 192 public API "
                       "calls, last layer's y out, per step",
                "eager": {"value": round(whole_job_gbs(world, step_bytes,
                                                       r["eager_ms"]), 1),
                          "unit": "GB/s",
                          "ms_per_step": round(r["eager_ms"], 4),
                          "wall_ms_per_step": round(r["eager_wall_ms"], 4),
                          "how": "the same copies with the 192 calls issued "
                                 "from Python through the ctypes binding "
                                 "every step (no graph), so the host-side "
                                 "cost of the binding and the C ABI counts"}},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }
    if r["extras"]:
        ex = dict(r["extras"])
        for key in ("prefill_stack_M512", "prefill_stack_u8_M512"):
            pf = ex.get(key)
            if pf:
                bf = _measured_tflops()
                pf["peak_TFLOP/s"] = bf[0]
                pf["frac_of_peak"] = round(pf["TFLOP/s"] / bf[0], 4)
                pf["peak_source"] = bf[1]
        line["extras"] = ex
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(args)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
