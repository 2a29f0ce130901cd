"""Benchmark of the tree-verify hot path on one GB300 (or N replicas under torchrun).

One step = tree_build + tree_attention + tree_accept over one batch of a synthetic
Llama-shaped workload (inputs resident in HBM).  Prints ONE JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Metric: effective HBM TB/s of the step = algorithmic bytes (each input byte read once, each
output byte written once) / step time; also tree nodes verified per second.  The L2 cache
(129 MB) is flushed by writing a 512 MB buffer before every timed step, outside the timed
events.  ``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same
workload (the slow plain reference this project is checked against).
"""
from __future__ import annotations

import os

# numpy's BLAS threads for the CPU oracle leg: every host core, set before numpy loads
_CORES = os.cpu_count() or 1
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CORES))

import argparse
import hashlib
import json
import math
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np
import torch

import workloads

DEFAULT_WORKLOAD = "llama2_7b"
METRIC = "tree-verify effective HBM TB/s (% of GB300 peak) and tree nodes verified/s"
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--prefix", type=int, default=None,
                    help="override the workload's prefix length (a smaller case for detailed profiling; "
                         "the JSON line then names the modified workload)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="launch through the API each step instead of "
                    "replaying CUDA graphs of the three operations")
    return ap.parse_args()


# ------------------------------------------------------------------------------------
# algorithmic bytes
# ------------------------------------------------------------------------------------
def algo_bytes(w, prefix_len):
    s = 4 if w.dtype == "f32" else 2
    W = (w.m + 63) // 64
    B, m = w.B, w.m
    build = B * w.rows * w.V * 4 + B * 4 + B * m * (4 * 3 + 8 * W + 8)
    kv = sum((int(L) + m) * w.Hkv * w.d * s * 2 for L in prefix_len)
    blocks = sum(math.ceil((int(L) + m) / workloads.BLOCK_SIZE) for L in prefix_len) * 4
    attn = 2 * B * m * w.Hq * w.d * s + kv + B * m * W * 8 + blocks + B * 4 + B * m * w.Hq * 4
    accept = B * m * w.V * s + B * m * 4 * 2 + B * m * 4 * 2 + B * 4 * 2
    return dict(tree_build=build, tree_attention=attn, tree_accept=accept, step=build + attn + accept)


def attention_flops(w, prefix_len):
    return 4 * w.d * w.Hq * w.m * sum(int(L) for L in prefix_len)


# ------------------------------------------------------------------------------------
# peaks, clocks, traffic
# ------------------------------------------------------------------------------------
def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense bf16 tensor peak in TFLOP/s (the burst figure: the attention call is timed alone
    inside a short step)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def attention_roofline(attn_bytes, attn_flops, attn_ms, hbm, tensor, traffic):
    """The attention call against its binding roof: the HBM copy bandwidth (algorithmic bytes /
    time), or the tensor pipe (FLOPs / time) where its FLOPs take longer at the bf16 peak than
    its bytes at the HBM peak (FLOPs per K/V byte, about m*g, past the ridge).  `hbm` and
    `tensor` are (peak, kind) pairs in GB/s and TFLOP/s."""
    (hbm_gbs, hbm_kind), (tf, tf_kind) = hbm, tensor
    kernel = "tree_attention (tcgen05 kernel + split-K combine)"
    if attn_flops / (tf * 1e12) > attn_bytes / (hbm_gbs * 1e9):
        achieved = attn_flops / (attn_ms * 1e-3) / 1e12
        return {"bound": "tensor", "kernel": kernel, "achieved": round(achieved, 1), "peak": tf,
                "peak_kind": tf_kind, "unit": "TFLOP/s", "frac": round(achieved / tf, 4), "traffic": traffic}
    achieved = attn_bytes / (attn_ms * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": kernel, "achieved": round(achieved, 1), "peak": hbm_gbs, "peak_kind": hbm_kind,
            "unit": "GB/s", "frac": round(achieved / hbm_gbs, 4), "traffic": traffic}


def kernel_source_hash():
    """Hash of the sources the attention kernels are built from (the roofline kernel)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_tree_eagle_gb300", "csrc")
    for f in ("common.cuh", "tree_attention_tc.cu"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload):
    """DRAM bytes per launch of the attention kernel from a committed ncu summary, or None
    if there is none for this workload or the kernels changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d[workload]
        if e.get("source_hash") != kernel_source_hash():
            return None
        return e["tree_attention_dram_bytes_per_launch"]
    except Exception:
        return None


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------
class Step:
    """Device buffers + outputs for one verify step of workload w (no allocation per step)."""

    def __init__(self, w, inp, dev):
        import speculative_decoding_tree_eagle_gb300 as ts
        self.ts, self.w, self.dev = ts, w, dev
        self.host = inp
        self.d = {k: v.to(dev) for k, v in inp.items() if torch.is_tensor(v) and v.dim() > 0}
        B, m, W = w.B, w.m, (w.m + 63) // 64
        self.tree = dict(tokens=torch.empty(B, m, dtype=torch.int32, device=dev),
                         parents=torch.empty(B, m, dtype=torch.int32, device=dev),
                         depth=torch.empty(B, m, dtype=torch.int32, device=dev),
                         mask=torch.empty(B, m, W, dtype=torch.int64, device=dev),
                         values=torch.empty(B, m, dtype=torch.float64, device=dev),
                         node_row=torch.empty(B, m, dtype=torch.int32, device=dev))
        self.out = torch.empty_like(self.d["q"])
        self.lse = torch.empty(B, m, w.Hq, dtype=torch.float32, device=dev)
        self.acc = dict(argmax=torch.empty(B, m, dtype=torch.int32, device=dev),
                        accept_len=torch.empty(B, dtype=torch.int32, device=dev),
                        accept_path=torch.empty(B, m, dtype=torch.int32, device=dev),
                        bonus=torch.empty(B, dtype=torch.int32, device=dev))
        dt = self.d["q"].dtype
        self.ws = [torch.empty(max(n, 256), dtype=torch.uint8, device=dev) for n in (
            ts.tree_build_workspace(B, w.V, w.k, w.depth, m),
            ts.tree_attention_workspace(dt, B, m, w.Hq, w.Hkv, w.d, w.max_prefix),
            ts.tree_accept_workspace(dt, B, m, w.V))]
        self.status = ts.new_status(dev)

    def build(self):
        self.ts.tree_build(self.d["draft_logp"], self.d["root_tokens"], self.w.k, self.w.depth, self.w.m,
                           out=self.tree, workspace=self.ws[0], status=self.status)

    def attention(self):
        d = self.d
        self.ts.tree_attention(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["prefix_len"],
                               self.tree["mask"], max_prefix=self.w.max_prefix, out=self.out, lse=self.lse,
                               workspace=self.ws[1], status=self.status)

    def accept(self):
        self.ts.tree_accept(self.d["logits"], self.tree["tokens"], self.tree["parents"], out=self.acc,
                            workspace=self.ws[2], status=self.status)

    def run(self):
        self.build()
        self.attention()
        self.accept()


def get_workload(args):
    w = workloads.WORKLOADS[args.workload]
    if args.prefix is not None:
        import dataclasses
        w = dataclasses.replace(w, name=f"{w.name}_prefix{args.prefix}", prefix=(args.prefix, args.prefix))
    return w


def run_ours(args, rank, world, dev):
    import speculative_decoding_tree_eagle_gb300 as ts
    from speculative_decoding_tree_eagle_gb300 import build as tsbuild
    tsbuild.build()
    ts.library()
    w = get_workload(args)
    inp = workloads.generate(w)
    step = Step(w, inp, dev)
    if w.plant_frac > 0:
        # the planting recipe needs the draft tree: take it from this library's own tree_build
        step.build()
        torch.cuda.synchronize()
        inp["logits"] = workloads.plant_paths(w, inp["logits"], step.tree["tokens"].cpu(),
                                              step.tree["parents"].cpu())
        step.d["logits"].copy_(inp["logits"])
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        flush.zero_()
        step.run()
    torch.cuda.synchronize()
    ts.check_status(step.status)
    ops = [step.build, step.attention, step.accept]
    per_step_launches = None
    step_op = step.run
    if not args.no_graph:
        # one CUDA graph for the whole step (the timed number: the kernels of the three
        # operations follow each other with programmatic dependent launch, as a caller's stream
        # would run them), and one graph per operation for the per-operation breakdown; both keep
        # host-side launch overhead (Python binding, argument checks) out of the device timeline
        n0 = ts.launch_count()
        g_step = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_step):
            step.run()
        per_step_launches = ts.launch_count() - n0
        graphs = []
        for op in ops:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                op()
            graphs.append(g)
        ops = [g.replay for g in graphs]
        step_op = g_step.replay
        for _ in range(2):
            step_op()
            for op in ops:
                op()
        torch.cuda.synchronize()

    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    t_wall0 = time.time()
    # timed region: K whole steps, L2 flushed before each
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    n0 = ts.launch_count()
    for i in range(args.steps):
        flush.zero_()
        evs[i][0].record(stream)
        step_op()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    launches = ts.launch_count() - n0 if per_step_launches is None else per_step_launches * args.steps
    barrier(world)
    # per-operation breakdown: the same K steps again, events between the operations.  With
    # graphs, the events are recorded inside one graph of the three operations (event-record
    # nodes between their kernels), so each time is that operation's own kernels and not the
    # device-side launch of a separate graph; without them (or without graph events in torch),
    # events go between the launches.
    op_times = []
    in_graph = False
    if not args.no_graph:
        try:
            ge = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
            g_ops = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_ops):
                ge[0].record()
                step.build()
                ge[1].record()
                step.attention()
                ge[2].record()
                step.accept()
                ge[3].record()
            for _ in range(2):
                g_ops.replay()
            torch.cuda.synchronize()
            for i in range(args.steps):
                flush.zero_()
                g_ops.replay()
                torch.cuda.synchronize()
                op_times.append([ge[j].elapsed_time(ge[j + 1]) for j in range(3)])
            in_graph = True
        except (TypeError, RuntimeError):
            op_times = []
    if not in_graph:
        pevs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush.zero_()
            e = pevs[i]
            e[0].record(stream)
            ops[0]()
            e[1].record(stream)
            ops[1]()
            e[2].record(stream)
            ops[2]()
            e[3].record(stream)
        torch.cuda.synchronize()
        op_times = [[e[j].elapsed_time(e[j + 1]) for j in range(3)] for e in pevs]
    # keep the GPU busy for at least ~1.5 s overall so the clock sampler sees the load
    while time.time() - t_wall0 < 1.5:
        flush.zero_()
        step_op()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ts.check_status(step.status)

    t_step = [e[0].elapsed_time(e[1]) for e in evs]
    t_build = [t[0] for t in op_times]
    t_attn = [t[1] for t in op_times]
    t_acc = [t[2] for t in op_times]
    total_ms = sum(t_step)
    total_ms = allreduce_max(total_ms, world, dev)
    ab = algo_bytes(w, inp["prefix_len"].tolist())
    ms = total_ms / args.steps
    value = world * ab["step"] / (ms * 1e-3) / 1e12
    peak, peak_kind = hbm_peak()
    mean = lambda x: sum(x) / len(x)
    attn_ms = mean(t_attn)
    traffic = ncu_traffic(args.workload)
    roofline = attention_roofline(ab["tree_attention"], attention_flops(w, inp["prefix_len"].tolist()), attn_ms,
                                  (peak, peak_kind), tensor_peak(), traffic)
    res = {
        "metric": METRIC, "value": round(value, 4), "unit": "TB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "ms_per_step_median": round(statistics.median(t_step), 5), "ms_per_step_min": round(min(t_step), 5),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.B, "q_heads": w.Hq, "kv_heads": w.Hkv, "head_dim": w.d,
                   "prefix": list(w.prefix), "tree_nodes": w.m, "top_k": w.k, "depth": w.depth, "vocab": w.V,
                   "block_size": workloads.BLOCK_SIZE, "l2": "flushed (512 MB write) before every timed step",
                   "launch": "API calls" if args.no_graph else
                             ("one CUDA graph per step (per-operation times: events recorded inside one graph "
                              "of the three operations)" if in_graph else
                              "one CUDA graph per step (per-operation times: one graph per operation)"),
                   "parallelism": f"replicas{world}"},
        "pct_of_hbm_peak": round(100 * value * 1e3 / peak, 2),
        "nodes_verified_per_s": round(world * w.B * w.m / (ms * 1e-3), 1),
        "nodes_verified_per_s_attention_accept": round(world * w.B * w.m / ((attn_ms + mean(t_acc)) * 1e-3), 1),
        "kernels_ms": {"tree_build": round(mean(t_build), 5), "tree_attention": round(attn_ms, 5),
                       "tree_accept": round(mean(t_acc), 5)},
        "kernels_tbs": {k: round(ab[k] / (mean(t) * 1e-3) / 1e12, 4) for k, t in
                        (("tree_build", t_build), ("tree_attention", t_attn), ("tree_accept", t_acc))},
        "algorithmic_bytes": ab,
        "attention_tflops": round(attention_flops(w, inp["prefix_len"].tolist()) / (attn_ms * 1e-3) / 1e12, 2),
        "attention_plan": ts.tree_attention_plan(step.d["q"].dtype, w.B, w.m, w.Hq, w.Hkv, w.d, w.max_prefix,
                                                 workloads.BLOCK_SIZE),
        "clocks": clocks,
        "gpu_launches": int(launches),
        "roofline": roofline,
    }
    res["next_rows"] = {"kv_commit": run_kv_commit(step, w, args, flush, stream, world),
                        "lm_head_argmax": run_lm_head(w, args, flush, stream, dev),
                        "efficient_head": run_efficient_head(w, args, flush, stream, dev),
                        "accept_sample": run_accept_sample(step, w, args, flush, stream, world),
                        "tree_prune": run_tree_prune(step, w, args, flush, stream)}
    if not args.no_e2e:
        res["e2e"] = run_e2e(step, w, ab, args, dev, world)
    return res, w, inp


# hidden size of the target model each workload is shaped after (the LM head is [V, d_model])
D_MODEL = {"llama2_7b": 4096, "llama3_8b_gqa": 4096, "llama2_70b_gqa": 8192}


def run_lm_head(w, args, flush, stream, dev):
    """The target LM head with the per-row argmax fused into its GEMM (the row after the hot
    path): hidden [B*m, d_model] x weight [V, d_model]^T, seeded Gaussian bf16 weights, K calls,
    L2 flushed before each."""
    import speculative_decoding_tree_eagle_gb300 as ts
    K = D_MODEL.get(w.name.split("_prefix")[0], 4096)
    M, V = w.B * w.m, w.V
    g = torch.Generator(device=dev).manual_seed(20260 + 99)
    hidden = torch.randn(M, K, generator=g, device=dev).to(torch.bfloat16)
    weight = (torch.randn(V, K, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    out = dict(argmax=torch.empty(M, dtype=torch.int32, device=dev),
               max_logit=torch.empty(M, dtype=torch.float32, device=dev))
    ws = torch.empty(max(256, ts.library().ts_lm_head_argmax_workspace(M, V, K)), dtype=torch.uint8, device=dev)
    status = ts.new_status(dev)
    times = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        ts.lm_head_argmax(hidden, weight, out=out, workspace=ws, status=status)
        b.record(stream)
        if i >= args.warmup:
            times.append((a, b))
    torch.cuda.synchronize()
    ts.check_status(status)
    ms = sum(a.elapsed_time(b) for a, b in times) / len(times)
    byts = (V * K + M * K) * 2 + M * 8
    flops = 2.0 * M * V * K
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except Exception:
        pass
    hbm = peaks.get("hbm_gbs", 6800.0)
    tf = peaks.get("bf16_tflops", 1900.0)
    tb_s = byts / (ms * 1e-3) / 1e12
    tflops = flops / (ms * 1e-3) / 1e12
    t_hbm, t_tc = byts / (hbm * 1e9), flops / (tf * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    frac = (tb_s * 1e3 / hbm) if bound == "hbm" else (tflops / tf)
    res = {"ms": round(ms, 5), "shape": {"rows": M, "vocab": V, "d_model": K}, "algorithmic_bytes": int(byts),
           "tb_s": round(tb_s, 4), "tflops": round(tflops, 2), "bound": bound, "frac_of_measured_peak": round(frac, 4),
           "logits_bytes_not_written": int(M * V * 4)}
    if not args.no_cpu_baseline and _WORLD == 1:
        # the oracle beside it: fp64 logits and argmax of a bounded sample of rows, scaled to all rows
        import oracle
        n = min(M, 8)
        hh, wh = hidden[:n].cpu(), weight.cpu()
        t0 = time.perf_counter()
        oracle.lm_head_argmax(hh, wh)
        res["oracle_ms"] = round((time.perf_counter() - t0) * 1e3 * M / n, 2)
        res["oracle_note"] = f"fp64 numpy oracle on {n} of {M} rows, scaled to all rows"
    del hidden, weight
    return res


def run_efficient_head(w, args, flush, stream, dev, rank=256, tile_tokens=1024, k_tile=2):
    """One draft step of the two-stage efficient head (the row after the hot path): the B*k
    frontier rows of a drafter with a d_model-wide hidden state, seeded Gaussian bf16 factors;
    rank, tile size and candidates per tile are a reading (the page states none)."""
    import speculative_decoding_tree_eagle_gb300 as ts
    d = D_MODEL.get(w.name.split("_prefix")[0], 4096)
    M, V, k = w.B * w.k, w.V, w.k
    g = torch.Generator(device=dev).manual_seed(20260 + 98)
    h = torch.randn(M, d, generator=g, device=dev).to(torch.bfloat16)
    B = (torch.randn(rank, d, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    A = (torch.randn(V, rank, generator=g, device=dev) * 0.05).to(torch.bfloat16)
    W = (torch.randn(V, d, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    L = ts.library()
    ws = torch.empty(max(256, L.ts_efficient_head_workspace(M, V, d, rank, tile_tokens, k_tile)), dtype=torch.uint8,
                     device=dev)
    status = ts.new_status(dev)
    times = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        ts.efficient_head(h, B, A, W, tile_tokens=tile_tokens, k_tile=k_tile, k=k, workspace=ws, status=status)
        b.record(stream)
        if i >= args.warmup:
            times.append((a, b))
    torch.cuda.synchronize()
    ts.check_status(status)
    ms = sum(a.elapsed_time(b) for a, b in times) / len(times)
    C = L.ts_efficient_head_candidates(V, tile_tokens, k_tile)
    byts = (V * rank + rank * d + M * d) * 2 + M * C * d * 2 + M * k * 8
    full_head = V * d * 2
    res = {"ms": round(ms, 5), "shape": {"rows": M, "vocab": V, "d_model": d, "rank": rank, "tile_tokens": tile_tokens,
                                         "k_tile": k_tile, "candidates": C, "k": k},
           "algorithmic_bytes": int(byts), "tb_s": round(byts / (ms * 1e-3) / 1e12, 4),
           "full_head_bytes": int(full_head), "bound": "hbm (low-rank head + gathered candidate rows)"}
    if not args.no_cpu_baseline and _WORLD == 1:
        import oracle
        n = min(M, 2)
        t0 = time.perf_counter()
        oracle.efficient_head(h[:n].cpu(), B.cpu(), A.cpu(), W.cpu(), tile_tokens, k_tile, k)
        res["oracle_ms"] = round((time.perf_counter() - t0) * 1e3 * M / n, 2)
        res["oracle_note"] = f"fp64 numpy oracle on {n} of {M} rows, scaled to all rows"
    del h, B, A, W
    return res


def run_accept_sample(step, w, args, flush, stream, world, temperature=1.0):
    """Verification at T > 0 by multi-round rejection sampling (the row after greedy
    acceptance), both proposal modes, on the step's own tree.  Target logits: the step's
    N(0,1) logits with one child of every expanded node raised to ln(V) + U(0, 4) (kept with
    probability ~0.4..1 per level), so that walks go several levels deep as in the pages'
    reported acceptance lengths; seeded uniforms.  L2 flushed before each call."""
    ts = step.ts
    d = step.d
    B, m, V = w.B, w.m, w.V
    tok, par, nrow = step.tree["tokens"], step.tree["parents"], step.tree["node_row"]
    par_h, tok_h = par.cpu().numpy(), tok.cpu().numpy()
    rng = np.random.default_rng(w.seed + 11)
    bi, ui, ti, vals = [], [], [], []
    for b in range(B):
        for u in range(m):
            kids = np.nonzero(par_h[b] == u)[0]
            if len(kids):
                bi.append(b), ui.append(u), ti.append(int(tok_h[b, kids[rng.integers(len(kids))]]))
                vals.append(math.log(V) + rng.uniform(0.0, 4.0))
    logits = d["logits"].clone()
    dev = logits.device
    idx = tuple(torch.tensor(x, dtype=torch.long, device=dev) for x in (bi, ui, ti))
    logits.index_put_(idx, torch.tensor(vals, dtype=torch.float32, device=dev).to(logits.dtype))
    g = torch.Generator(device=dev).manual_seed(w.seed + 12)
    uniforms = torch.rand(B, m, generator=g, device=dev)
    out = dict(accept_len=torch.empty(B, dtype=torch.int32, device=dev),
               accept_path=torch.empty(B, m, dtype=torch.int32, device=dev),
               bonus=torch.empty(B, dtype=torch.int32, device=dev))
    L = ts.library()
    ws = torch.empty(max(256, L.ts_tree_accept_sample_workspace(B, V, 1)), dtype=torch.uint8, device=dev)
    elt = logits.element_size()
    res = {"temperature": temperature, "input": "step logits, one child per expanded node raised to ln(V)+U(0,4)"}
    for mode in ("point", "draft"):
        times = []
        for i in range(args.warmup + args.steps):
            flush.zero_()
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            ts.tree_accept_sample(logits, tok, par, uniforms, temperature, q_mode=mode, draft_logp=d["draft_logp"],
                                  node_row=nrow, out=out, workspace=ws, status=step.status)
            b_.record(stream)
            if i >= args.warmup:
                times.append((a, b_))
        torch.cuda.synchronize()
        ts.check_status(step.status)
        ms = sum(a.elapsed_time(b_) for a, b_ in times) / len(times)
        alen = out["accept_len"].cpu().numpy()
        # one read of every visited node's target row, one more of the last node's (the draw);
        # draft mode also reads the draft row of every visited node that has children
        byts = int(sum(int(a_) + 1 for a_ in alen) * V * elt)
        if mode == "draft":
            path = out["accept_path"].cpu().numpy()
            has = [set(par_h[b][par_h[b] >= 0].tolist()) for b in range(B)]
            byts += int(sum(1 for b in range(B) for j in range(alen[b]) if path[b, j] in has[b]) * V * 4)
        r = {"ms": round(ms, 5), "mean_accept_len": round(float(alen.mean()), 3),
             "bytes_min": byts, "gb_s": round(byts / (ms * 1e-3) / 1e9, 1),
             "bound": "latency (one CTA per sequence walks the tree; a few row passes per level)"}
        if not args.no_cpu_baseline and world == 1:
            import oracle
            lh = logits.float().cpu().numpy()
            dh = d["draft_logp"].cpu().numpy() if mode == "draft" else None
            t0 = time.perf_counter()
            ref = oracle.accept_sample(lh, tok_h, par_h, uniforms.cpu().numpy(), temperature, mode, dh,
                                       nrow.cpu().numpy())
            r["oracle_ms"] = round((time.perf_counter() - t0) * 1e3, 2)
            r["oracle_same_len"] = float((ref[0] == alen).mean())
        res[mode] = r
    del logits
    return res


def run_tree_prune(step, w, args, flush, stream, costs=(1.0, 10.0, 0.05)):
    """Cost-aware pruning of the step's tree before verification (the harness row): three
    launches, no host sync inside the events; the cost model (t_draft, t_fixed, t_node) is an
    illustrative one in arbitrary units."""
    ts = step.ts
    tree = {k: step.tree[k] for k in ("tokens", "parents", "depth", "values", "node_row")}
    B, m = w.B, w.m
    dev = tree["tokens"].device
    ws = torch.empty(max(256, ts.library().ts_tree_prune_workspace(B, m)), dtype=torch.uint8, device=dev)
    times = []
    for i in range(args.warmup + args.steps):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        out = ts.tree_prune(tree, *costs, workspace=ws, status=step.status, sync=False)
        b.record(stream)
        if i >= args.warmup:
            times.append((a, b))
    torch.cuda.synchronize()
    ts.check_status(step.status)
    ms = sum(a.elapsed_time(b) for a, b in times) / len(times)
    n = int(out["n"].item())
    W = (n + 63) // 64
    byts = B * m * (4 * 4 + 8) + B * n * (4 * 5 + 8 + 8 * W) + B * 4
    res = {"ms": round(ms, 5), "costs": list(costs), "n": n, "algorithmic_bytes": int(byts),
           "bound": "latency (three small launches)"}
    if not args.no_cpu_baseline and _WORLD == 1:
        import oracle
        hh = {k: v.cpu().numpy() for k, v in tree.items()}
        t0 = time.perf_counter()
        oracle.tree_prune(hh["tokens"], hh["parents"], hh["depth"], hh["values"], *costs, node_row=hh["node_row"])
        res["oracle_ms"] = round((time.perf_counter() - t0) * 1e3, 2)
    return res


def run_kv_commit(step, w, args, flush, stream, world):
    """The KV commit of the step's accepted paths (the row after the hot path): K calls on
    the step's own accept outputs, block table and prefix lengths restored before each call
    (outside the events), L2 flushed."""
    ts = step.ts
    d = step.d
    table0 = d["block_table"].clone()
    plen0 = d["prefix_len"].clone()
    out = dict(freed_blocks=torch.empty_like(table0), freed_count=torch.empty_like(plen0))
    alen = step.acc["accept_len"].clone()
    apath = step.acc["accept_path"].clone()
    times = []
    for i in range(args.warmup + args.steps):
        d["block_table"].copy_(table0)
        d["prefix_len"].copy_(plen0)
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        ts.kv_commit(d["k_cache"], d["v_cache"], d["block_table"], d["prefix_len"], apath, alen, out=out,
                     status=step.status)
        b.record(stream)
        if i >= args.warmup:
            times.append((a, b))
    torch.cuda.synchronize()
    ts.check_status(step.status)
    d["block_table"].copy_(table0)
    d["prefix_len"].copy_(plen0)
    ms = sum(a.elapsed_time(b) for a, b in times) / len(times)
    al = alen.cpu().tolist()
    pl = apath.cpu().tolist()
    moved = sum(sum(1 for j in range(n) if pl[bb][j] != j) for bb, n in enumerate(al))
    row = w.Hkv * w.d * (2 if w.dtype == "bf16" else 4)
    max_blocks = int(table0.shape[1])
    byts = moved * row * 2 * 2 + w.B * (max_blocks * 4 * 3 + w.m * 4 + 12)
    res = {"ms": round(ms, 5), "accepted_rows": int(sum(al)), "moved_rows": int(moved),
           "algorithmic_bytes": int(byts), "bound": "latency (a few rows per sequence; one CTA each)"}
    cache_bytes = d["k_cache"].numel() * d["k_cache"].element_size() * 2
    if not args.no_cpu_baseline and world == 1 and cache_bytes <= (256 << 20):
        # the oracle beside it (cpu-baseline leg): same caches, table, lengths and paths
        import oracle
        view = (lambda t: t.cpu().view(torch.int16).numpy()) if w.dtype == "bf16" else (lambda t: t.cpu().numpy())
        kh, vh = view(d["k_cache"]), view(d["v_cache"])
        th, lh, ph, ah = table0.cpu().numpy(), plen0.cpu().numpy(), apath.cpu().numpy(), alen.cpu().numpy()
        t0 = time.perf_counter()
        reps = 0
        while reps < 3 or time.perf_counter() - t0 < 1.0:
            oracle.kv_commit(kh, vh, th, lh, ph, ah, w.m, workloads.BLOCK_SIZE)
            reps += 1
        res["oracle_ms"] = round((time.perf_counter() - t0) / reps * 1e3, 3)
        res["oracle_note"] = "fp64 numpy oracle on the host (copies the whole cache per call), same inputs"
    return res


def run_e2e(step, w, ab, args, dev, world):
    """Same metric through the public API with host buffers: every step copies its inputs
    from pinned host memory and reads the tree + acceptance result back."""
    names = ["draft_logp", "root_tokens", "q", "k_cache", "v_cache", "block_table", "prefix_len", "logits"]
    host = {n: step.host[n].pin_memory() for n in names}
    outs = {"tokens": step.tree["tokens"], "parents": step.tree["parents"], "accept_len": step.acc["accept_len"],
            "accept_path": step.acc["accept_path"], "bonus": step.acc["bonus"]}
    host_out = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in outs.items()}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in outs.values())
    stream = torch.cuda.current_stream()
    times = []
    for i in range(args.warmup + args.steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for n in names:
            step.d[n].copy_(host[n], non_blocking=True)
        step.run()
        for n, t in outs.items():
            host_out[n].copy_(t, non_blocking=True)
        b.record(stream)
        b.synchronize()
        if i >= args.warmup:
            times.append(a.elapsed_time(b))
    total = allreduce_max(sum(times), world, dev)
    ms = total / args.steps
    return {"value": round(world * ab["step"] / (ms * 1e-3) / 1e12, 4), "unit": "TB/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


# ------------------------------------------------------------------------------------
# CPU oracle (reported baseline / reference arm)
# ------------------------------------------------------------------------------------
def oracle_sample_step(w, inp, heads):
    """One bounded sample of the step on the fp64 oracle: the whole tree_build and
    tree_accept, and tree_attention for ``heads`` query heads of every sequence."""
    import oracle
    tr = oracle.tree_build(inp["draft_logp"].numpy(), inp["root_tokens"].numpy(), w.k, w.depth, w.m)
    sel = [(b, i, h) for b in range(w.B) for i in range(w.m) for h in heads]
    oracle.tree_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"].numpy(),
                          inp["prefix_len"].numpy(), tr["mask"], 1.0 / math.sqrt(w.d), select=sel)
    amax = oracle.target_argmax(inp["logits"])
    oracle.accept_longest_path(tr["tokens"], tr["parents"], amax)


def oracle_sample_bytes(w, ab, heads):
    frac = len(heads) / w.Hq
    return ab["tree_build"] + ab["tree_attention"] * frac + ab["tree_accept"]


def pick_heads(w):
    g = w.Hq // w.Hkv
    n = max(1, min(w.Hq, 4))
    return [h * g % w.Hq for h in range(n)] if g > 1 else list(range(n))


def cpu_baseline(w, inp, budget_s=12.0):
    ab = algo_bytes(w, inp["prefix_len"].tolist())
    heads = pick_heads(w)
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle_sample_step(w, inp, heads)
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = (time.perf_counter() - t0) / n
    byts = oracle_sample_bytes(w, ab, heads)
    return {"value": round(byts / dt / 1e12, 8), "unit": "TB/s", "cores": _CORES, "kind": "oracle",
            "sample": f"fp64 numpy oracle: full tree_build + tree_accept, tree_attention for {len(heads)} of "
                      f"{w.Hq} query heads (all sequences and nodes); {n} repetitions, {dt:.3f} s each; "
                      f"metric scaled by the sample's algorithmic bytes; numpy's BLAS may use all {_CORES} "
                      f"threads (the attention products), the tree passes run single-threaded"}


def run_reference(args, rank, world):
    w = get_workload(args)
    inp = workloads.generate(w)
    ab = algo_bytes(w, inp["prefix_len"].tolist())
    heads = pick_heads(w)
    for _ in range(args.warmup):
        oracle_sample_step(w, inp, heads)
    ts_ = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_sample_step(w, inp, heads)
        ts_.append(time.perf_counter() - t0)
    ms = 1e3 * sum(ts_) / len(ts_)
    byts = oracle_sample_bytes(w, ab, heads)
    value = byts / (ms * 1e-3) / 1e12
    sample = (f"fp64 numpy oracle: full tree_build + tree_accept, tree_attention for {len(heads)} of {w.Hq} "
              f"query heads; metric scaled by the sample's algorithmic bytes; numpy's BLAS may use all "
              f"{_CORES} threads (the attention products), the tree passes run single-threaded")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 8), "unit": "TB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.B, "q_heads": w.Hq, "kv_heads": w.Hkv, "head_dim": w.d,
                       "prefix": list(w.prefix), "tree_nodes": w.m, "vocab": w.V},
            "cpu_baseline": {"value": round(value, 8), "unit": "TB/s", "cores": _CORES, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 8), "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------------------------
# distributed plumbing (replicas only: no data-path collective)
# ------------------------------------------------------------------------------------
_PG = None
_WORLD = 1


def init_dist(args):
    global _PG
    global _WORLD
    world = int(os.environ.get("WORLD_SIZE", "1"))
    _WORLD = world
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        _PG = dist
    return rank, world, local


def barrier(world):
    if world > 1 and _PG is not None:
        _PG.barrier()


def allreduce_max(x, world, dev):
    if world <= 1 or _PG is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev if _PG.get_backend() == "nccl" else "cpu")
    _PG.all_reduce(t, op=_PG.ReduceOp.MAX)
    return float(t.item())


def main():
    args = parse()
    if args.impl == "reference":
        # the oracle arm uses no GPU and no collective: rank 0 alone runs it, the other
        # ranks leave at once (no process group is formed)
        rank, world = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    rank, world, local = init_dist(args)
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    res, w, inp = run_ours(args, rank, world, dev)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            res["cpu_baseline"] = cpu_baseline(w, inp)
        print(json.dumps(res), flush=True)
    if world > 1 and _PG is not None:
        _PG.destroy_process_group()


if __name__ == "__main__":
    main()
