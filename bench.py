"""Benchmark of the tree-verify hot path on one GB300 (or N replicas under torchrun).

One step = tree_build + tree_attention + tree_accept over one batch of a synthetic
Llama-shaped workload (inputs resident in HBM).  Prints ONE JSON line (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

The default workload is the long-context sweep: batch 4, 32 query / 8 KV heads, head dim 128,
a 32768-token paged bf16 prefix per sequence, and four draft trees (an 8-node chain and
dynamic trees of 32, 64 and 128 nodes) over a 128256-token vocabulary.  One step of it is
one verify step of each of the four trees; its value is the sweep's algorithmic bytes over
the sum of the four step times.  The line's ``per_config`` object then holds every workload
measured on its own: the four trees of the sweep and the Llama-2-7B, Llama-3-8B and
Llama-2-70B shaped workloads (``--no-per-config`` skips the three model-shaped ones).

Metric: effective HBM TB/s of the step = algorithmic bytes (each input byte read once, each
output byte written once) / step time; also tree nodes verified per second.  The L2 cache
(129 MB) is flushed by writing a 512 MB buffer before every timed graph replay, outside the
timed events.  ``--impl reference`` times the fp64 CPU oracle on a bounded sample of the same
workload (the slow plain reference this project is checked against).
"""
from __future__ import annotations

import os

# numpy's BLAS threads for the CPU oracle leg: every host core unless the caller set a
# count (the single-thread oracle timing runs in a child process with a count of 1)
_CORES = os.cpu_count() or 1
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CORES))
_ORACLE_THREADS = int(os.environ["OPENBLAS_NUM_THREADS"])

import argparse
import dataclasses
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

# the long-context configuration: one batch shape, four tree sizes
SWEEPS = {"long_context_sweep": ("long_context_m8", "long_context_m32", "long_context_m64", "long_context_m128")}
DEFAULT_WORKLOAD = "long_context_sweep"
# measured on their own beside the default workload (the sweep's trees are measured in it)
OTHER_CONFIGS = ("llama2_7b", "llama3_8b_gqa", "llama2_70b_gqa")
METRIC = "tree-verify effective HBM TB/s (% of GB300 peak) and tree nodes verified/s"
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.WORKLOADS) + sorted(SWEEPS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--prefix", type=int, default=None,
                    help="override the workload's prefix length (a smaller case for detailed profiling; "
                         "the JSON line then names the modified workload)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="measure only --workload (no model-shaped configurations beside it)")
    ap.add_argument("--no-next-rows", action="store_true", help="skip the rows after the hot path")
    ap.add_argument("--no-graph", action="store_true", help="launch through the API each step instead of "
                    "replaying CUDA graphs of the three operations")
    ap.add_argument("--oracle-child", default=None, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-budget", type=float, default=None, help=argparse.SUPPRESS)
    return ap.parse_args(argv)


def workload_list(name, prefix=None):
    """The workloads one step of ``name`` runs: one, or the four trees of a sweep."""
    names = SWEEPS.get(name, (name,))
    out = []
    for n in names:
        w = workloads.WORKLOADS[n]
        if prefix is not None:
            w = dataclasses.replace(w, name=f"{w.name}_prefix{prefix}", prefix=(prefix, prefix))
        out.append(w)
    return out


def workload_name(name, prefix=None):
    return name if prefix is None else f"{name}_prefix{prefix}"


def launch_desc(args):
    if args.no_graph:
        return "API calls"
    return ("one CUDA graph per verify step, the three operations' kernels chained by programmatic "
            "dependent launch; per-operation times are marginal: t(build), t(build+attention) - "
            "t(build), t(step) - t(build+attention), each a graph replayed after an L2 flush")


def config_of(name, args, world):
    """The ``config`` object of the JSON line (the same for both arms)."""
    ws = workload_list(name, args.prefix)
    w0 = ws[0]
    one = len(ws) == 1
    pick = (lambda f: f(w0)) if one else (lambda f: [f(w) for w in ws])
    return {"workload": workload_name(name, args.prefix), "batch": w0.B, "q_heads": w0.Hq, "kv_heads": w0.Hkv,
            "head_dim": w0.d, "prefix": list(w0.prefix), "tree_nodes": pick(lambda w: w.m),
            "top_k": pick(lambda w: w.k), "depth": pick(lambda w: w.depth), "vocab": w0.V,
            "block_size": workloads.BLOCK_SIZE, "l2": "flushed (512 MB write) before every timed graph replay",
            "launch": launch_desc(args), "parallelism": f"replicas{world}"}


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


def roof_time_s(attn_bytes, attn_flops, hbm_gbs, tf):
    """Time of the attention call at its binding roof."""
    return max(attn_bytes / (hbm_gbs * 1e9), attn_flops / (tf * 1e12))


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


class Case:
    """One workload resident on the device with the CUDA graphs that time it.

    ``step`` replays the whole verify step; ``build`` and ``build_attn`` the prefixes of it
    that give the marginal per-operation times (they sum to the step); ``attn`` the attention
    call alone (its isolated time, launch latency of a graph included)."""

    def __init__(self, w, args, dev, flush):
        import speculative_decoding_tree_eagle_gb300 as ts
        self.ts, self.w = ts, w
        self.inp = workloads.generate(w)
        self.step = Step(w, self.inp, dev)
        step = self.step
        if w.plant_frac > 0:
            # the planting recipe needs the draft tree: take it from this library's own tree_build
            step.build()
            torch.cuda.synchronize()
            self.inp["logits"] = workloads.plant_paths(w, self.inp["logits"], step.tree["tokens"].cpu(),
                                                       step.tree["parents"].cpu())
            step.d["logits"].copy_(self.inp["logits"])
        for _ in range(args.warmup):
            flush.zero_()
            step.run()
        torch.cuda.synchronize()
        ts.check_status(step.status)
        self.graphs = None
        self.per_step_launches = None
        if not args.no_graph:
            n0 = ts.launch_count()
            g_step = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_step):
                step.run()
            self.per_step_launches = ts.launch_count() - n0
            g_b, g_ba, g_a = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_b):
                step.build()
            with torch.cuda.graph(g_ba):
                step.build()
                step.attention()
            with torch.cuda.graph(g_a):
                step.attention()
            self.graphs = dict(step=g_step, build=g_b, build_attn=g_ba, attn=g_a)
            for _ in range(2):
                for g in self.graphs.values():
                    g.replay()
            torch.cuda.synchronize()
        self.ab = algo_bytes(w, self.inp["prefix_len"].tolist())
        self.flops = attention_flops(w, self.inp["prefix_len"].tolist())
        self.t = None

    def _run(self, what):
        if self.graphs is not None:
            self.graphs[what].replay()
            return
        s = self.step
        if what in ("step", "build", "build_attn"):
            s.build()
        if what in ("step", "build_attn", "attn"):
            s.attention()
        if what == "step":
            s.accept()

    def time_steps(self, K, flush, stream):
        """K timed replays of each graph (step first), L2 flushed before every replay, one
        event pair around each replay on the launching stream."""
        kinds = ("step", "build", "build_attn", "attn")
        evs = {k: [] for k in kinds}
        n_api = 0
        for _ in range(K):
            for k in kinds:
                flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                n0 = self.ts.launch_count()
                a.record(stream)
                self._run(k)
                b.record(stream)
                if k == "step":
                    n_api += self.ts.launch_count() - n0
                evs[k].append((a, b))
        torch.cuda.synchronize()
        self.t = {k: [a.elapsed_time(b) for a, b in v] for k, v in evs.items()}
        # kernels launched by the K timed steps (a graph replay does not pass through the API's
        # launch counter, so it counts the captured step's launches once per replay)
        self.step_launches = self.per_step_launches * K if self.per_step_launches is not None else n_api
        self.ts.check_status(self.step.status)
        return self.t

    def summary(self, hbm, tensor, traffic):
        t = self.t
        mean = lambda x: sum(x) / len(x)
        w, ab = self.w, self.ab
        ms = mean(t["step"])
        t_b = mean(t["build"])
        t_ba = mean(t["build_attn"])
        attn = t_ba - t_b
        acc = ms - t_ba
        peak = hbm[0]
        roof = attention_roofline(ab["tree_attention"], self.flops, attn, hbm, tensor, traffic)
        t_roof = roof_time_s(ab["tree_attention"], self.flops, hbm[0], tensor[0])
        aa_bytes = ab["tree_attention"] + ab["tree_accept"]
        plan = self.ts.tree_attention_plan(self.step.d["q"].dtype, w.B, w.m, w.Hq, w.Hkv, w.d, w.max_prefix,
                                           workloads.BLOCK_SIZE)
        return {
            "ms_per_step": round(ms, 5), "ms_per_step_median": round(statistics.median(t["step"]), 5),
            "ms_per_step_min": round(min(t["step"]), 5),
            "value": round(ab["step"] / (ms * 1e-3) / 1e12, 4), "unit": "TB/s",
            "pct_of_hbm_peak": round(100 * ab["step"] / (ms * 1e-3) / 1e9 / peak, 2),
            "nodes_verified_per_s": round(w.B * w.m / (ms * 1e-3), 1),
            "nodes_verified_per_s_attention_accept": round(w.B * w.m / ((attn + acc) * 1e-3), 1),
            "kernels_ms": {"tree_build": round(t_b, 5), "tree_attention": round(attn, 5),
                           "tree_accept": round(acc, 5)},
            "kernels_tbs": {"tree_build": round(ab["tree_build"] / (t_b * 1e-3) / 1e12, 4),
                            "tree_attention": round(ab["tree_attention"] / (attn * 1e-3) / 1e12, 4),
                            "tree_accept": round(ab["tree_accept"] / (acc * 1e-3) / 1e12, 4)},
            "attention_ms_isolated": round(mean(t["attn"]), 5),
            "attention_accept_pct_of_hbm_peak": round(100 * aa_bytes / ((attn + acc) * 1e-3) / 1e9 / peak, 2),
            "attention_tflops": round(self.flops / (attn * 1e-3) / 1e12, 2),
            "attention_frac_of_binding_roof": round(t_roof / (attn * 1e-3), 4),
            "algorithmic_bytes": ab, "attention_flops": int(self.flops),
            "attention_plan": plan, "roofline": roof,
        }

    def free(self):
        self.graphs = None
        self.step = None


def time_cases(cases, args, flush, stream, world):
    """The timed region: barrier + synchronize on both sides of K replays per case."""
    barrier(world)
    torch.cuda.synchronize()
    for c in cases:
        c.time_steps(args.steps, flush, stream)
    torch.cuda.synchronize()
    barrier(world)


def next_rows_for(case, args, flush, stream, dev, with_oracle):
    step, w = case.step, case.w
    return {"kv_commit": run_kv_commit(step, w, args, flush, stream, with_oracle),
            "lm_head_argmax": run_lm_head(w, args, flush, stream, dev, with_oracle),
            "efficient_head": run_efficient_head(w, args, flush, stream, dev, with_oracle),
            "accept_sample": run_accept_sample(step, w, args, flush, stream, with_oracle),
            "tree_prune": run_tree_prune(step, w, args, flush, stream, with_oracle)}


def run_ours(args, rank, world, dev):
    import speculative_decoding_tree_eagle_gb300 as ts
    from speculative_decoding_tree_eagle_gb300 import build as tsbuild
    tsbuild.build()
    ts.library()
    name = args.workload
    wl = workload_list(name, args.prefix)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    hbm, tensor = hbm_peak(), tensor_peak()
    oracle_here = not args.no_cpu_baseline and world == 1 and rank == 0

    # ---- the headline workload: every tree of it resident, graphs captured, then timed ----
    cases = [Case(w, args, dev, flush) for w in wl]
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    t_wall0 = time.time()
    time_cases(cases, args, flush, stream, world)
    # keep the GPU busy for at least ~1.5 s overall so the clock sampler sees the load
    while time.time() - t_wall0 < 1.5:
        flush.zero_()
        cases[-1]._run("step")
    torch.cuda.synchronize()
    clocks = sampler.stop()

    step_ms = [sum(c.t["step"][i] for c in cases) for i in range(args.steps)]
    total_ms = allreduce_max(sum(step_ms), world, dev)
    ms = total_ms / args.steps
    step_bytes = sum(c.ab["step"] for c in cases)
    nodes = sum(c.w.B * c.w.m for c in cases)
    value = world * step_bytes / (ms * 1e-3) / 1e12
    per_case = {c.w.name: c.summary(hbm, tensor, ncu_traffic(c.w.name)) for c in cases}
    attn_ms = sum(per_case[c.w.name]["kernels_ms"]["tree_attention"] for c in cases)
    acc_ms = sum(per_case[c.w.name]["kernels_ms"]["tree_accept"] for c in cases)
    attn_bytes = sum(c.ab["tree_attention"] for c in cases)
    attn_flops = sum(c.flops for c in cases)
    if len(cases) == 1:
        roofline = dict(per_case[wl[0].name]["roofline"])
    else:
        # the sweep's attention against the HBM roof (the spec unit), with the fraction of
        # the binding roofs beside it (sum over the trees of max(bytes/HBM, FLOPs/tensor) / time)
        traffic = [ncu_traffic(c.w.name) for c in cases]
        achieved = attn_bytes / (attn_ms * 1e-3) / 1e9
        roofline = {"bound": "hbm", "kernel": "tree_attention (tcgen05 kernel + split-K combine), all four trees",
                    "achieved": round(achieved, 1), "peak": hbm[0], "peak_kind": hbm[1], "unit": "GB/s",
                    "frac": round(achieved / hbm[0], 4),
                    "traffic": sum(traffic) if all(x is not None for x in traffic) else None,
                    "frac_of_binding_roofs": round(
                        sum(roof_time_s(c.ab["tree_attention"], c.flops, hbm[0], tensor[0]) for c in cases)
                        / (attn_ms * 1e-3), 4)}
    launches = sum(c.step_launches for c in cases)
    w0 = wl[0]
    res = {
        "metric": METRIC, "value": round(value, 4), "unit": "TB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "ms_per_step_median": round(statistics.median(step_ms), 5), "ms_per_step_min": round(min(step_ms), 5),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w0.dtype == "bf16" else "f32", "data": "synthetic",
        "config": config_of(name, args, world),
        "pct_of_hbm_peak": round(100 * value * 1e3 / hbm[0], 2),
        "nodes_verified_per_s": round(world * nodes / (ms * 1e-3), 1),
        "nodes_verified_per_s_attention_accept": round(world * nodes / ((attn_ms + acc_ms) * 1e-3), 1),
        "attention_accept_pct_of_hbm_peak": round(
            100 * (attn_bytes + sum(c.ab["tree_accept"] for c in cases)) / ((attn_ms + acc_ms) * 1e-3) / 1e9
            / hbm[0], 2),
        "kernels_ms": {k: round(sum(per_case[c.w.name]["kernels_ms"][k] for c in cases), 5)
                       for k in ("tree_build", "tree_attention", "tree_accept")},
        "kernels_ms_method": "marginal (sums to the step): t(build), t(build+attention) - t(build), "
                             "t(step) - t(build+attention), each a CUDA graph replayed after an L2 flush",
        "algorithmic_bytes": {k: sum(c.ab[k] for c in cases) for k in ("tree_build", "tree_attention",
                                                                       "tree_accept", "step")},
        "attention_tflops": round(attn_flops / (attn_ms * 1e-3) / 1e12, 2),
        "clocks": clocks,
        "gpu_launches": int(launches),
        "roofline": roofline,
    }
    if not args.no_e2e:
        res["e2e"] = run_e2e(cases, args, dev, world)
    if oracle_here:
        res["cpu_baseline"] = cpu_baseline(wl, [c.inp for c in cases], budget_s=12.0, single_thread_of=name,
                                           args=args)
    per_config = {}
    for c in cases:
        e = per_case[c.w.name]
        if oracle_here:
            e["cpu_baseline"] = cpu_baseline([c.w], [c.inp], budget_s=2.0)
        per_config[c.w.name] = e
    if len(cases) == 1 and not args.no_next_rows:
        res["next_rows"] = next_rows_for(cases[0], args, flush, stream, dev, oracle_here)
    for c in cases:
        c.free()
    del cases
    torch.cuda.empty_cache()

    # ---- the other configurations, one at a time ----
    if not args.no_per_config and name in SWEEPS:
        for cname in OTHER_CONFIGS:
            w = workload_list(cname, args.prefix)[0]
            c = Case(w, args, dev, flush)
            time_cases([c], args, flush, stream, world)
            e = c.summary(hbm, tensor, ncu_traffic(w.name))
            if oracle_here:
                e["cpu_baseline"] = cpu_baseline([w], [c.inp], budget_s=2.0)
            if not args.no_next_rows:
                e["next_rows"] = next_rows_for(c, args, flush, stream, dev, oracle_here and cname == "llama2_7b")
            per_config[w.name] = e
            c.free()
            del c
            torch.cuda.empty_cache()
    res["per_config"] = per_config
    return res


def run_e2e(cases, args, dev, world):
    """The same metric through the public API with host buffers: every step copies each tree's
    inputs from pinned host memory, runs the three calls and reads the tree and the
    acceptance result back."""
    names = ["draft_logp", "root_tokens", "q", "k_cache", "v_cache", "block_table", "prefix_len", "logits"]
    hosts, outs, h_outs = [], [], []
    for c in cases:
        step = c.step
        hosts.append({n: step.host[n].pin_memory() for n in names})
        o = {"tokens": step.tree["tokens"], "parents": step.tree["parents"], "accept_len": step.acc["accept_len"],
             "accept_path": step.acc["accept_path"], "bonus": step.acc["bonus"]}
        outs.append(o)
        h_outs.append({n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for n, t in o.items()})
    h2d = sum(t.numel() * t.element_size() for h in hosts for t in h.values())
    d2h = sum(t.numel() * t.element_size() for o in outs for t in o.values())
    stream = torch.cuda.current_stream()
    times = []
    for i in range(args.warmup + args.steps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for c, host, o, ho in zip(cases, hosts, outs, h_outs):
            for n in names:
                c.step.d[n].copy_(host[n], non_blocking=True)
            c.step.run()
            for n, t in o.items():
                ho[n].copy_(t, non_blocking=True)
        b.record(stream)
        b.synchronize()
        if i >= args.warmup:
            times.append(a.elapsed_time(b))
    total = allreduce_max(sum(times), world, dev)
    ms = total / args.steps
    step_bytes = sum(c.ab["step"] for c in cases)
    del hosts, h_outs
    return {"value": round(world * step_bytes / (ms * 1e-3) / 1e12, 4), "unit": "TB/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


# hidden size of the target model each workload is shaped after (the LM head is [V, d_model])
D_MODEL = {"llama2_7b": 4096, "llama3_8b_gqa": 4096, "llama2_70b_gqa": 8192}


def run_lm_head(w, args, flush, stream, dev, with_oracle):
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
    if with_oracle:
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


def run_efficient_head(w, args, flush, stream, dev, with_oracle, rank=256, tile_tokens=1024, k_tile=2):
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
    if with_oracle:
        import oracle
        n = min(M, 2)
        t0 = time.perf_counter()
        oracle.efficient_head(h[:n].cpu(), B.cpu(), A.cpu(), W.cpu(), tile_tokens, k_tile, k)
        res["oracle_ms"] = round((time.perf_counter() - t0) * 1e3 * M / n, 2)
        res["oracle_note"] = f"fp64 numpy oracle on {n} of {M} rows, scaled to all rows"
    del h, B, A, W
    return res


def run_accept_sample(step, w, args, flush, stream, with_oracle, temperature=1.0):
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
        if with_oracle:
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


def run_tree_prune(step, w, args, flush, stream, with_oracle, costs=(1.0, 10.0, 0.05)):
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
    if with_oracle:
        import oracle
        hh = {k: v.cpu().numpy() for k, v in tree.items()}
        t0 = time.perf_counter()
        oracle.tree_prune(hh["tokens"], hh["parents"], hh["depth"], hh["values"], *costs, node_row=hh["node_row"])
        res["oracle_ms"] = round((time.perf_counter() - t0) * 1e3, 2)
    return res


def run_kv_commit(step, w, args, flush, stream, with_oracle):
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
    if with_oracle and cache_bytes <= (256 << 20):
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


# ------------------------------------------------------------------------------------
# CPU oracle (reported baseline / reference arm)
# ------------------------------------------------------------------------------------
def oracle_sample(w, inp, heads):
    """One bounded sample of a verify step on the fp64 oracle: sequence 0 only, its whole
    tree_build and tree_accept, and tree_attention for ``heads`` query heads of it (every
    node).  Returns the sample's algorithmic bytes (the unit the metric is scaled by)."""
    import oracle
    tr = oracle.tree_build(inp["draft_logp"][:1].numpy(), inp["root_tokens"][:1].numpy(), w.k, w.depth, w.m)
    sel = [(0, i, h) for i in range(w.m) for h in heads]
    oracle.tree_attention(inp["q"][:1], inp["k_cache"], inp["v_cache"], inp["block_table"][:1].numpy(),
                          inp["prefix_len"][:1].numpy(), tr["mask"], 1.0 / math.sqrt(w.d), select=sel)
    amax = oracle.target_argmax(inp["logits"][:1])
    oracle.accept_longest_path(tr["tokens"], tr["parents"], amax)


def oracle_sample_bytes(w, inp, heads):
    w1 = dataclasses.replace(w, B=1)
    ab = algo_bytes(w1, inp["prefix_len"][:1].tolist())
    return ab["tree_build"] + ab["tree_attention"] * len(heads) / w.Hq + ab["tree_accept"]


def sample_heads(w):
    # query head 0 (every node of sequence 0): a sweep step of the oracle stays near 4 s
    return [0]


def _sample_desc(ws, reps, dt, threads):
    parts = ", ".join(f"{w.name}: {len(sample_heads(w))} of {w.Hq} query heads" for w in ws)
    return (f"fp64 numpy oracle on sequence 0 of each batch: its whole tree_build and tree_accept, "
            f"tree_attention for every node of one query head ({parts}); {reps} repetitions of "
            f"{dt:.3f} s; metric scaled by the sample's algorithmic bytes; numpy's BLAS on {threads} "
            f"thread(s) (the attention products), the tree passes single-threaded")


def oracle_rate(ws, inps, budget_s):
    """Repeat the sample over all workloads of ``ws`` until ``budget_s`` is spent: (bytes/s, reps, s/rep)."""
    byts = sum(oracle_sample_bytes(w, inp, sample_heads(w)) for w, inp in zip(ws, inps))
    t0 = time.perf_counter()
    n = 0
    while True:
        for w, inp in zip(ws, inps):
            oracle_sample(w, inp, sample_heads(w))
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = (time.perf_counter() - t0) / n
    return byts / dt, n, dt


def cpu_baseline(ws, inps, budget_s, single_thread_of=None, args=None):
    """The oracle as it stands on this host: all cores; with ``single_thread_of`` also the same
    sample on one thread (a child process with one BLAS thread)."""
    rate, n, dt = oracle_rate(ws, inps, budget_s)
    res = {"value": round(rate / 1e12, 8), "unit": "TB/s", "cores": _ORACLE_THREADS, "kind": "oracle",
           "sample": _sample_desc(ws, n, dt, _ORACLE_THREADS)}
    if single_thread_of is not None:
        env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
        cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--oracle-child", single_thread_of,
               "--oracle-budget", str(budget_s)]
        if args is not None and args.prefix is not None:
            cmd += ["--prefix", str(args.prefix)]
        try:
            r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600, cwd=ROOT)
            line = [l for l in r.stdout.splitlines() if l.startswith("{")][-1]
            one = json.loads(line)
            res["single_thread"] = {"value": one["value"], "unit": "TB/s", "cores": 1, "sample": one["sample"]}
        except Exception as e:  # reported, not fatal: the GPU line stands without it
            res["single_thread"] = {"value": None, "error": f"{type(e).__name__}: {e}"[:200]}
    return res


def oracle_child(args):
    ws = workload_list(args.oracle_child, args.prefix)
    inps = [workloads.generate(w) for w in ws]
    rate, n, dt = oracle_rate(ws, inps, args.oracle_budget or 10.0)
    print(json.dumps({"value": round(rate / 1e12, 8), "sample": _sample_desc(ws, n, dt, _ORACLE_THREADS)}),
          flush=True)


def run_reference(args, rank, world):
    ws = workload_list(args.workload, args.prefix)
    inps = [workloads.generate(w) for w in ws]
    byts = sum(oracle_sample_bytes(w, inp, sample_heads(w)) for w, inp in zip(ws, inps))
    for _ in range(args.warmup):
        for w, inp in zip(ws, inps):
            oracle_sample(w, inp, sample_heads(w))
    ts_ = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        for w, inp in zip(ws, inps):
            oracle_sample(w, inp, sample_heads(w))
        ts_.append(time.perf_counter() - t0)
    ms = 1e3 * sum(ts_) / len(ts_)
    value = byts / (ms * 1e-3) / 1e12
    sample = _sample_desc(ws, len(ts_), ms / 1e3, _ORACLE_THREADS)
    return {"impl": "reference", "metric": METRIC, "value": round(value, 8), "unit": "TB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(args.workload, args, world),
            "cpu_baseline": {"value": round(value, 8), "unit": "TB/s", "cores": _ORACLE_THREADS, "kind": "oracle",
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
    if args.oracle_child is not None:
        oracle_child(args)
        return
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
    res = run_ours(args, rank, world, dev)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1 and _PG is not None:
        _PG.destroy_process_group()


if __name__ == "__main__":
    main()
