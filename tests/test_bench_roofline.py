"""The bench line's roofline object takes the attention call's binding roof (CPU only)."""
import pytest

import bench
import workloads

HBM = (6795.5, "measured")
TENSOR = (1872.8, "measured")


@pytest.mark.parametrize("name,bound", [("llama2_7b", "hbm"), ("llama2_70b_gqa", "tensor"),
                                        ("long_context_m32", "hbm"), ("long_context_m128", "tensor")])
def test_binding_roof_of_the_fixed_length_workloads(name, bound):
    """Attention FLOPs per K/V byte are about m*g: 60 and 128 sit below the ridge of the two
    peaks (~276), 480 and 512 above it."""
    w = workloads.WORKLOADS[name]
    lens = [w.prefix[0]] * w.B
    byts, flops = bench.algo_bytes(w, lens)["tree_attention"], bench.attention_flops(w, lens)
    r = bench.attention_roofline(byts, flops, 0.1, HBM, TENSOR, None)
    assert r["bound"] == bound


def test_fraction_is_achieved_over_peak_in_the_chosen_unit():
    # 1e9 bytes and 1e12 FLOPs in 1 ms: 1e12 B/s = 1000 GB/s, or 1000 TFLOP/s
    r = bench.attention_roofline(1e9, 1e11, 1.0, HBM, TENSOR, 123)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["achieved"] == 1000.0
    assert r["frac"] == round(1000.0 / 6795.5, 4) and r["traffic"] == 123
    r = bench.attention_roofline(1e8, 1e12, 1.0, HBM, TENSOR, None)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["achieved"] == 1000.0
    assert r["frac"] == round(1000.0 / 1872.8, 4) and r["peak"] == 1872.8


def test_algorithmic_bytes_are_the_documented_per_unit_counts():
    """The roofline's numerator, counted by hand from the per-unit figures: each input byte read
    once, each output byte written once (Llama-2-7B shape: B 1, 51 draft rows of 32000 fp32,
    m 60, 32 heads of 128, 2048-token prefix in 16-token pages; long-context m64: B 4, 71 rows
    of 128256, m 64, 32/8 heads, 32768-token prefixes)."""
    w = workloads.WORKLOADS["llama2_7b"]
    b = bench.algo_bytes(w, [2048])
    # draft rows in, root token in; tokens/parents/depth int32, one mask word, fp64 value out
    assert b["tree_build"] == 51 * 32000 * 4 + 4 + 60 * (3 * 4 + 8 + 8)
    # K and V of prefix + tree, Q and out, one mask word per node, 132 page ids, the prefix
    # length, the fp32 log-sum-exp per (node, head)
    assert b["tree_attention"] == ((2048 + 60) * 32 * 128 * 2 * 2 + 2 * 60 * 32 * 128 * 2 + 60 * 8
                                   + 132 * 4 + 4 + 60 * 32 * 4)
    # bf16 logits, tokens + parents in; argmax + path out; length + bonus out
    assert b["tree_accept"] == 60 * 32000 * 2 + 60 * 8 + 60 * 8 + 8
    assert b["step"] == b["tree_build"] + b["tree_attention"] + b["tree_accept"] == 45899856

    w = workloads.WORKLOADS["long_context_m64"]
    lens = [32768] * 4
    b = bench.algo_bytes(w, lens)
    assert b["tree_build"] == 4 * 71 * 128256 * 4 + 4 * 4 + 4 * 64 * (3 * 4 + 8 + 8)
    assert b["tree_attention"] == 4 * ((32768 + 64) * 8 * 128 * 2 * 2 + 2 * 64 * 32 * 128 * 2 + 64 * 8
                                       + 2052 * 4 + 4 + 64 * 32 * 4)
    assert b["tree_accept"] == 4 * (64 * 128256 * 2 + 64 * 8 + 64 * 8 + 8)
    # 4 d FLOPs per (query row, prefix key): two d-long dot products, multiply and add
    assert bench.attention_flops(w, lens) == 4 * 128 * (64 * 32) * (4 * 32768)


def test_reference_arm_line_has_the_contract_keys_and_our_config():
    """One process, the tiny workload: the reference arm (the fp64 oracle on the host) prints
    one JSON line with the contract's keys, and its ``config`` is the object the GPU arm
    prints for the same arguments."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    argv = ["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "0"]
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py")] + argv, capture_output=True,
                       text=True, timeout=300, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1 and d["value"] > 0
    assert d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"] == bench.config_of("tiny", bench.parse(argv), 1)
