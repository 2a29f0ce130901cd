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
