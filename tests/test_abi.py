"""The C-ABI library builds, loads and exports every declared entry point; host-side
validation rejects bad arguments before any launch (CPU only: no compute call)."""
import ctypes
import os
import re

import pytest

import speculative_decoding_tree_eagle_gb300 as ts
from speculative_decoding_tree_eagle_gb300 import build as tsbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "treespec.h")

TS_OK, TS_ERR_INVALID, TS_ERR_UNSUPPORTED = 0, -1, -2


@pytest.fixture(scope="module")
def lib():
    tsbuild.build()
    return ts.library()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ts_[a-z_]+)\s*\(", text)))


def test_header_declares_the_three_operations():
    syms = declared_symbols()
    for s in ("ts_tree_build", "ts_tree_attention", "ts_tree_accept", "ts_kv_commit"):
        assert s in syms


def test_every_declared_symbol_is_exported(lib):
    for s in declared_symbols():
        assert hasattr(lib, s), s


def test_status_strings(lib):
    assert ts.status_string(0) == "TS_OK"
    for c in (-1, -2, -3, -4, -5, -6):
        assert ts.status_string(c).startswith("TS_ERR_")
    assert lib.ts_version() == 1


def _build(lib, B=1, V=100, k=2, depth=3, m=8, ptr=1):
    P = ptr
    return lib.ts_tree_build(P, P, B, V, k, depth, m, P, P, P, P, None, None, P, 1 << 20, None, None)


def test_tree_build_validation(lib):
    assert _build(lib, B=0) == TS_ERR_INVALID
    assert _build(lib, m=0) == TS_ERR_INVALID
    assert _build(lib, k=17) == TS_ERR_UNSUPPORTED
    assert _build(lib, depth=17) == TS_ERR_UNSUPPORTED
    assert _build(lib, m=257) == TS_ERR_UNSUPPORTED
    assert _build(lib, m=12) == TS_ERR_INVALID          # m-1 > k + (depth-1)k^2 = 10
    assert _build(lib, V=1) == TS_ERR_INVALID           # k > V
    assert _build(lib, ptr=None) == TS_ERR_INVALID      # null pointers
    assert lib.ts_tree_build_workspace(1, 100, 2, 3, 12) == 0


def _attn(lib, dt=1, B=1, m=8, Hq=4, Hkv=1, d=128, maxp=64, nb=10, bs=16, mb=8, scale=0.1, ptr=1):
    P = ptr
    return lib.ts_tree_attention(P, P, P, dt, nb, bs, P, mb, P, maxp, P, B, m, Hq, Hkv, d, scale, P, None,
                                 P, 1 << 20, None, None)


def test_tree_attention_validation(lib):
    assert _attn(lib, Hq=6, Hkv=4) == TS_ERR_INVALID          # Hq % Hkv
    assert _attn(lib, dt=7) == TS_ERR_INVALID
    assert _attn(lib, m=300) == TS_ERR_UNSUPPORTED
    assert _attn(lib, d=512) == TS_ERR_UNSUPPORTED
    assert _attn(lib, maxp=-1) == TS_ERR_INVALID
    assert _attn(lib, mb=4) == TS_ERR_INVALID                 # 4*16 < 64 + 8
    assert _attn(lib, ptr=None) == TS_ERR_INVALID
    assert _attn(lib, scale=float("nan")) == TS_ERR_INVALID
    assert _attn(lib, nb=0) == TS_ERR_INVALID


def _accept(lib, dt=1, B=1, m=8, V=100, ptr=1):
    P = ptr
    return lib.ts_tree_accept(P, dt, P, P, B, m, V, P, P, P, P, P, 1 << 20, None, None)


def test_tree_accept_validation(lib):
    assert _accept(lib, B=0) == TS_ERR_INVALID
    assert _accept(lib, V=0) == TS_ERR_INVALID
    assert _accept(lib, dt=3) == TS_ERR_INVALID
    assert _accept(lib, m=257) == TS_ERR_UNSUPPORTED
    assert _accept(lib, ptr=None) == TS_ERR_INVALID


def _commit(lib, dt=1, nb=10, bs=16, hkv=2, d=128, maxb=4, B=1, m=8, ptr=1):
    P = ptr
    return lib.ts_kv_commit(P, P, dt, nb, bs, hkv, d, P, maxb, P, P, P, B, m, P, P, None, None)


def test_kv_commit_validation(lib):
    assert _commit(lib, B=0) == TS_ERR_INVALID
    assert _commit(lib, m=0) == TS_ERR_INVALID
    assert _commit(lib, bs=0) == TS_ERR_INVALID
    assert _commit(lib, maxb=0) == TS_ERR_INVALID
    assert _commit(lib, dt=3) == TS_ERR_INVALID
    assert _commit(lib, d=3) == TS_ERR_INVALID          # bf16 rows of 6 bytes
    assert _commit(lib, m=257) == TS_ERR_UNSUPPORTED
    assert _commit(lib, ptr=None) == TS_ERR_INVALID


def _sample(lib, dt=1, B=1, m=8, V=100, T=1.0, mode=0, R=3, ptr=1, draft=1, ws=None, wsb=0):
    P = ptr
    return lib.ts_tree_accept_sample(P, dt, P, P, P, draft, draft, R, B, m, V, T, mode, P, P, P, ws, wsb, None, None)


def test_tree_accept_sample_validation(lib):
    assert _sample(lib, B=0) == TS_ERR_INVALID
    assert _sample(lib, V=0) == TS_ERR_INVALID
    assert _sample(lib, dt=3) == TS_ERR_INVALID
    assert _sample(lib, mode=2) == TS_ERR_INVALID
    for T in (0.0, -1.0, float("inf"), float("nan")):
        assert _sample(lib, T=T) == TS_ERR_INVALID
    assert _sample(lib, m=257) == TS_ERR_UNSUPPORTED
    assert _sample(lib, V=(1 << 20) + 1) == TS_ERR_UNSUPPORTED
    assert _sample(lib, ptr=None) == TS_ERR_INVALID
    assert _sample(lib, mode=1, draft=None) == TS_ERR_INVALID       # draft mode needs the rows
    assert _sample(lib, mode=1, R=0) == TS_ERR_INVALID
    assert _sample(lib, mode=1) == TS_ERR_INVALID                    # and a workspace
    assert _sample(lib, mode=1, ws=1, wsb=16) == -3                  # too small
    assert lib.ts_tree_accept_sample_workspace(1, 100, 0) == 0
    assert lib.ts_tree_accept_sample_workspace(2, 100, 1) >= 2 * 2 * 104 * 4
    assert lib.ts_tree_accept_sample_workspace(2, 100, 7) == 0


def _prune(lib, B=2, m=8, td=1.0, tf=1.0, tn=0.1, ptr=1, nr=None, nro=None, ws=1, wsb=1 << 20):
    P = ptr
    return lib.ts_tree_prune(P, P, P, P, nr, B, m, td, tf, tn, P, P, P, P, P, P, nro, P, P, ws, wsb, None, None)


def test_tree_prune_validation(lib):
    assert _prune(lib, B=0) == TS_ERR_INVALID
    assert _prune(lib, m=0) == TS_ERR_INVALID
    assert _prune(lib, m=257) == TS_ERR_UNSUPPORTED
    assert _prune(lib, td=-1.0) == TS_ERR_INVALID
    assert _prune(lib, tn=float("nan")) == TS_ERR_INVALID
    assert _prune(lib, tf=float("inf")) == TS_ERR_INVALID
    assert _prune(lib, td=0.0, tf=0.0, tn=0.0) == TS_ERR_INVALID   # no cost at all
    assert _prune(lib, ptr=None) == TS_ERR_INVALID
    assert _prune(lib, nro=1) == TS_ERR_INVALID                    # node_row_out without node_row
    assert _prune(lib, wsb=16) == -3
    assert lib.ts_tree_prune_workspace(2, 8) >= 2 * 8 * 8
    assert lib.ts_tree_prune_workspace(2, 257) == 0


def test_selftest_validation(lib):
    assert lib.ts_selftest_bounded_wait(2, 1, None, None) == TS_ERR_INVALID
    assert lib.ts_selftest_bounded_wait(0, None, None, None) == TS_ERR_INVALID


def test_workspace_queries_are_positive_for_valid_sizes(lib):
    assert lib.ts_tree_build_workspace(8, 128256, 10, 7, 64) > 0
    assert lib.ts_tree_accept_workspace(1, 8, 64, 128256) > 0
    assert lib.ts_tree_attention_workspace(1, 4, 128, 32, 8, 128, 32768) > 0


def test_binding_refuses_cpu_tensors(lib):
    import torch
    with pytest.raises(ValueError):
        ts.tree_accept(torch.zeros(1, 2, 4), torch.zeros(1, 2, dtype=torch.int32),
                       torch.zeros(1, 2, dtype=torch.int32))


def test_binding_covers_every_public_call(lib):
    """Every public name of the binding exists, and each public library call of the header
    that a Python user needs has a binding function of the same name without the ts_ prefix
    (the self-test, version, status, launch-count, plan, workspace and no-allocation entry
    points are reached through ``library()``)."""
    for name in ts.__all__:
        assert hasattr(ts, name), name
    internal = ("ts_selftest_", "ts_version", "ts_status_string", "ts_launch_count", "_workspace",
                "ts_tree_accept_noalloc", "ts_efficient_head_candidates", "ts_tree_attention_plan")
    for sym in declared_symbols():
        if any(part in sym for part in internal):
            continue
        assert sym[3:] in ts.__all__, sym


@pytest.mark.parametrize("name,row_groups,chunks,tiles", [
    ("llama2_7b", 1, 4, 5),            # 2108 keys = 17 tiles; 32 units on 152 SMs
    ("llama3_8b_gqa", 2, 2, 33),       # one chunk would leave SMs idle: split in two halves
    ("llama2_70b_gqa", 4, 1, 33),      # 512 CTAs already fill several waves
    ("long_context_m8", 1, 4, 65),     # 257 tiles over 4 chunks
    ("long_context_m32", 1, 4, 65),
    ("long_context_m64", 2, 2, 129),
    ("long_context_m128", 4, 2, 129),
])
def test_attention_plan_on_a_gb300(lib, name, row_groups, chunks, tiles, monkeypatch):
    """The planner's split of each workload for 152 SMs: row groups of 128 GEMM rows
    (node x head in group), chunks per (sequence, KV head, row group) and tiles per chunk."""
    import torch
    import workloads
    for var in ("TREESPEC_ATTN_SPLIT", "TREESPEC_ATTN_MC", "TREESPEC_ATTN_ISSUE"):
        monkeypatch.delenv(var, raising=False)
    w = workloads.WORKLOADS[name]
    plan = ts.tree_attention_plan(torch.bfloat16, w.B, w.m, w.Hq, w.Hkv, w.d, w.max_prefix, 16, num_sms=152)
    assert plan["path"] == "tensor-core"
    assert (plan["row_groups"], plan["chunks"], plan["tiles_per_chunk"]) == (row_groups, chunks, tiles)
    assert plan["row_groups"] == -(-w.m * (w.Hq // w.Hkv) // 128)
    assert plan["chunks"] * plan["tiles_per_chunk"] >= -(-(w.max_prefix + w.m) // 128)
    assert (plan["split"] == "one chunk") == (plan["chunks"] == 1)


def test_attention_plan_paths_and_validation(lib):
    import torch
    # fp32 and d = 64 take the CUDA-core kernel; no SM count is needed for them
    assert ts.tree_attention_plan(torch.float32, 1, 8, 1, 1, 64, 16, 16, num_sms=152)["path"] == "cuda-core"
    assert ts.tree_attention_plan(torch.bfloat16, 1, 8, 4, 1, 64, 16, 16, num_sms=152)["path"] == "cuda-core"
    out = (ctypes.c_int * 6)()
    assert lib.ts_tree_attention_plan_for_sms(1, 1, 8, 4, 1, 128, 64, 16, 0, out) == TS_ERR_INVALID
    assert lib.ts_tree_attention_plan_for_sms(1, 1, 8, 6, 4, 128, 64, 16, 152, out) == TS_ERR_INVALID
    assert lib.ts_tree_attention_plan_for_sms(1, 1, 8, 4, 1, 128, 64, 16, 152, None) == TS_ERR_INVALID
