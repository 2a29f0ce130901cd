"""GPU tree_attention vs the fp64 oracle.

fp32 inputs: max abs error <= 1e-5.  bf16 inputs (fp32 accumulation, P rounded to bf16 for
the PV product): every element within 2e-2 absolute or 1e-2 relative.  Small cases compare
every output; the full workloads compare sampled (sequence, node, head) outputs.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_tree_eagle_gb300 as ts
import workloads
from gpu_helpers import (assert_attention_close, dev, full_workload, lib, oracle_tree, sample_rows,
                         scale_of, words_i64)

pytestmark = pytest.mark.gpu


def _run(inp, w, tree_mask_bool, mask_words, select=None, gpu_inputs=None, with_lse=True):
    lib()
    status = ts.new_status(dev())
    g = gpu_inputs or {k: inp[k].to(dev()) for k in ("q", "k_cache", "v_cache", "block_table", "prefix_len")}
    out, lse = ts.tree_attention(g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["prefix_len"],
                                 words_i64(mask_words), max_prefix=w.max_prefix, status=status,
                                 with_lse=with_lse)
    ts.check_status(status)
    ref, ref_lse = oracle.tree_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"].numpy(),
                                         inp["prefix_len"].numpy(), tree_mask_bool, scale_of(w), select=select)
    dtype = inp["q"].dtype
    assert_attention_close(out, ref, dtype, where=select)
    if with_lse:
        got_lse = lse.double().cpu().numpy()
        if select is not None:
            got_lse = np.array([got_lse[b, i, h] for (b, i, h) in select])
            ref_lse = np.array([ref_lse[b, i, h] for (b, i, h) in select])
        tol = 1e-5 if dtype == torch.float32 else 1e-2
        assert np.abs(got_lse - ref_lse).max() <= tol
    return out


def test_tiny_fp32_page_tree():
    w, inp, tree = full_workload("tiny")
    _run(inp, w, tree["mask"], tree["mask_words"])


def _small(name, **kw):
    w = workloads.custom(name=name, **kw)
    inp = workloads.generate(w, with_logits=False)
    tree = oracle_tree(inp, w)
    return w, inp, tree


# (B, Hq, Hkv, d, prefix range, m, k, depth): rows = m*Hq/Hkv spans 1 to 4 row groups of 128
# rows; the prefixes span several 128-key tiles and end mid-tile; some force split-K over chunks.
SMALL = [
    dict(B=2, Hq=8, Hkv=2, prefix=(150, 150), m=8, k=2, depth=3),            # 32 rows, one M tile
    dict(B=3, Hq=8, Hkv=2, prefix=(1, 700), m=8, k=2, depth=3),              # ragged prefixes
    dict(B=2, Hq=64, Hkv=8, prefix=(300, 300), m=60, k=8, depth=6),          # 480 rows: 2 row groups
    dict(B=1, Hq=32, Hkv=8, prefix=(1000, 1000), m=128, k=10, depth=8),      # 512 rows, 2 mask words
    dict(B=2, Hq=4, Hkv=4, prefix=(64, 64), m=60, k=10, depth=6),            # MHA, prefix = one tile
    dict(B=1, Hq=4, Hkv=1, prefix=(5000, 5000), m=32, k=10, depth=8),        # long: split-K
    dict(B=2, Hq=2, Hkv=1, prefix=(0, 0), m=64, k=10, depth=7),              # no prefix: tree only
    dict(B=1, Hq=1, Hkv=1, prefix=(33, 33), m=256, k=16, depth=16, V=64),    # 256 nodes, 4 mask words
    dict(B=2, Hq=8, Hkv=1, prefix=(128, 128), m=1, k=2, depth=2),            # m = 1: decode attention
]


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: f"B{c['B']}_H{c['Hq']}x{c['Hkv']}_L{c['prefix'][1]}_m{c['m']}")
def test_bf16_small_all_outputs(cfg):
    w, inp, tree = _small("attn_small", **cfg)
    _run(inp, w, tree["mask"], tree["mask_words"])


@pytest.mark.parametrize("bs", [32, 64, 128])
def test_bf16_block_sizes(bs, monkeypatch):
    monkeypatch.setattr(workloads, "BLOCK_SIZE", bs)
    w, inp, tree = _small(f"attn_bs{bs}", B=2, Hq=8, Hkv=2, prefix=(200, 420), m=16, k=4, depth=4)
    assert inp["k_cache"].shape[2] == bs
    _run(inp, w, tree["mask"], tree["mask_words"])


def test_bf16_head_dim_64_cuda_core_path():
    w, inp, tree = _small("attn_d64", B=2, Hq=4, Hkv=2, d=64, prefix=(70, 90), m=8, k=2, depth=3)
    _run(inp, w, tree["mask"], tree["mask_words"])


def test_fp32_gqa_ragged():
    w, inp, tree = _small("attn_f32", B=2, Hq=6, Hkv=3, d=96, prefix=(10, 40), m=12, k=3, depth=4, dtype="f32")
    _run(inp, w, tree["mask"], tree["mask_words"])


def test_non_finite_garbage_after_sequence_end_is_ignored():
    """Cache slots past L_b + m in a sequence's last block may hold anything (here NaN/inf):
    they must not reach the output."""
    w, inp, tree = _small("attn_garbage", B=2, Hq=8, Hkv=2, prefix=(100, 170), m=8, k=2, depth=3)
    kc, vc = inp["k_cache"].clone(), inp["v_cache"].clone()
    bs = kc.shape[2]
    for b in range(w.B):
        n = int(inp["prefix_len"][b]) + w.m
        last = int(inp["block_table"][b, (n - 1) // bs])
        if n % bs:
            kc[last, :, n % bs:, :] = float("nan")
            vc[last, :, n % bs:, :] = float("inf")
    inp = dict(inp, k_cache=kc, v_cache=vc)
    _run(inp, w, tree["mask"], tree["mask_words"])


def test_bad_block_id_is_reported():
    lib()
    w, inp, tree = _small("attn_badblk", B=1, Hq=4, Hkv=1, prefix=(100, 100), m=8, k=2, depth=3)
    table = inp["block_table"].clone()
    table[0, 2] = int(inp["num_blocks"]) + 5
    status = ts.new_status(dev())
    ts.tree_attention(inp["q"].to(dev()), inp["k_cache"].to(dev()), inp["v_cache"].to(dev()), table.to(dev()),
                      inp["prefix_len"].to(dev()), words_i64(tree["mask_words"]), max_prefix=w.max_prefix,
                      status=status)
    assert int(status.item()) == -6


def test_prefix_above_max_prefix_is_reported():
    lib()
    w, inp, tree = _small("attn_badlen", B=1, Hq=4, Hkv=1, prefix=(100, 100), m=8, k=2, depth=3)
    status = ts.new_status(dev())
    ts.tree_attention(inp["q"].to(dev()), inp["k_cache"].to(dev()), inp["v_cache"].to(dev()),
                      inp["block_table"].to(dev()), torch.tensor([101], dtype=torch.int32, device=dev()),
                      words_i64(tree["mask_words"]), max_prefix=100, status=status)
    assert int(status.item()) == -6


@pytest.mark.parametrize("name", ["llama2_7b", "llama3_8b_gqa", "llama2_70b_gqa", "long_context_m8",
                                  "long_context_m32", "long_context_m64", "long_context_m128"])
def test_workloads_full_size_sampled(name):
    w = workloads.WORKLOADS[name]
    inp = workloads.generate(w, with_logits=False)
    tree = oracle_tree(inp, w)
    sel = sample_rows(w, np.random.default_rng(w.seed))
    _run(inp, w, tree["mask"], tree["mask_words"], select=sel)


SPLITS = [("direct", 0), ("cluster:2", 1), ("cluster:4", 1), ("cluster:8", 1), ("global:3", 2), ("global:11", 2)]
ROW_CASES = [dict(B=2, Hq=8, Hkv=2, m=30, k=5, depth=6),      # 120 rows: one row group
             dict(B=1, Hq=16, Hkv=4, m=60, k=8, depth=6)]     # 240 rows: two row groups


@pytest.mark.parametrize("multicast", [True, False], ids=["multicast", "no_multicast"])
@pytest.mark.parametrize("rows_case", ROW_CASES, ids=["one_row_group", "two_row_groups"])
@pytest.mark.parametrize("split,mode", SPLITS, ids=[s for s, _ in SPLITS])
def test_every_split_mode_repeated_calls(split, mode, rows_case, multicast, monkeypatch):
    """Force each way of splitting a sequence over CTAs (one chunk, chunks merged inside a
    cluster, chunks merged through the workspace) with chunks long enough to wrap the K/V
    ring several times, with and without the row groups sharing K/V tiles by multicast;
    five calls in a row must agree exactly and match the oracle."""
    lib()
    rows = rows_case["m"] * rows_case["Hq"] // rows_case["Hkv"]
    if rows <= 128 and not multicast:
        pytest.skip("one row group: nothing to multicast")
    if rows > 128 and multicast and split == "cluster:8":
        pytest.skip("2 row groups x 8 chunks exceed the largest cluster (8 CTAs)")
    monkeypatch.setenv("TREESPEC_ATTN_SPLIT", split)
    if not multicast:
        monkeypatch.setenv("TREESPEC_ATTN_MC", "1")
    w, inp, tree = _small("attn_split", prefix=(1900, 1900), **rows_case)
    plan = ts.tree_attention_plan(inp["q"].dtype, w.B, w.m, w.Hq, w.Hkv, w.d, w.max_prefix, 16)
    assert plan["split"] == {0: "one chunk", 1: "cluster merge", 2: "workspace merge"}[mode], plan
    assert plan["multicast"] == (2 if rows > 128 and multicast else 1), plan
    g = {k: inp[k].to(dev()) for k in ("q", "k_cache", "v_cache", "block_table", "prefix_len")}
    first = None
    for _ in range(5):
        status = ts.new_status(dev())
        out, _ = ts.tree_attention(g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["prefix_len"],
                                   words_i64(tree["mask_words"]), max_prefix=w.max_prefix, status=status)
        ts.check_status(status)
        if first is None:
            first = out.clone()
        else:
            assert torch.equal(out, first)
    ref, _ = oracle.tree_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"].numpy(),
                                   inp["prefix_len"].numpy(), tree["mask"], scale_of(w))
    assert_attention_close(first, ref, torch.bfloat16)


@pytest.mark.parametrize("cfg", [dict(B=3, Hq=32, Hkv=8, prefix=(100, 2000), m=64, k=10, depth=7),    # 2 row groups
                                 dict(B=2, Hq=64, Hkv=8, prefix=(700, 1500), m=60, k=8, depth=6),     # 4 row groups
                                 dict(B=2, Hq=24, Hkv=2, prefix=(300, 900), m=32, k=6, depth=5)],     # 3 row groups
                         ids=["2_groups", "4_groups", "3_groups"])
def test_multicast_equals_separate_loads(cfg, monkeypatch):
    """Row groups that receive their K/V tiles by TMA multicast compute exactly what they
    compute from their own loads (ragged prefixes, garbage past each sequence's end); the
    split is fixed (one chunk) so that the two runs sum in the same order."""
    lib()
    monkeypatch.setenv("TREESPEC_ATTN_SPLIT", "direct")
    w, inp, tree = _small("attn_mc", **cfg)
    kc, vc = inp["k_cache"].clone(), inp["v_cache"].clone()
    bs = kc.shape[2]
    for b in range(w.B):
        n = int(inp["prefix_len"][b]) + w.m
        last = int(inp["block_table"][b, (n - 1) // bs])
        if n % bs:
            kc[last, :, n % bs:, :] = float("nan")
            vc[last, :, n % bs:, :] = float("inf")
    inp = dict(inp, k_cache=kc, v_cache=vc)
    g = {k: inp[k].to(dev()) for k in ("q", "k_cache", "v_cache", "block_table", "prefix_len")}
    outs = []
    for mc in ("default", "1"):
        if mc == "1":
            monkeypatch.setenv("TREESPEC_ATTN_MC", "1")
        plan = ts.tree_attention_plan(inp["q"].dtype, w.B, w.m, w.Hq, w.Hkv, w.d, w.max_prefix, 16)
        assert (plan["multicast"] > 1) == (mc == "default"), plan
        status = ts.new_status(dev())
        out, lse = ts.tree_attention(g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["prefix_len"],
                                     words_i64(tree["mask_words"]), max_prefix=w.max_prefix, status=status)
        ts.check_status(status)
        outs.append((out.clone(), lse.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    ref, _ = oracle.tree_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"].numpy(),
                                   inp["prefix_len"].numpy(), tree["mask"], scale_of(w))
    assert_attention_close(outs[0][0], ref, torch.bfloat16)


@pytest.mark.parametrize("split", ["auto", "global:2", "global:3", "direct"])
def test_ragged_batch_longest_first(split, monkeypatch):
    """Sequences of very different lengths (several shorter than one chunk): the CTAs are
    dispatched longest sequence first and short sequences leave their later chunks empty;
    every output matches the oracle."""
    lib()
    if split != "auto":
        monkeypatch.setenv("TREESPEC_ATTN_SPLIT", split)
    w, inp, tree = _small("attn_ragged", B=6, Hq=16, Hkv=4, prefix=(5, 3000), m=16, k=4, depth=4)
    lens = inp["prefix_len"].tolist()
    assert max(lens) - min(lens) > 1000, lens
    _run(inp, w, tree["mask"], tree["mask_words"])


@pytest.mark.parametrize("split", ["direct", "cluster:2", "global:3"])
@pytest.mark.parametrize("cfg", [dict(B=2, Hq=8, Hkv=2, prefix=(1500, 2300), m=30, k=5, depth=6),    # 1 row group
                                 dict(B=2, Hq=32, Hkv=8, prefix=(900, 2100), m=64, k=10, depth=7),   # 2 row groups
                                 dict(B=2, Hq=64, Hkv=8, prefix=(700, 1500), m=60, k=8, depth=6)],   # 4 row groups
                         ids=["1_group", "2_groups", "4_groups"])
def test_one_and_two_mma_issuers_agree(cfg, split, monkeypatch):
    """Q K^T and P V issued by one thread (in issue order) or by two threads (each gated by its
    barriers, the softmax waiting until P V has read a P buffer before rewriting it): the same
    MMAs in the same order per accumulator, so the outputs and log-sum-exps are bit-identical,
    and both match the oracle."""
    lib()
    monkeypatch.setenv("TREESPEC_ATTN_SPLIT", split)
    w, inp, tree = _small("attn_issue", **cfg)
    g = {k: inp[k].to(dev()) for k in ("q", "k_cache", "v_cache", "block_table", "prefix_len")}
    outs = []
    for issue in ("1", "2"):
        monkeypatch.setenv("TREESPEC_ATTN_ISSUE", issue)
        status = ts.new_status(dev())
        out, lse = ts.tree_attention(g["q"], g["k_cache"], g["v_cache"], g["block_table"], g["prefix_len"],
                                     words_i64(tree["mask_words"]), max_prefix=w.max_prefix, status=status)
        ts.check_status(status)
        outs.append((out.clone(), lse.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    ref, _ = oracle.tree_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"].numpy(),
                                   inp["prefix_len"].numpy(), tree["mask"], scale_of(w))
    assert_attention_close(outs[1][0], ref, torch.bfloat16)
