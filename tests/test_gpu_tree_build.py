"""GPU tree_build vs the fp64 oracle: bit-exact tokens, parents, depth, mask and values."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_tree_eagle_gb300 as ts
import workloads
from gpu_helpers import dev, lib

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _run_and_compare(draft_logp: torch.Tensor, roots: torch.Tensor, k, depth, m, gpu_logp=None):
    lib()
    status = ts.new_status(dev())
    x = gpu_logp if gpu_logp is not None else draft_logp.to(dev())
    got = ts.tree_build(x, roots.to(dev()), k, depth, m, status=status)
    ts.check_status(status)
    ref = oracle.tree_build(draft_logp.numpy(), roots.numpy(), k, depth, m)
    for key in ("tokens", "parents", "depth", "node_row"):
        np.testing.assert_array_equal(got[key].cpu().numpy(), ref[key], err_msg=key)
    np.testing.assert_array_equal(got["mask"].cpu().numpy().view(np.uint64), ref["mask_words"])
    np.testing.assert_array_equal(got["values"].cpu().numpy(), ref["values"])
    return got, ref


def test_hand_case_reproduces_page_tree():
    with open(os.path.join(GOLDEN, "hand_build_case.json")) as f:
        g = json.load(f)
    V, ids = g["vocab"], g["token_ids"]
    rows = []
    for r in g["rows"]:
        p = np.full(V, (1.0 - sum(pr for _, pr in r["top"])) / (V - len(r["top"])))
        for w_, pr in r["top"]:
            p[ids[w_]] = pr
        rows.append(np.log(p).astype(np.float32))
    logp = torch.from_numpy(np.stack(rows))[None].contiguous()
    got, _ = _run_and_compare(logp, torch.tensor([ids[g["root"]]], dtype=torch.int32), 2, 3, 8)
    assert got["parents"][0].tolist() == g["expected"]["parents"]
    assert got["tokens"][0].tolist() == [ids[w_] for w_ in g["expected"]["words"]]


@pytest.mark.parametrize("name", ["tiny", "llama2_7b", "llama3_8b_gqa", "llama2_70b_gqa", "long_context_m8",
                                  "long_context_m32", "long_context_m64", "long_context_m128"])
def test_workloads_full_size(name):
    w = workloads.WORKLOADS[name]
    inp = workloads.generate(w, with_attention=False, with_logits=False)
    _run_and_compare(inp["draft_logp"], inp["root_tokens"], w.k, w.depth, w.m)


def _logp(B, R, V, seed, sigma=2.0):
    g = torch.Generator().manual_seed(seed)
    return torch.log_softmax(torch.randn(B, R, V, generator=g) * sigma, dim=-1).contiguous()


@pytest.mark.parametrize("k,depth,m,V", [(1, 7, 8, 500), (2, 3, 1, 100), (16, 16, 256, 64), (10, 6, 60, 1001),
                                         (3, 5, 40, 4099), (4, 2, 21, 33), (8, 8, 129, 2048)])
def test_edge_shapes(k, depth, m, V):
    B = 3
    R = 1 + (depth - 1) * k
    logp = _logp(B, R, V, seed=k * 100 + depth)
    roots = torch.tensor([0, V - 1, V // 2], dtype=torch.int32)
    _run_and_compare(logp, roots, k, depth, m)


def test_ties_everywhere():
    """Values quantised to multiples of 0.5 (and -0.0): ties in top-k, frontier and rerank."""
    g = torch.Generator().manual_seed(9)
    B, k, depth, m, V = 2, 4, 5, 40, 300
    R = 1 + (depth - 1) * k
    logp = -(torch.round(torch.randn(B, R, V, generator=g).abs() * 2) / 2)
    logp[0, 0, 7] = -0.0
    logp[0, 0, 3] = 0.0
    _run_and_compare(logp.contiguous(), torch.tensor([1, 2], dtype=torch.int32), k, depth, m)


@pytest.mark.parametrize("order", ["ascending", "descending", "constant", "one_finite"])
def test_row_orders_that_defeat_early_bounds(order):
    """Row layouts chosen against the streaming top-k: every element a new best (ascending), no
    candidate after the first batch (descending), ties everywhere (constant: the k smallest
    indices win), and a single finite entry per row (the rest of each top-k is -inf, taken by
    smallest index).  Rows long enough for several batches per warp."""
    B, k, depth, m, V = 2, 6, 4, 30, 40000
    R = 1 + (depth - 1) * k
    ramp = torch.linspace(-20.0, -1.0, V)
    if order == "ascending":
        logp = ramp.expand(B, R, V)
    elif order == "descending":
        logp = ramp.flip(0).expand(B, R, V)
    elif order == "constant":
        logp = torch.full((B, R, V), -3.0)
    else:
        logp = torch.full((B, R, V), float("-inf"))
        g = torch.Generator().manual_seed(5)
        pos = torch.randint(0, V, (B, R), generator=g)
        logp.scatter_(2, pos.unsqueeze(-1), -0.5)
    _run_and_compare(logp.contiguous(), torch.tensor([3, 4], dtype=torch.int32), k, depth, m)


def test_many_rows_one_warp_each():
    """More draft rows than 32 per SM: one warp per row (the whole row in one segment)."""
    B, k, depth, m, V = 64, 10, 8, 64, 3000
    R = 1 + (depth - 1) * k
    logp = _logp(B, R, V, seed=17)
    roots = torch.arange(B, dtype=torch.int32) % V
    _run_and_compare(logp, roots, k, depth, m)


def test_unaligned_rows_take_the_scalar_path():
    B, k, depth, m, V = 2, 3, 4, 20, 1024
    R = 1 + (depth - 1) * k
    logp = _logp(B, R, V, seed=3)
    flat = torch.empty(B * R * V + 1, device=dev())
    gpu = flat[1:].view(B, R, V)
    gpu.copy_(logp.to(dev()))
    _run_and_compare(logp, torch.tensor([5, 6], dtype=torch.int32), k, depth, m, gpu_logp=gpu)


def test_positive_logprob_breaks_connectivity_is_reported():
    """A child value above its parent's (log-prob > 0) can make the rerank pick a node
    without its parent: the kernel reports TS_ERR_DEVICE_CHECK instead of a broken tree."""
    lib()
    V = 50
    logp = torch.full((1, 3, V), -10.0)
    logp[0, 0, 1], logp[0, 0, 2] = -1.0, -5.0     # root row: children 1 (-1), 2 (-5)
    logp[0, 1, 3], logp[0, 1, 4] = -9.0, -9.5     # row of the first frontier slot
    logp[0, 2, 5], logp[0, 2, 6] = 8.0, -9.9      # row of child 2: a positive "log-prob"
    status = ts.new_status(dev())
    ts.tree_build(logp.to(dev()), torch.tensor([0], dtype=torch.int32, device=dev()), 2, 2, 3, status=status)
    assert int(status.item()) == -6
    with pytest.raises(ValueError):
        oracle.tree_build(logp.numpy(), np.array([0]), 2, 2, 3)
