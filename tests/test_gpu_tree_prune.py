"""GPU cost-aware tree pruning vs the oracle.

The rerank positions and the pruned trees are integer work and must match exactly.  The node
count n is an argmax of rates the GPU computes in fp32 (fp32 exp of the values, fp32 sums);
near a flat optimum it may pick a neighbour of the oracle's n, so the test requires the GPU's
n to reach the oracle's best rate within 1e-5 (relative) and then compares the pruned tree
with the oracle's tree for that same n.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_tree_eagle_gb300 as ts
import workloads
from gpu_helpers import dev, lib

pytestmark = pytest.mark.gpu

COSTS = [(1.0, 10.0, 0.05), (0.5, 2.0, 0.2), (0.0, 1.0, 0.001), (3.0, 30.0, 0.02)]


def _confident_rows(w, seed):
    """Draft rows whose k planted tokens carry most of the mass (logit ln(V) + U(-1, 3) over
    N(0, 1) noise), as a confident drafter's would; the workload's own rows are nearly flat."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(w.B, w.rows, w.V, generator=g)
    idx = torch.randint(0, w.V, (w.B, w.rows, w.k), generator=g)
    boost = math.log(w.V) - 1.0 + 4.0 * torch.rand(w.B, w.rows, w.k, generator=g)
    x.scatter_(2, idx, boost)
    return torch.log_softmax(x, dim=-1).contiguous()


def _tree(name):
    w = workloads.WORKLOADS[name]
    logp = _confident_rows(w, w.seed)
    roots = torch.randint(0, w.V, (w.B,), generator=torch.Generator().manual_seed(w.seed + 1)).to(torch.int32)
    lib()
    status = ts.new_status(dev())
    tree = ts.tree_build(logp.to(dev()), roots.to(dev()), w.k, w.depth, w.m, status=status)
    ts.check_status(status)
    return w, tree


def _check(tree, got, costs):
    h = {k: v.cpu().numpy() for k, v in tree.items() if k in ("tokens", "parents", "depth", "values", "node_row")}
    n = int(got["n"].item())
    _, _, rate = oracle.tree_prune(h["tokens"], h["parents"], h["depth"], h["values"], *costs)
    assert rate[n - 1] >= rate.max() * (1 - 1e-5), (n, int(np.argmax(rate)) + 1)
    _, ref, _ = oracle.tree_prune(h["tokens"], h["parents"], h["depth"], h["values"], *costs,
                                  node_row=h.get("node_row"), n=n)
    for key in ("tokens", "parents", "depth", "kept", "node_row"):
        np.testing.assert_array_equal(got[key].cpu().numpy(), ref[key], err_msg=key)
    np.testing.assert_array_equal(got["values"].cpu().numpy(), ref["values"])
    np.testing.assert_array_equal(got["mask"].cpu().numpy().view(np.uint64), ref["mask_words"])
    np.testing.assert_allclose(got["expected"].cpu().numpy(), ref["expected"], rtol=1e-5)
    return n


@pytest.mark.parametrize("costs", COSTS)
@pytest.mark.parametrize("name", ["llama2_7b", "llama3_8b_gqa", "llama2_70b_gqa", "long_context_m128",
                                  "long_context_m8"])
def test_workload_trees_match_the_oracle(name, costs):
    w, tree = _tree(name)
    status = ts.new_status(dev())
    got = ts.tree_prune(tree, *costs, status=status)
    ts.check_status(status)
    n = _check(tree, got, costs)
    assert 1 <= n <= w.m


def test_free_and_prohibitive_verification():
    w, tree = _tree("llama2_70b_gqa")
    got = ts.tree_prune(tree, 1.0, 1.0, 0.0)
    assert int(got["n"].item()) == w.m
    for key in ("tokens", "parents", "depth", "node_row"):
        assert torch.equal(got[key], tree[key])
    assert torch.equal(got["mask"], tree["mask"])
    got = ts.tree_prune(tree, 0.0, 0.0, 1e6)
    assert int(got["n"].item()) == 1
    assert (got["parents"].cpu() == -1).all() and (got["kept"].cpu() == 0).all()


def test_pruned_mask_drives_the_verify_kernels():
    """The pruned tree is a valid input of tree_accept: the greedy walk over it equals the oracle
    walk on the pruned tokens and parents."""
    w, tree = _tree("llama2_7b")
    got = ts.tree_prune(tree, 1.0, 10.0, 0.05)
    n = int(got["n"].item())
    g = torch.Generator().manual_seed(3)
    logits = torch.randn(w.B, n, w.V, generator=g).to(torch.bfloat16)
    acc = ts.tree_accept(logits.to(dev()), got["tokens"].contiguous(), got["parents"].contiguous())
    ref = oracle.accept_longest_path(got["tokens"].cpu().numpy(), got["parents"].cpu().numpy(),
                                     oracle.target_argmax(logits))
    np.testing.assert_array_equal(acc["accept_len"].cpu().numpy(), ref[0])
    np.testing.assert_array_equal(acc["bonus"].cpu().numpy(), ref[2])


def test_bad_and_broken_trees_are_reported():
    w, tree = _tree("llama2_70b_gqa")
    t = {k: v.clone() for k, v in tree.items()}
    t["parents"][0, 5] = 7                               # a parent after its child
    status = ts.new_status(dev())
    got = ts.tree_prune(t, 1.0, 10.0, 0.05, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -6
    assert (got["tokens"][0].cpu() == -1).all() and float(got["expected"][0]) == 0.0
    assert (got["tokens"][1].cpu() >= 0).all()
    # root -> a (-0.1) -> b (+0.5), root -> c (-0.2): b ranks first, and with t_node alone the
    # best count is 2, which keeps b without its parent
    small = dict(tokens=torch.tensor([[5, 6, 7, 8]], dtype=torch.int32),
                 parents=torch.tensor([[-1, 0, 1, 0]], dtype=torch.int32),
                 depth=torch.tensor([[0, 1, 2, 1]], dtype=torch.int32),
                 values=torch.tensor([[0.0, -0.1, 0.5, -0.2]], dtype=torch.float64))
    small = {k: v.to(dev()) for k, v in small.items()}
    status = ts.new_status(dev())
    got = ts.tree_prune(small, 0.0, 0.0, 1.0, status=status)
    torch.cuda.synchronize()
    assert int(got["n"].item()) == 2 and int(status.item()) == -6
    assert (got["tokens"].cpu() == -1).all()
