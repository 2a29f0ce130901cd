"""Pins of the oracle's EAGLE-2 tree construction (CPU only)."""
import json
import math
import os

import numpy as np
import pytest
import torch

import workloads
from oracle import row_topk, tree_build
from oracle.tree_build import tree_build_one

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def hand_case():
    with open(os.path.join(GOLDEN, "hand_build_case.json")) as f:
        g = json.load(f)
    V, ids = g["vocab"], g["token_ids"]
    rows = []
    for r in g["rows"]:
        p = np.zeros(V, dtype=np.float64)
        top = {ids[w]: pr for w, pr in r["top"]}
        rest = (1.0 - sum(top.values())) / (V - len(top))
        p[:] = rest
        for t, pr in top.items():
            p[t] = pr
        rows.append(np.log(p).astype(np.float32))
    return g, np.stack(rows)


def test_hand_case_reproduces_page_tree():
    """Expand top-2, rerank top-8 must give [It,is,has,a,the,to,good,be] (rainlin.net, 7.1/7.2/四)."""
    g, logp = hand_case()
    ids = g["token_ids"]
    out = tree_build_one(logp, ids[g["root"]], g["k"], g["depth"], g["m"])
    exp = g["expected"]
    assert out["tokens"].tolist() == [ids[w] for w in exp["words"]]
    assert out["parents"].tolist() == exp["parents"]
    assert out["depth"].tolist() == exp["depth"]
    np.testing.assert_allclose(np.exp(out["values"]), exp["global_value"], rtol=1e-6)


def test_hand_case_expansion_prefers_global_value():
    """'the' (0.11) loses the layer-2 frontier to 'to' (0.175) although its own confidence
    0.2 is above... the frontier is chosen by the path product, not the local confidence."""
    g, logp = hand_case()
    ids = g["token_ids"]
    out = tree_build_one(logp, ids[g["root"]], 2, 3, 8)
    toks = out["tokens"].tolist()
    # 'be' is the child of 'to', so 'to' was expanded; 'the' has no child in the tree
    assert out["parents"][toks.index(ids["be"])] == toks.index(ids["to"])
    assert toks.index(ids["the"]) not in out["parents"].tolist()


def _check_invariants(out, logp, k, depth, m):
    tokens, parents, dep, vals, mask = (out[x] for x in ("tokens", "parents", "depth", "values", "mask"))
    assert parents[0] == -1 and dep[0] == 0 and vals[0] == 0.0
    for i in range(1, m):
        p = parents[i]
        assert 0 <= p < i                                  # parents precede children
        assert dep[i] == dep[p] + 1
        assert vals[i] <= vals[p]                          # value never grows down a path
        assert mask[i].sum() == dep[i] + 1 and mask[i, 0] and mask[i, i]
    for i in range(1, m):                                  # siblings carry distinct tokens
        sib = [j for j in range(1, m) if parents[j] == parents[i] and j != i]
        assert all(tokens[j] != tokens[i] for j in sib)
    # depth non-decreasing in flat order (flatten by depth)
    assert all(dep[i] <= dep[i + 1] for i in range(m - 1))


def test_product_rule_and_invariants_random():
    """exp(V) equals the product of the draft confidences on the root path (rainlin.net 7.1)."""
    for (k, depth, m, V, seed) in [(2, 3, 8, 50, 1), (3, 4, 20, 64, 2), (4, 5, 40, 128, 3), (1, 6, 7, 30, 4)]:
        rng = np.random.default_rng(seed)
        R = 1 + (depth - 1) * k
        logits = rng.normal(0, 2, size=(R, V))
        logp = (logits - np.log(np.exp(logits).sum(1, keepdims=True))).astype(np.float32)
        out = tree_build_one(logp, 0, k, depth, m)
        _check_invariants(out, logp, k, depth, m)
        # recompute the confidence product along each path from the draft rows directly
        # (brute force: find for every node the row and the token that produced it)
        for i in range(1, m):
            prod, node = 1.0, i
            while node != 0:
                prod *= math.exp(float(_lp_of(out, logp, node, k)))
                node = out["parents"][node]
            assert abs(math.exp(out["values"][i]) - prod) <= 1e-12 * prod


def _lp_of(out, logp, node, k):
    # the token's log-prob in the row its parent was expanded with: search all rows for the
    # token among that row's top-k (brute force, independent of the frontier bookkeeping)
    tok = out["tokens"][node]
    cands = [logp[r][tok] for r in range(logp.shape[0]) if tok in row_topk(logp[r], k)[0]]
    # all rows that could have produced it; the parent's path value pins which one
    target = out["values"][node] - out["values"][out["parents"][node]]
    best = min(cands, key=lambda x: abs(float(x) - target))
    assert abs(float(best) - target) < 1e-9
    return best


def test_brute_force_tiny_exhaustive_selection():
    """Brute force on tiny inputs: enumerate every candidate by explicit recursion over
    the frontier rule, then check the reranked set is the m-1 best by value."""
    rng = np.random.default_rng(11)
    k, depth, V = 2, 3, 12
    R = 1 + (depth - 1) * k
    for trial in range(20):
        logits = rng.normal(0, 2, size=(R, V))
        logp = (logits - np.log(np.exp(logits).sum(1, keepdims=True))).astype(np.float32)
        m = int(rng.integers(2, 11))
        out = tree_build_one(logp, 0, k, depth, m)
        # all candidate values by brute force
        vals = []
        l1 = np.argsort(-logp[0], kind="stable")[:k]
        layer = [(float(logp[0][t]), 1) for t in l1]
        vals += layer
        front = sorted(range(len(layer)), key=lambda x: -layer[x][0])[:k]
        prev = layer
        for l in range(2, depth + 1):
            cur = []
            for j, f in enumerate(front):
                row = logp[1 + (l - 2) * k + j]
                for t in np.argsort(-row, kind="stable")[:k]:
                    cur.append((prev[f][0] + float(row[t]), l))
            vals += cur
            front = sorted(range(len(cur)), key=lambda x: -cur[x][0])[:k]
            prev = cur
        best = sorted(vals, key=lambda x: (-x[0], x[1]))[: m - 1]
        assert sorted(np.round(out["values"][1:], 12).tolist()) == sorted(np.round([b[0] for b in best], 12).tolist())


def test_topk_ties_lower_id():
    row = np.array([0.0, -1.0, -0.5, -0.5, -0.0, -2.0], dtype=np.float32)
    ids, vals = row_topk(row, 4)
    assert ids.tolist() == [0, 4, 2, 3]


def test_chain_k1():
    rng = np.random.default_rng(3)
    R, V = 7, 20
    logits = rng.normal(0, 2, size=(R, V))
    logp = (logits - np.log(np.exp(logits).sum(1, keepdims=True))).astype(np.float32)
    out = tree_build_one(logp, 5, 1, 7, 8)
    assert out["parents"].tolist() == [-1, 0, 1, 2, 3, 4, 5, 6]
    assert out["tokens"][1:].tolist() == [int(np.argmax(logp[r])) for r in range(7)]


def test_m1_root_only():
    out = tree_build_one(np.zeros((1, 4), np.float32), 3, 2, 1, 1)
    assert out["tokens"].tolist() == [3] and out["parents"].tolist() == [-1]


def test_too_few_candidates():
    with pytest.raises(ValueError):
        tree_build_one(np.zeros((1, 4), np.float32), 3, 2, 1, 4)


def test_workload_batch_shapes():
    w = workloads.WORKLOADS["tiny"]
    inp = workloads.generate(w)
    out = tree_build(inp["draft_logp"].numpy(), inp["root_tokens"].numpy(), w.k, w.depth, w.m)
    assert out["tokens"].shape == (w.B, w.m) and out["mask_words"].shape == (w.B, w.m, 1)
    assert out["tokens"][0, 0] == int(inp["root_tokens"][0])


@pytest.mark.parametrize("k,depth,m", [(2, 3, 8), (3, 4, 20), (4, 5, 40), (1, 6, 7), (5, 3, 31)])
def test_node_row_names_the_row_that_drew_the_children(k, depth, m):
    """Each row's top-k lives in its own block of token ids (row r owns ids r*k .. r*k+k-1), so
    the row a node's children came from can be read off the children's tokens, with no
    frontier bookkeeping.  A node that was expanded carries that row; every other node -1."""
    R = 1 + (depth - 1) * k
    V = R * k + 16
    rng = np.random.default_rng(k * 100 + depth * 10 + m)
    logp = np.full((R, V), -30.0)
    for r in range(R):
        logp[r, r * k:(r + 1) * k] = np.log(rng.dirichlet(np.ones(k)) * 0.9)
    logp = logp.astype(np.float32)
    out = tree_build_one(logp, V - 1, k, depth, m)
    rows_seen = {}
    for i in range(1, m):
        rows_seen.setdefault(int(out["parents"][i]), set()).add(int(out["tokens"][i]) // k)
    expanded = 0
    for p in range(m):
        if p in rows_seen:
            assert rows_seen[p] == {int(out["node_row"][p])}
        if out["node_row"][p] >= 0:
            expanded += 1
            assert out["depth"][p] < depth
    # rows are distinct, the root uses row 0, and no more rows than were drawn
    rows = [int(r) for r in out["node_row"] if r >= 0]
    assert len(rows) == len(set(rows)) and out["node_row"][0] == 0 and expanded <= R


def test_node_row_root_only():
    out = tree_build_one(np.zeros((1, 4), np.float32), 3, 2, 1, 1)
    assert out["node_row"].tolist() == [-1]
