"""Pins of the oracle's cost-aware tree pruning (CPU only)."""
import itertools

import numpy as np
import pytest

import workloads
from oracle import ancestor_mask, tree_build
from oracle.tree_prune import expected_tokens, rerank_order, tree_prune


def _tree(seed, k=3, depth=4, m=20, V=40, sigma=1.5):
    rng = np.random.default_rng(seed)
    R = 1 + (depth - 1) * k
    x = rng.normal(0, sigma, size=(1, R, V))
    logp = (x - np.log(np.exp(x).sum(-1, keepdims=True))).astype(np.float32)
    return logp, tree_build(logp, np.array([0]), k, depth, m)


def test_expected_tokens_match_a_monte_carlo_walk():
    """Each node's token is emitted by the target with its draft probability (siblings
    exclusive): the mean accepted length plus one equals 1 + sum exp(V)."""
    logp, t = _tree(1, m=30)
    par, val, tok = t["parents"][0], t["values"][0], t["tokens"][0]
    m = len(par)
    kids = {u: [c for c in range(m) if par[c] == u] for u in range(m)}
    lp = {c: val[c] - (val[par[c]] if par[c] > 0 else 0.0) for c in range(1, m)}
    rng = np.random.default_rng(2)
    N, total = 40000, 0
    for _ in range(N):
        u, n = 0, 1
        while kids[u]:
            probs = [np.exp(lp[c]) for c in kids[u]]
            r = rng.random()
            acc = np.cumsum(probs)
            j = int(np.searchsorted(acc, r, side="right"))
            if j >= len(probs):
                break
            u, n = kids[u][j], n + 1
        total += n
    order = rerank_order(val, t["depth"][0])
    e = expected_tokens(val, order, m)
    sd = np.sqrt(m) / np.sqrt(N)                        # generous bound on the mean's std
    assert abs(total / N - e) < 5 * sd


def _connected_subsets(par, n):
    m = len(par)
    for comb in itertools.combinations(range(1, m), n - 1):
        s = set(comb) | {0}
        if all(par[c] in s for c in comb):
            yield s


@pytest.mark.parametrize("seed", [3, 4, 5])
def test_rerank_prefix_is_the_best_connected_subtree(seed):
    logp, t = _tree(seed, k=2, depth=4, m=12, V=20)
    par, val, dep = t["parents"][0], t["values"][0], t["depth"][0]
    order = rerank_order(val, dep)
    for n in range(1, 9):
        pre = set([0] + order[: n - 1])
        assert all(par[c] in pre for c in pre if c), "prefix not connected"
        best = max(sum(np.exp(val[c]) for c in s if c) for s in _connected_subsets(par, n))
        assert abs(expected_tokens(val, order, n) - 1.0 - best) < 1e-12


def test_free_and_prohibitive_verification():
    logp, t = _tree(6)
    args = (t["tokens"], t["parents"], t["depth"], t["values"])
    n, out, _ = tree_prune(*args, t_draft=1.0, t_fixed=1.0, t_node=0.0)
    assert n == t["tokens"].shape[1]
    np.testing.assert_array_equal(out["tokens"], t["tokens"])
    np.testing.assert_array_equal(out["mask_words"], t["mask_words"])
    n, out, _ = tree_prune(*args, t_draft=0.0, t_fixed=0.0, t_node=1e6)
    assert n == 1 and out["parents"].tolist() == [[-1]]


def test_rate_is_maximised_and_the_pruned_tree_is_a_subtree():
    w = workloads.WORKLOADS["llama2_70b_gqa"]
    inp = workloads.generate(w, with_attention=False, with_logits=False)
    t = tree_build(inp["draft_logp"].numpy(), inp["root_tokens"].numpy(), w.k, w.depth, w.m)
    n, out, rate = tree_prune(t["tokens"], t["parents"], t["depth"], t["values"], 50.0, 30.0, 0.05,
                              node_row=t["node_row"])
    assert 1 < n < w.m and rate[n - 1] == rate.max() and (rate[: n - 1] < rate[n - 1]).all()
    for b in range(w.B):
        kept = out["kept"][b]
        assert kept[0] == 0 and (np.diff(kept) > 0).all()
        for j in range(1, n):                            # parents map to the kept parent
            assert kept[out["parents"][b, j]] == t["parents"][b, kept[j]]
        np.testing.assert_array_equal(out["tokens"][b], t["tokens"][b, kept])
        np.testing.assert_array_equal(out["node_row"][b], t["node_row"][b, kept])
        mk = ancestor_mask(out["parents"][b])
        assert (mk.sum(1) == out["depth"][b] + 1).all()
        assert abs(out["expected"][b] - 1.0 - np.exp(out["values"][b][1:]).sum()) < 1e-12
