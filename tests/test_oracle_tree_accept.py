"""Pins of the oracle's acceptance (CPU only)."""
import itertools
import json
import os

import numpy as np
import torch

from oracle import accept_longest_path, target_argmax
from oracle.tree_accept import accept_one

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _greedy_walk(tokens, parents, amax):
    """Sequential verification: from the root, descend to the child whose token is the
    target's argmax at the current node, one level at a time (distinct sibling tokens)."""
    cur, path = 0, [0]
    while True:
        nxt = [c for c in range(len(tokens)) if parents[c] == cur and tokens[c] == amax[cur]]
        if not nxt:
            break
        assert len(nxt) == 1
        cur = nxt[0]
        path.append(cur)
    return len(path), path, amax[cur]


def test_hand_planted_worked_tree():
    """Target agrees with 'is' after 'It', 'a' after 'is', 'good' after 'a' ->
    accept [It, is, a, good] and the bonus token predicted after 'good'."""
    with open(os.path.join(GOLDEN, "worked_tree.json")) as f:
        g = json.load(f)
    words, parents = g["words"], g["parents"]
    tok = {w: 100 + i for i, w in enumerate(words)}
    tokens = [tok[w] for w in words]
    amax = [7] * 8
    amax[words.index("It")] = tok["is"]
    amax[words.index("is")] = tok["a"]
    amax[words.index("a")] = tok["good"]
    amax[words.index("good")] = 4242
    n, path, bonus = accept_one(tokens, parents, amax)
    assert n == 4 and path[:4] == [0, 1, 3, 6] and path[4:] == [-1] * 4 and bonus == 4242


def test_nothing_accepted():
    n, path, bonus = accept_one([5, 6, 7], [-1, 0, 0], [9, 1, 2])
    assert n == 1 and path == [0, -1, -1] and bonus == 9


def test_brute_force_all_trees_m_le_6():
    """Every parent array with parents before children, m <= 6, random tokens from a small
    alphabet with distinct siblings: the definition == the sequential greedy walk."""
    rng = np.random.default_rng(0)
    for m in range(1, 7):
        for par in itertools.product(*[range(i) for i in range(1, m)]):
            parents = [-1] + list(par)
            for _ in range(3):
                tokens = [int(rng.integers(0, 50))]
                for c in range(1, m):
                    used = {tokens[s] for s in range(1, c) if parents[s] == parents[c]}
                    t = int(rng.integers(0, 8))
                    while t in used:
                        t = (t + 1) % 8
                    tokens.append(t)
                amax = [int(rng.integers(0, 8)) for _ in range(m)]
                n, path, bonus = accept_one(tokens, parents, amax)
                gn, gpath, gbonus = _greedy_walk(tokens, parents, amax)
                assert n == gn and path[:n] == gpath and bonus == gbonus


def test_duplicate_siblings_longest_wins():
    """Reading for user trees with equal sibling tokens: the longest matching path wins,
    equal lengths -> lowest flat index of the end node."""
    tokens = [0, 5, 5, 6]
    parents = [-1, 0, 0, 2]
    amax = [5, 9, 6, 1]
    n, path, bonus = accept_one(tokens, parents, amax)
    assert n == 3 and path[:3] == [0, 2, 3] and bonus == 1
    n, path, _ = accept_one([0, 5, 5], [-1, 0, 0], [5, 1, 1])
    assert n == 2 and path[:2] == [0, 1]


def test_argmax_lowest_index_on_ties_and_bf16_exact():
    x = torch.tensor([[[1.0, 3.0, 3.0, 2.0], [-1.0, -1.0, -2.0, -1.0]]])
    assert target_argmax(x).tolist() == [[1, 0]]
    xb = torch.tensor([[[1.0, 1.00390625, 1.0078125]]], dtype=torch.bfloat16)  # adjacent bf16 values
    assert target_argmax(xb).tolist() == [[2]]


def test_batched_shapes():
    lens, paths, bonus = accept_longest_path(np.array([[1, 2], [3, 4]]), np.array([[-1, 0], [-1, 0]]),
                                             np.array([[2, 0], [0, 0]]))
    assert lens.tolist() == [2, 1] and paths.tolist() == [[0, 1], [0, -1]] and bonus.tolist() == [0, 0]


def test_argmax_ignoring_nan_hand_cases():
    """NaN is never the argmax, -inf is an ordinary value, a row of NaN only gives -1."""
    from oracle import target_argmax_ignoring_nan
    nan, inf = float("nan"), float("inf")
    rows = [[nan, 1.0, 3.0, 3.0], [nan, -inf, -inf, nan], [nan, nan, nan, nan], [3.0, nan, 3.0, 2.0],
            [-inf, nan, 5.0, nan], [-0.0, 0.0, nan, -1.0]]
    got = target_argmax_ignoring_nan(np.array([rows]))
    assert got.tolist() == [[2, 1, -1, 0, 2, 0]]


def test_argmax_ignoring_nan_equals_a_sort_over_the_kept_entries():
    """Random rows with NaNs sprinkled: the answer is the first entry of the kept (value,
    index) pairs sorted by value descending, index ascending; without NaN it is np.argmax."""
    from oracle import target_argmax_ignoring_nan
    rng = np.random.default_rng(5)
    x = np.round(rng.normal(size=(3, 40, 23)) * 2)
    x[rng.random(x.shape) < 0.3] = np.nan
    x[0, 0] = np.nan
    got = target_argmax_ignoring_nan(x)
    for b in range(3):
        for i in range(40):
            kept = sorted((-v, j) for j, v in enumerate(x[b, i]) if not np.isnan(v))
            assert got[b, i] == (kept[0][1] if kept else -1)
    clean = np.round(rng.normal(size=(2, 7, 50)))
    assert np.array_equal(target_argmax_ignoring_nan(clean), target_argmax(clean))
