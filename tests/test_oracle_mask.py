"""Pins of the oracle's ancestor mask against what the pages fix (CPU only)."""
import json
import os

import numpy as np

from oracle import ancestor_mask, mask_to_words, words_to_mask

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_worked_example_printed_row():
    """'good' sees exactly [It, is, a, good] (rainlin.net/posts/eagle, section 四)."""
    g = _load("worked_tree.json")
    words, parents = g["words"], g["parents"]
    mask = ancestor_mask(parents)
    row = words.index(g["printed_row"]["query"])
    seen = [words[j] for j in range(len(words)) if mask[row, j]]
    assert seen == g["printed_row"]["sees"]


def test_worked_example_all_rows_bit_exact():
    g = _load("worked_tree.json")
    words = mask_to_words(ancestor_mask(g["parents"]))
    assert [int(w[0]) for w in words] == [int(x, 16) for x in g["mask_words_from_rule"]]


def test_siblings_invisible():
    """'a' and 'the' are siblings: neither sees the other (same section)."""
    g = _load("worked_tree.json")
    w = g["words"]
    mask = ancestor_mask(g["parents"])
    a, the = w.index("a"), w.index("the")
    assert not mask[a, the] and not mask[the, a]


def _random_tree(rng, m):
    return [-1] + [int(rng.integers(0, i)) for i in range(1, m)]


def test_recurrence_matches_parent_walk():
    """Independent construction: mask[i] = mask[parent[i]] | {i}, parents first."""
    rng = np.random.default_rng(5)
    for m in (1, 2, 7, 63, 64, 65, 130, 256):
        for _ in range(3):
            par = _random_tree(rng, m)
            rec = np.zeros((m, m), dtype=bool)
            for i in range(m):
                if par[i] >= 0:
                    rec[i] = rec[par[i]]
                rec[i, i] = True
            assert np.array_equal(rec, ancestor_mask(par))
            assert np.array_equal(words_to_mask(mask_to_words(rec), m), rec)


def test_chain_is_causal():
    """A chain tree gives the ordinary causal mask M[i, j] = 1 for j <= i (lesty.tech, section 5)."""
    m = 9
    mask = ancestor_mask([-1] + list(range(m - 1)))
    assert np.array_equal(mask, np.tril(np.ones((m, m), dtype=bool)))


def test_popcount_is_depth_plus_one():
    rng = np.random.default_rng(7)
    par = _random_tree(rng, 40)
    mask = ancestor_mask(par)
    for i in range(40):
        d, n = 0, i
        while par[n] != -1:
            n, d = par[n], d + 1
        assert mask[i].sum() == d + 1 and mask[i, 0] and mask[i, i]


def test_rejects_cycles():
    import pytest
    with pytest.raises(ValueError):
        ancestor_mask([-1, 2, 1])
