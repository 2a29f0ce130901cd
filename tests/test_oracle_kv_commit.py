"""Pins of the KV-commit oracle ("lesty.tech — EAGLE-2 vs. Medusa", section 8).

Each check reaches the expected result by a route other than the oracle's own per-row
address arithmetic: hand-written expected rows for the page's example, a gather of the
whole logical sequence through the old and the new block table, page conservation, and
attention over the committed cache against attention over a freshly written one.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _cache(num_blocks, Hkv, bs, d):
    """Every element of a row holds a code of (page, head, slot) so rows are distinguishable."""
    k = np.zeros((num_blocks, Hkv, bs, d))
    for p in range(num_blocks):
        for h in range(Hkv):
            for s in range(bs):
                k[p, h, s, :] = 1000.0 * p + 100.0 * h + s + np.arange(d) / 1000.0
    return k, -k


def _logical_rows(cache, table_row, n, bs):
    """The first n logical rows of one sequence, gathered page by page (all heads)."""
    rows = []
    for page_idx in range(-(-n // bs)):
        page = int(table_row[page_idx])
        for s in range(bs):
            if len(rows) < n:
                rows.append(cache[page, :, s, :].copy())
    return rows


def test_page_example_keeps_x1_x2_x4():
    """The page's example: surviving nodes {x1, x2, x4}, rejected {x3, x5} (plus x6, x7 so
    that a whole page is released).  Node i sits at logical position L + i."""
    bs, Hkv, d, L, m = 4, 2, 3, 10, 8
    table = np.array([[7, 2, 5, 0, 3, 1]])          # logical page -> physical page
    k, v = _cache(8, Hkv, bs, d)
    path = np.array([[0, 1, 2, 4, -1, -1, -1, -1]])
    k2, v2, t2, plen, freed, nfreed, bad = oracle.kv_commit(k, v, table, np.array([L]), path,
                                                            np.array([4]), m, bs)
    assert not bad[0] and int(plen[0]) == 14
    # positions 10..17 were pages 2 (10, 11) and 3 (12..15) and 4 (16, 17); after the commit
    # positions 10, 11, 12, 13 hold the rows of nodes 0, 1, 2, 4 = old positions 10, 11, 12, 14
    expect = {10: (5, 2), 11: (5, 3), 12: (0, 0), 13: (0, 2)}   # new position -> old (page, slot)
    for pos, (op, os_) in expect.items():
        page, slot = int(t2[0, pos // bs]), pos % bs
        np.testing.assert_array_equal(k2[page, :, slot, :], k[op, :, os_, :])
        np.testing.assert_array_equal(v2[page, :, slot, :], v[op, :, os_, :])
    # ceil(14 / 4) = 4 pages kept, ceil(18 / 4) = 5 were used: logical page 4 (physical 3) freed
    assert int(nfreed[0]) == 1 and int(freed[0, 0]) == 3 and int(t2[0, 4]) == -1
    assert list(t2[0, :4]) == [7, 2, 5, 0] and int(t2[0, 5]) == 1  # untouched beyond the tree


def _random_case(rng, B=3, Hkv=2, d=4, bs=4, m=9):
    L = rng.integers(0, 20, size=B)
    need = [-(-(int(l) + m) // bs) for l in L]
    max_blocks = max(need) + 1
    num_blocks = sum(need) + 2
    perm = rng.permutation(num_blocks)
    table = np.full((B, max_blocks), -1)
    o = 0
    for b in range(B):
        table[b, :need[b]] = perm[o:o + need[b]]
        o += need[b]
    k, v = _cache(num_blocks, Hkv, bs, d)
    a = rng.integers(1, m + 1, size=B)
    path = np.full((B, m), -1)
    for b in range(B):
        rest = np.sort(rng.choice(np.arange(1, m), size=int(a[b]) - 1, replace=False))
        path[b, :a[b]] = np.concatenate([[0], rest])
    return k, v, table, L, path, a, m, bs


@pytest.mark.parametrize("seed", range(6))
def test_committed_sequence_is_prefix_then_accepted_nodes(seed):
    rng = np.random.default_rng(seed)
    k, v, table, L, path, a, m, bs = _random_case(rng)
    k2, v2, t2, plen, freed, nfreed, bad = oracle.kv_commit(k, v, table, L, path, a, m, bs)
    assert not bad.any()
    for b in range(len(L)):
        before_k = _logical_rows(k, table[b], int(L[b]) + m, bs)
        before_v = _logical_rows(v, table[b], int(L[b]) + m, bs)
        after_k = _logical_rows(k2, t2[b], int(plen[b]), bs)
        after_v = _logical_rows(v2, t2[b], int(plen[b]), bs)
        want = list(range(int(L[b]))) + [int(L[b]) + int(p) for p in path[b, :a[b]]]
        assert int(plen[b]) == len(want)
        for j, src in enumerate(want):
            np.testing.assert_array_equal(after_k[j], before_k[src])
            np.testing.assert_array_equal(after_v[j], before_v[src])
        # pages: kept + freed = previously used, nothing listed twice
        used = [int(x) for x in table[b, :-(-(int(L[b]) + m) // bs)]]
        kept = [int(x) for x in t2[b] if x >= 0 and int(x) in used]
        fl = [int(x) for x in freed[b, :nfreed[b]]]
        assert sorted(kept + fl) == sorted(used) and len(set(fl)) == len(fl)
        assert all(x == -1 for x in freed[b, nfreed[b]:])


def test_chain_acceptance_moves_nothing():
    rng = np.random.default_rng(11)
    k, v, table, L, path, a, m, bs = _random_case(rng)
    a = np.full_like(a, m)
    path = np.tile(np.arange(m), (len(L), 1))
    k2, v2, t2, plen, freed, nfreed, bad = oracle.kv_commit(k, v, table, L, path, a, m, bs)
    np.testing.assert_array_equal(k2, k)
    np.testing.assert_array_equal(v2, v)
    assert list(plen) == [int(x) + m for x in L] and not nfreed.any()


@pytest.mark.parametrize("case", ["len0", "len_over_m", "not_root", "not_increasing", "bad_page"])
def test_contract_breaks_leave_the_sequence_untouched(case):
    rng = np.random.default_rng(3)
    k, v, table, L, path, a, m, bs = _random_case(rng, B=2)
    if case == "len0":
        a[0] = 0
    elif case == "len_over_m":
        a[0] = m + 1
    elif case == "not_root":
        a[0] = 3
        path[0, :3] = [1, 2, 3]
    elif case == "not_increasing":
        a[0] = 3
        path[0, :3] = [0, 4, 2]
    else:
        table[0, int(L[0]) // bs] = k.shape[0] + 7
    k2, v2, t2, plen, freed, nfreed, bad = oracle.kv_commit(k, v, table, L, path, a, m, bs)
    assert bad[0] and not bad[1]
    assert int(plen[0]) == int(L[0]) and (t2[0] == table[0]).all() and nfreed[0] == 0


def test_attention_after_commit_equals_attention_over_a_fresh_cache():
    """The next step's root attends to the committed prefix: through the committed cache it
    must see exactly what a cache written token by token with the accepted rows holds."""
    rng = np.random.default_rng(5)
    Hkv, Hq, d, bs, m = 2, 4, 8, 4, 7
    k, v, table, L, path, a, _, _ = _random_case(rng, B=2, Hkv=Hkv, d=d, bs=bs, m=m)
    k = rng.standard_normal(k.shape)
    v = rng.standard_normal(v.shape)
    k2, v2, t2, plen, freed, nfreed, bad = oracle.kv_commit(k, v, table, L, path, a, m, bs)
    B = len(L)
    # fresh cache: prefix rows, then the accepted nodes' rows, written contiguously
    n_new = [int(plen[b]) + 1 for b in range(B)]             # + the next root's own row
    pages = [-(-n // bs) for n in n_new]
    fk = np.zeros((sum(pages), Hkv, bs, d))
    fv = np.zeros_like(fk)
    ftab = np.full((B, max(pages)), -1)
    q = rng.standard_normal((B, 1, Hq, d))
    root_k = rng.standard_normal((B, Hkv, d))
    root_v = rng.standard_normal((B, Hkv, d))
    o = 0
    for b in range(B):
        ftab[b, :pages[b]] = np.arange(o, o + pages[b])
        o += pages[b]
        rows_k = _logical_rows(k, table[b], int(L[b]) + m, bs)
        rows_v = _logical_rows(v, table[b], int(L[b]) + m, bs)
        want = list(range(int(L[b]))) + [int(L[b]) + int(p) for p in path[b, :a[b]]]
        for j, src in enumerate(want + [None]):
            page, slot = int(ftab[b, j // bs]), j % bs
            fk[page, :, slot, :] = rows_k[src] if src is not None else root_k[b]
            fv[page, :, slot, :] = rows_v[src] if src is not None else root_v[b]
    # the committed cache gets the next root's row at its new position (a page past the end
    # may have been freed: give it one)
    ck, cv, ctab = k2.copy(), v2.copy(), t2.copy()
    spare = list(range(k.shape[0], k.shape[0] + B))
    ck = np.concatenate([ck, np.zeros((B, Hkv, bs, d))])
    cv = np.concatenate([cv, np.zeros((B, Hkv, bs, d))])
    for b in range(B):
        pos = int(plen[b])
        if ctab[b, pos // bs] < 0:
            ctab[b, pos // bs] = spare[b]
        ck[int(ctab[b, pos // bs]), :, pos % bs, :] = root_k[b]
        cv[int(ctab[b, pos // bs]), :, pos % bs, :] = root_v[b]
    mask = np.ones((B, 1, 1), dtype=bool)
    scale = 1.0 / math.sqrt(d)
    out_c, lse_c = oracle.tree_attention(torch.from_numpy(q), torch.from_numpy(ck), torch.from_numpy(cv), ctab,
                                         np.array(plen), mask, scale)
    out_f, lse_f = oracle.tree_attention(torch.from_numpy(q), torch.from_numpy(fk), torch.from_numpy(fv), ftab,
                                         np.array(plen), mask, scale)
    np.testing.assert_array_equal(out_c, out_f)
    np.testing.assert_array_equal(lse_c, lse_f)
