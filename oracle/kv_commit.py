"""Oracle: commit the accepted path's K/V after a verify step (TEST INFRASTRUCTURE ONLY).

Source (web page, by title and section):

* "lesty.tech — EAGLE-2 vs. Medusa", section 8 (KV cache management and speculative
  rollback): the tree's K/V are written into reserved scratch pages of the paged cache
  during the verify pass; afterwards only the nodes of the accepted path are kept, the
  block table is updated to commit them, and the pages of the rejected nodes go back to
  the free pool.

Reading (the page describes pointer updates only, which is exact when every tree node owns
a page; with multi-token pages the accepted rows must also be compacted): tree node i of
sequence b lives at logical position ``L_b + i`` of the paged sequence (the layout
``tree_attention`` reads).  Committing ``accept_path[b, 0..a-1]`` (``a = accept_len[b]``,
root first) moves the K/V rows at logical positions ``L_b + accept_path[b, j]`` to
``L_b + j`` for every KV head, reading every source before writing any destination, sets
the prefix length to ``L_b + a``, and releases the pages that covered positions
``[L_b + a, L_b + m)`` but no committed position: logical pages
``ceil((L_b + a) / bs) .. ceil((L_b + m) / bs) - 1``.  Their physical ids are listed in
``freed_blocks[b]`` (in logical-page order, -1 padded, ``freed_count[b]`` of them) and their
block-table entries become -1.  A sequence whose inputs break the contract (accept length
outside 1..m, a path that does not start at the root or does not increase, a page id out of
range) is left untouched and reported.

Pins (tests/test_oracle_kv_commit.py): the page's own example (accepted nodes
{x1, x2, x4}, rejected {x3, x5}); the committed logical sequence equals the prefix followed
by the accepted nodes' rows, read through the old and the new block table (checked by an
independent gather); a chain acceptance moves nothing; conservation of pages (kept + freed
= previously used, no page listed twice); and, end to end, attention of the next root over
the committed cache equals attention over a freshly written cache holding the same tokens.
"""
from __future__ import annotations

import numpy as np


def _phys(table_row, pos, bs):
    """(physical page, slot) of logical position ``pos`` through one block-table row."""
    return int(table_row[pos // bs]), pos % bs


def kv_commit(k_cache, v_cache, block_table, prefix_len, accept_path, accept_len, m, block_size):
    """Returns (k_cache, v_cache, block_table, prefix_len, freed_blocks, freed_count, bad).

    All inputs are left unchanged; the outputs are new arrays.  ``k_cache``/``v_cache`` are
    ``[num_blocks, Hkv, block_size, d]``; ``block_table`` ``[B, max_blocks]`` int;
    ``prefix_len`` ``[B]``; ``accept_path`` ``[B, m]`` (-1 padded); ``accept_len`` ``[B]``.
    ``bad[b]`` is True for a sequence that was left untouched because its inputs break the
    contract.
    """
    k = np.array(k_cache, copy=True)
    v = np.array(v_cache, copy=True)
    table = np.array(block_table, copy=True)
    plen = np.array(prefix_len, copy=True)
    B, max_blocks = table.shape
    num_blocks = k.shape[0]
    bs = int(block_size)
    freed = np.full((B, max_blocks), -1, dtype=np.int64)
    nfreed = np.zeros(B, dtype=np.int64)
    bad = np.zeros(B, dtype=bool)
    for b in range(B):
        L = int(plen[b])
        a = int(accept_len[b])
        path = [int(x) for x in accept_path[b][:max(a, 0)]]
        n_used = -(-(L + m) // bs)
        n_keep = -(-(L + a) // bs) if a >= 1 else 0
        ok = L >= 0 and 1 <= a <= m and path[0] == 0 and n_used <= max_blocks
        ok = ok and all(path[j] < path[j + 1] for j in range(a - 1)) and path[-1] < m
        if ok:
            pages_touched = set(range(L // bs, n_used))
            ok = all(0 <= int(table[b, i]) < num_blocks for i in pages_touched)
        if not ok:
            bad[b] = True
            continue
        row = table[b].copy()
        # every source row first, then every destination
        src_k = [k[_phys(row, L + p, bs)[0], :, _phys(row, L + p, bs)[1], :].copy() for p in path]
        src_v = [v[_phys(row, L + p, bs)[0], :, _phys(row, L + p, bs)[1], :].copy() for p in path]
        for j in range(a):
            page, slot = _phys(row, L + j, bs)
            k[page, :, slot, :] = src_k[j]
            v[page, :, slot, :] = src_v[j]
        for idx, i in enumerate(range(n_keep, n_used)):
            freed[b, idx] = table[b, i]
            table[b, i] = -1
        nfreed[b] = max(0, n_used - n_keep)
        plen[b] = L + a
    return k, v, table, plen, freed, nfreed, bad
