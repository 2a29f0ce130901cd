"""Oracle: greedy acceptance over the verified tree.

Sources (web pages, by title and section):

* "lesty.tech — EAGLE-2 vs. Medusa", section 4 (greedy case): a draft token is accepted
  iff it equals the base model's argmax given everything before it — for a tree node,
  the argmax of the target distribution computed at its parent's position (the parent's
  root path being its context).  The printed formula is cut off; this is the reading.
* "rainlin.net/posts/eagle", section 3.2 (Verification) and section 四: one tree pass
  verifies all paths; the longest valid branch is accepted.

Definitions:

* ``target_argmax``: per (b, node) the vocabulary index of the largest logit; equal
  values -> lowest index (numpy's argmax returns the first maximum).  Values are compared
  exactly as given (bf16 logits are widened without rounding).
* ``target_argmax_ignoring_nan``: the same over the values that are not NaN (the pages'
  logits are finite; this fixes what a NaN row entry does: it is never the argmax, -inf
  counts as a value, and a row with nothing but NaN gives -1).
* ``accept_longest_path``: a node is *valid* if every non-root node on its root path
  carries the token equal to the target argmax at its parent.  The accepted node is the
  valid node of greatest depth (ties -> lowest flat index).  ``accept_len`` = its depth
  + 1 (the root counts), ``accept_path`` = root..node (padded with -1), ``bonus`` = the
  target argmax at the accepted node (the extra token every verify step yields).

Pins (tests/test_oracle_tree_accept.py): the hand-planted case on the page's worked
tree, and brute force over every tree with m <= 6 against the sequential greedy walk
(descend to the child whose token matches, one level at a time).
"""
from __future__ import annotations

import numpy as np


def target_argmax(logits) -> np.ndarray:
    """[B, m, V] -> int64 [B, m]: first index of the row maximum."""
    if hasattr(logits, "detach"):
        import torch
        logits = logits.detach().to(torch.float32).cpu().numpy()
    return np.argmax(np.asarray(logits), axis=-1).astype(np.int64)


def target_argmax_ignoring_nan(logits) -> np.ndarray:
    """[B, m, V] -> int64 [B, m]: first index of the largest value that is not NaN; -1 for a
    row of NaN only.  Written as an explicit loop over the rows."""
    if hasattr(logits, "detach"):
        import torch
        logits = logits.detach().to(torch.float32).cpu().numpy()
    x = np.asarray(logits)
    B, m, V = x.shape
    out = np.full((B, m), -1, dtype=np.int64)
    for b in range(B):
        for i in range(m):
            row = x[b, i]
            keep = np.nonzero(~np.isnan(row))[0]
            if len(keep) == 0:
                continue
            best = row[keep].max()
            out[b, i] = int(keep[row[keep] == best][0])
    return out


def accept_one(tokens, parents, amax):
    tokens = [int(t) for t in tokens]
    parents = [int(p) for p in parents]
    amax = [int(a) for a in amax]
    m = len(tokens)
    best, best_depth = 0, 0
    for n in range(m):
        node, depth, ok = n, 0, True
        while node != 0:
            par = parents[node]
            if not (0 <= par < node):
                raise ValueError("parents must precede children")
            if tokens[node] != amax[par]:
                ok = False
                break
            node, depth = par, depth + 1
        if ok and depth > best_depth:
            best, best_depth = n, depth
    path = []
    node = best
    while node != -1:
        path.append(node)
        node = parents[node] if node != 0 else -1
    path.reverse()
    return len(path), path + [-1] * (m - len(path)), amax[best]


def accept_longest_path(tokens, parents, amax):
    """Batched: returns (accept_len [B], accept_path [B, m], bonus [B]) as int64 arrays."""
    tokens = np.asarray(tokens)
    parents = np.asarray(parents)
    amax = np.asarray(amax)
    B, m = tokens.shape
    lens = np.zeros(B, dtype=np.int64)
    paths = np.zeros((B, m), dtype=np.int64)
    bonus = np.zeros(B, dtype=np.int64)
    for b in range(B):
        lens[b], p, bonus[b] = accept_one(tokens[b], parents[b], amax[b])
        paths[b] = p
    return lens, paths, bonus
