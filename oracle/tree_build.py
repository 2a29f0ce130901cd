"""Oracle: EAGLE-2 dynamic draft-tree construction and the tree-attention mask (fp64).

Sources (web pages, by title and section):

* "rainlin.net/posts/eagle" (大模型投机解码（二）：EAGLE 系列), section 7.1 (扩展阶段,
  Expansion): from the current deepest layer, the top-k nodes by *global acceptance
  value* are expanded by the draft model; the global value of a node is the product of
  the draft confidences of the tokens on its root path.  The confidence is the draft
  model's softmax probability (section 六, calibration paragraph).  Here the product is
  kept as a sum of log-probabilities: V(node) = sum of log p over the root path.
* same page, section 7.2 (重排阶段, Reranking): from *all* nodes take the top-m by value,
  shallow nodes preferred, so the selection stays a connected tree; then flatten to a
  1-D sequence and build the tree-attention mask.
* same page, section 四 (树状草稿 / Tree Attention): each token sees exactly its
  root-to-node ancestors (itself included); worked example [It, is, has, a, the, to,
  good, be] where "good" sees [It, is, a, good].
* "lesty.tech — EAGLE-2 vs. Medusa", section 5 (Tree-Attention Mask Fusion): the mask
  is built by walking parent pointers from each node up to the root.

Readings where the pages are silent (each listed in the design notes):

* every expanded node gets k children (the same k as the frontier width);
* the draft model is replaced by pre-drawn rows: frontier slot j of layer l-1 is expanded
  with draft row ``1 + (l-2)*k + j``; the root uses row 0;
* within a row, top-k is by value descending, equal values -> lower token id;
* frontier selection ties -> lower layer-local candidate index (``slot*k + child rank``);
* rerank order: value descending, then shallower depth, then layer-local index;
* flatten order: root first, then by (depth, parent's flat index, child rank), which
  reproduces the page's worked sequence;
* the root is node 0 with value 0 and is always kept; ``m`` counts the root.
* ``node_row`` names, per flattened node, the draft row its children were drawn from
  (root: row 0; an expanded frontier node of layer l in slot j: ``1 + (l-1)*k + j``; -1
  for a node that was never expanded).  Stochastic verification needs it: the draft
  distribution q at a node is that row.

Pins (tests/test_oracle_tree_build.py, tests/test_oracle_mask.py): the page's worked
mask row, a hand-built case that must reproduce the page's tree and order, the product
rule exp(V) = prod(confidences), ancestor closure, monotone values, parents before
children, popcount(mask row) = depth + 1, and the mask recurrence
mask[i] = mask[parent[i]] | bit(i) as an independent construction.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List

import numpy as np


def row_topk(logp_row: np.ndarray, k: int):
    """Top-k (token ids, values) of one draft row: value descending, ties -> lower id."""
    vals = np.asarray(logp_row)
    order = np.argsort(-vals, kind="stable")  # stable: equal values keep ascending ids
    ids = order[:k]
    return ids.astype(np.int64), vals[ids]


@dataclass
class _Cand:
    layer: int     # depth below the root (1..depth)
    idx: int       # layer-local index: child rank for layer 1, slot*k + rank afterwards
    token: int
    parent: int    # candidate id of the parent, -1 for the root
    rank: int      # rank among the parent's k children
    value: float   # V = V(parent) + log p, fp64, accumulated root -> leaf
    slot: int = -1  # position in its layer's frontier (expanded), -1 if never expanded


def _expand(logp: np.ndarray, k: int, depth: int) -> List[_Cand]:
    """Section 7.1: grow the candidate tree layer by layer from the deepest frontier."""
    topk = [row_topk(logp[r], k) for r in range(logp.shape[0])]
    cands: List[_Cand] = []
    ids, lps = topk[0]
    layer = []
    for c in range(k):
        cands.append(_Cand(1, c, int(ids[c]), -1, c, 0.0 + float(lps[c])))
        layer.append(len(cands) - 1)
    frontier = sorted(layer, key=lambda x: (-cands[x].value, cands[x].idx))[:k]
    for l in range(2, depth + 1):
        for j, par in enumerate(frontier):
            cands[par].slot = j
        layer = []
        for j, par in enumerate(frontier):
            ids, lps = topk[1 + (l - 2) * k + j]
            for c in range(k):
                cands.append(_Cand(l, j * k + c, int(ids[c]), par, c,
                                   cands[par].value + float(lps[c])))
                layer.append(len(cands) - 1)
        frontier = sorted(layer, key=lambda x: (-cands[x].value, cands[x].idx))[:k]
    return cands


def ancestor_mask(parents) -> np.ndarray:
    """Boolean [m, m]: entry (i, j) is True iff j is i itself or one of its ancestors.

    Built by walking parent pointers from i to the root ("lesty.tech", section 5).
    Raises on a parent index out of range or a cycle.
    """
    par = [int(p) for p in parents]
    m = len(par)
    mask = np.zeros((m, m), dtype=bool)
    for i in range(m):
        node, steps = i, 0
        while node != -1:
            if not (0 <= node < m) or steps > m:
                raise ValueError("invalid parent array")
            mask[i, node] = True
            node = par[node]
            steps += 1
    return mask


def mask_to_words(mask: np.ndarray) -> np.ndarray:
    """Pack a boolean [m, m] mask into uint64 words [m, ceil(m/64)], bit j%64 of word j//64."""
    m = mask.shape[0]
    W = (m + 63) // 64
    words = np.zeros((m, W), dtype=np.uint64)
    for i in range(m):
        for j in range(m):
            if mask[i, j]:
                words[i, j // 64] |= np.uint64(1) << np.uint64(j % 64)
    return words


def words_to_mask(words: np.ndarray, m: int) -> np.ndarray:
    out = np.zeros((words.shape[0], m), dtype=bool)
    for i in range(words.shape[0]):
        for j in range(m):
            out[i, j] = bool((int(words[i, j // 64]) >> (j % 64)) & 1)
    return out


def tree_build_one(logp: np.ndarray, root_token: int, k: int, depth: int, m: int) -> dict:
    """One sequence: ``logp`` is the fp32 draft log-prob rows [1 + (depth-1)k, V]."""
    if m < 1:
        raise ValueError("m must count at least the root")
    cands = _expand(logp, k, depth) if m > 1 else []
    if m - 1 > len(cands):
        raise ValueError("m - 1 exceeds the number of candidates")
    # Section 7.2: rerank all candidates, keep the top m-1 (the root is always kept).
    order = sorted(range(len(cands)), key=lambda x: (-cands[x].value, cands[x].layer, cands[x].idx))
    chosen = set(order[: m - 1])
    for x in chosen:
        if cands[x].parent != -1 and cands[x].parent not in chosen:
            raise ValueError("reranked selection is not a connected tree (log-probs > 0?)")
    # Flatten: root, then by (depth, parent's flat index, child rank).
    flat = {}
    seq = []
    for l in range(1, depth + 1):
        here = [x for x in chosen if cands[x].layer == l]
        here.sort(key=lambda x: (0 if cands[x].parent == -1 else flat[cands[x].parent], cands[x].rank))
        for x in here:
            flat[x] = 1 + len(seq)
            seq.append(x)
    tokens = np.zeros(m, dtype=np.int64)
    parents = np.zeros(m, dtype=np.int64)
    depth_out = np.zeros(m, dtype=np.int64)
    values = np.zeros(m, dtype=np.float64)
    node_row = np.full(m, -1, dtype=np.int64)
    tokens[0], parents[0], depth_out[0], values[0] = root_token, -1, 0, 0.0
    if m > 1:
        node_row[0] = 0
    for pos, x in enumerate(seq, start=1):
        c = cands[x]
        tokens[pos] = c.token
        parents[pos] = 0 if c.parent == -1 else flat[c.parent]
        depth_out[pos] = c.layer
        values[pos] = c.value
        if c.slot >= 0:
            node_row[pos] = 1 + (c.layer - 1) * k + c.slot
    mask = ancestor_mask(parents)
    return dict(tokens=tokens, parents=parents, depth=depth_out, values=values, node_row=node_row,
                mask=mask, mask_words=mask_to_words(mask), n_candidates=len(cands))


def tree_build(draft_logp, root_tokens, k: int, depth: int, m: int) -> dict:
    """Batched tree construction.  ``draft_logp``: [B, 1+(depth-1)k, V] fp32 log-probs.

    Returns int64 ``tokens``, ``parents``, ``depth``, ``node_row`` [B, m], fp64 ``values`` [B, m],
    bool ``mask`` [B, m, m] and uint64 ``mask_words`` [B, m, ceil(m/64)].
    """
    logp = np.asarray(draft_logp, dtype=np.float32)
    roots = np.asarray(root_tokens).astype(np.int64)
    per = [tree_build_one(logp[b], int(roots[b]), k, depth, m) for b in range(logp.shape[0])]
    return {key: np.stack([p[key] for p in per]) for key in
            ("tokens", "parents", "depth", "values", "node_row", "mask", "mask_words")}
