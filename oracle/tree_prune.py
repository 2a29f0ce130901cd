"""Oracle: cost-aware pruning of the draft tree before verification — TEST INFRASTRUCTURE ONLY.

Sources (web pages, by title and section):

* "jialefu.github.io — EAGLE-4 efficient LM head", section "EAGLE-Harness": the harness
  builds the tree from draft and target costs and the draft confidence, may prune the tree
  before verification, and estimates the expected accepted-token count from the draft
  probabilities (its own heuristics are not given).
* "rainlin.net/posts/eagle", section 7.1: the value of a node is the product of the draft
  confidences on its root path; section 六: the draft confidence tracks the acceptance rate.

Readings (each listed in the design notes):

* Expected tokens of one verification of a tree S (root included): 1 + sum over the non-root
  nodes i of S of exp(V_i).  With the confidence read as the probability that the target
  emits that token, node i is on the accepted path with probability exp(V_i) (siblings are
  exclusive), and the expected accepted length is the sum of those probabilities; the step
  adds one token of its own.
* Candidate trees are the prefixes of the rerank order (value descending, then shallower, then
  lower flat index): values never increase along a root path (log-probabilities <= 0), so
  every prefix is a connected tree, and the prefix of n - 1 nodes holds the largest value
  sum of any connected tree of n nodes.
* One node count n for the whole batch (the verification pass has one shape [B, n]), chosen
  to maximise the expected tokens per unit time
      rate(n) = sum_b (1 + sum of exp(V) over the first n - 1 nodes of b)
                / (t_draft + t_fixed + t_node * B * n),
  ties -> the smaller n.  t_draft (the drafting time of the round), t_fixed and t_node (the
  verification pass's fixed and per-node time) are inputs.
* The kept nodes keep their flat order; parents, depths, draft rows and the ancestor mask
  are re-indexed to it.  Early stopping inside drafting is not covered: the drafter here is
  a table of pre-drawn rows, with no drafting loop to stop.

Pins (tests/test_oracle_tree_prune.py): a Monte Carlo walk in which each child's token is
emitted with its draft probability reproduces 1 + sum exp(V); brute force over every
connected subtree of small trees shows the rerank prefix has the largest value sum for its
size; free verification keeps every node, prohibitive verification keeps only the root; the
pruned tree is a subtree of the original with the mask of its own parent array.
"""
from __future__ import annotations

import numpy as np

from .tree_build import ancestor_mask, mask_to_words


def rerank_order(values, depth) -> list:
    """Non-root nodes in rerank order: value descending, then shallower, then lower index."""
    m = len(values)
    return sorted(range(1, m), key=lambda i: (-float(values[i]), int(depth[i]), i))


def expected_tokens(values, order, n: int) -> float:
    """1 + sum of exp(V) over the first n - 1 nodes of ``order`` (fp64)."""
    return 1.0 + float(sum(np.exp(float(values[i])) for i in order[: n - 1]))


def tree_prune(tokens, parents, depth, values, t_draft: float, t_fixed: float, t_node: float, node_row=None,
               n=None):
    """Batched pruning.  ``values`` fp64 [B, m] (from tree_build, flat order).  ``n`` forces
    the kept node count (the rates are still returned).

    Returns (n, out, rate) with n the kept node count (root included), ``rate`` fp64 [m] the
    rate of every candidate n = 1..m, and ``out`` holding int64 ``tokens``, ``parents``,
    ``depth``, ``node_row`` (if given), ``kept`` (old flat index of each kept node) [B, n],
    fp64 ``values`` [B, n], ``expected`` [B] and uint64 ``mask_words`` [B, n, ceil(n/64)]."""
    tokens, parents, depth = np.asarray(tokens), np.asarray(parents), np.asarray(depth)
    values = np.asarray(values, dtype=np.float64)
    B, m = values.shape
    orders = [rerank_order(values[b], depth[b]) for b in range(B)]
    rate = np.zeros(m)
    for c in range(1, m + 1):
        tok = sum(expected_tokens(values[b], orders[b], c) for b in range(B))
        rate[c - 1] = tok / (t_draft + t_fixed + t_node * B * c)
    best = int(np.argmax(rate)) + 1 if n is None else int(n)   # first maximum: ties -> smaller n
    out = {k: np.zeros((B, best), dtype=np.int64) for k in ("tokens", "parents", "depth", "kept")}
    if node_row is not None:
        out["node_row"] = np.zeros((B, best), dtype=np.int64)
    out["values"] = np.zeros((B, best))
    out["expected"] = np.zeros(B)
    masks = []
    for b in range(B):
        keep = sorted([0] + orders[b][: best - 1])
        new = {old: j for j, old in enumerate(keep)}
        for j, old in enumerate(keep):
            out["kept"][b, j] = old
            out["tokens"][b, j] = tokens[b, old]
            out["parents"][b, j] = -1 if old == 0 else new[int(parents[b, old])]
            out["depth"][b, j] = depth[b, old]
            out["values"][b, j] = values[b, old]
            if node_row is not None:
                out["node_row"][b, j] = np.asarray(node_row)[b, old]
        out["expected"][b] = expected_tokens(values[b], orders[b], best)
        masks.append(mask_to_words(ancestor_mask(out["parents"][b])))
    out["mask_words"] = np.stack(masks)
    return best, out, rate
