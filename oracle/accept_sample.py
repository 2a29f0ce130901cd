"""Oracle: stochastic (temperature T > 0) acceptance over the verified tree — TEST
INFRASTRUCTURE ONLY (fp64).

Source (web page, by title and section): "lesty.tech — EAGLE-2 vs. Medusa", section 4
(Mathematical Verification: Lossless Rejection Sampling).  For sampling at T > 0 the page
gives the chain form: a candidate x proposed by the draft distribution q is kept with
probability min(1, p(x) / q(x)), p being the base model's distribution; on a rejection the
step ends and one token is drawn from the residual max(0, p - q) / (1 - sum_y min(p, q)).
Kept candidates followed by one residual draw reproduce p exactly.

Readings (the page prints no tree form; each is listed in the design notes):

* p at node u is softmax(logits[u] / T) over the whole vocabulary (the target model's
  distribution for the position after u's root path).
* Tree form (multi-round rejection): starting at the root, the children of the current
  node are tried in increasing flat index (= child rank).  Each trial uses one uniform
  r in [0, 1) and keeps child x iff r * q(x) < p(x) — the event of probability
  min(1, p(x)/q(x)).  The first kept child becomes the current node and the walk goes one
  level down.  After a rejected child x, p becomes the page's residual
  norm(max(0, p - q)) and x leaves the proposal: q(x) = 0, q renormalised.  When every
  child is rejected, or the node has none, the step emits one token drawn from the
  current p (the residual) — the bonus.
* The proposal q, two modes:
    - ``q_mode = "point"``: every candidate is its own deterministic proposal, q = a unit
      mass on x.  The test reads r < p(x), and a rejection just removes x's mass from p.
      This is the lossless reading for EAGLE-2's trees, whose children are the draft's
      top-k, chosen without sampling.
    - ``q_mode = "draft"``: q is the draft model's distribution at the node, exp of the
      draft row the node's children were taken from (``node_row``), renormalised.  This
      is the page's formula taken literally; it reproduces p when the children were drawn
      from q without replacement.
* Uniforms are inputs, one per node: ``uniforms[b, c]`` decides the trial of child c (a
  node is tried at most once per step), and ``uniforms[b, 0]`` (the root is never tried)
  draws the bonus.
* The bonus is drawn by inverse CDF over token ids in increasing order: the smallest y
  whose cumulative residual mass exceeds r * (total mass).
* A residual with zero total mass (reached only through rounding, since in exact
  arithmetic it implies p == q, whose candidates are always kept) leaves p unchanged.
  A proposal whose remaining mass is zero stays zero, so the next test reads 0 < p(x).

Outputs per sequence: accept_len (nodes on the kept path, root included), accept_path
(flat indices, then -1) and bonus (the drawn token).  Two margins say how close the step came
to another outcome: ``margin`` = min over the trials taken of |r - p(x)/q(x)| (inf without
trials) and ``bonus_margin`` = the distance of the inverse-CDF target r * total to the drawn
token's cumulative bounds, over the total.  A GPU path computing p in fp32 may take another
branch only where one of them is small.

Pins (tests/test_oracle_accept_sample.py): the first emitted token is distributed as p
(exact enumeration over uniforms on a grid for a small chain, a chi-square test on trees in
both modes, with draft-mode children drawn from q without replacement); the one-candidate
chain case reproduces the page's acceptance probability and residual formula; the
second token, conditioned on the first being a kept draft, is distributed as the child's
p; as T -> 0 with point proposals the walk becomes the greedy longest-path acceptance.
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    if hasattr(x, "detach"):
        import torch
        return x.detach().to(torch.float64).cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def softmax_t(logits_row, temperature: float) -> np.ndarray:
    """softmax(logits / T) in fp64."""
    z = _f64(logits_row) / float(temperature)
    z = z - z.max()
    e = np.exp(z)
    return e / e.sum()


def _children(parents, u):
    return [c for c in range(len(parents)) if int(parents[c]) == u]


def _draw(p: np.ndarray, r: float):
    """Inverse CDF over increasing ids: the first y with cumsum(p)[y] > r * sum(p)."""
    total = p.sum()
    t = r * total
    cum = np.cumsum(p)
    y = int(np.searchsorted(cum, t, side="right"))
    if y >= len(p):                                   # t at the top end: the last id with mass
        y = int(np.nonzero(p > 0)[0][-1])
    lo = cum[y - 1] if y > 0 else 0.0
    return y, min(t - lo, cum[y] - t) / total


def accept_sample_one(logits, tokens, parents, uniforms, temperature: float, q_mode: str = "point",
                      draft_rows=None, node_row=None):
    """One sequence.  ``logits`` [m, V]; ``draft_rows`` [R, V] fp32 log-probs and ``node_row``
    [m] are needed for q_mode "draft".  Returns (accept_len, path list, bonus, margin,
    bonus_margin)."""
    if q_mode not in ("point", "draft"):
        raise ValueError("q_mode is 'point' or 'draft'")
    L = _f64(logits)
    m = L.shape[0]
    par = [int(x) for x in parents]
    if par[0] != -1 or any(not (0 <= par[i] < i) for i in range(1, m)):
        raise ValueError("parents[0] must be -1 and parents[i] in [0, i)")
    r = _f64(uniforms)
    path, u, margin = [0], 0, np.inf
    while True:
        p = softmax_t(L[u], temperature)
        kids = _children(par, u)
        q = None
        if q_mode == "draft" and kids:
            row = int(node_row[u])
            if row < 0:
                raise ValueError("a node with children has no draft row")
            q = np.exp(_f64(draft_rows[row]))
            q = q / q.sum()
        kept = None
        for c in kids:
            x = int(tokens[c])
            qx = 1.0 if q is None else q[x]
            ratio = np.inf if qx == 0.0 else p[x] / qx
            margin = min(margin, abs(r[c] - ratio))
            if r[c] * qx < p[x]:
                kept = c
                break
            # rejected: p <- norm(max(0, p - q)), x leaves the proposal
            if q is None:
                res = p.copy()
                res[x] = max(0.0, p[x] - 1.0)
            else:
                res = np.maximum(0.0, p - q)
            if res.sum() > 0.0:
                p = res / res.sum()
            if q is not None:
                q[x] = 0.0
                if q.sum() > 0.0:
                    q = q / q.sum()
        if kept is None:
            bonus, mb = _draw(p, r[0])
            return len(path), path, bonus, margin, mb
        path.append(kept)
        u = kept


def accept_sample(logits, tokens, parents, uniforms, temperature: float, q_mode: str = "point",
                  draft_logp=None, node_row=None):
    """Batched: ``logits`` [B, m, V], ``tokens``/``parents``/``uniforms`` [B, m],
    ``draft_logp`` [B, R, V] and ``node_row`` [B, m] for q_mode "draft".

    Returns int64 accept_len [B], accept_path [B, m] (-1 padded), bonus [B] and fp64
    margin [B] and bonus_margin [B]."""
    L = _f64(logits)
    B, m = L.shape[0], L.shape[1]
    alen = np.zeros(B, dtype=np.int64)
    apath = np.full((B, m), -1, dtype=np.int64)
    bonus = np.zeros(B, dtype=np.int64)
    margin = np.zeros(B)
    bmargin = np.zeros(B)
    for b in range(B):
        a, path, y, mg, mb = accept_sample_one(
            L[b], np.asarray(tokens)[b], np.asarray(parents)[b], np.asarray(uniforms)[b], temperature, q_mode,
            None if draft_logp is None else np.asarray(draft_logp)[b],
            None if node_row is None else np.asarray(node_row)[b])
        alen[b], bonus[b], margin[b], bmargin[b] = a, y, mg, mb
        apath[b, :a] = path
    return alen, apath, bonus, margin, bmargin
