"""Oracle: the draft model's two-stage efficient LM head (TEST INFRASTRUCTURE ONLY).

Source (web page, by title and section): "jialefu.github.io — EAGLE-4 efficient LM head",
sections "EAGLE Efficient LM Head" (stage one: a low-rank head scores the whole vocabulary and
candidates are selected by top-k; stage two: the full LM-head rows of the candidates are
gathered and their logits recomputed from the original hidden states) and "A variant based
on local Top-k" (the selection runs per vocabulary tile, fused with the tile's matrix
multiplication; the tiles' candidates are concatenated).

Definitions (per row r of hidden [M, d]; low-rank factors B [rank, d] and A [V, rank]; full
head W [V, d]):

1. ``u = bf16(B @ h)`` — the low-rank projection, rounded to bf16 (the tensor-core operand of
   the next product; the page leaves its precision open: reading).
2. ``scores = A @ u`` (fp64 here); the vocabulary is cut into tiles of ``tile_tokens``
   consecutive ids; each tile keeps its ``k_tile`` best ids (score descending, ties -> lower
   id; a tile with fewer ids keeps them all).  Candidates = the tiles' ids, tile by tile.
3. ``logits[c] = W[c] @ h`` for every candidate (fp64 here).
4. Output: the ``k`` candidates with the largest logits (ties -> lower id), in that order,
   with log-probabilities normalised over the candidate set,
   ``lp = logit - logsumexp(candidate logits)`` (the page samples from the candidates; the mass
   of the other ids is not computed: reading).

Pins (tests/test_oracle_efficient_head.py): when every id is a candidate (k_tile =
tile_tokens) the output equals the exact full-vocabulary top-k and log-softmax; explicit
per-tile loops for the candidate sets; ties; and a single tile reduces to global top-k on the
low-rank scores.
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    if hasattr(x, "detach"):
        import torch
        return x.detach().to(torch.float64).cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def _bf16_round(x: np.ndarray) -> np.ndarray:
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def candidates(hidden, lr_b, lr_a, tile_tokens: int, k_tile: int) -> np.ndarray:
    """int64 [M, C] candidate ids, C = n_tiles * k_tile (-1 where a short tile has fewer ids)."""
    h, B, A = _f64(hidden), _f64(lr_b), _f64(lr_a)
    u = _bf16_round((h @ B.T).astype(np.float32))
    scores = u @ A.T                                   # [M, V]
    M, V = scores.shape
    n_tiles = -(-V // tile_tokens)
    out = np.full((M, n_tiles * k_tile), -1, dtype=np.int64)
    for r in range(M):
        for t in range(n_tiles):
            lo, hi = t * tile_tokens, min(V, (t + 1) * tile_tokens)
            ids = np.arange(lo, hi)
            order = sorted(ids, key=lambda i: (-scores[r, i], i))[:k_tile]
            out[r, t * k_tile:t * k_tile + len(order)] = order
    return out


def efficient_head(hidden, lr_b, lr_a, weight, tile_tokens: int, k_tile: int, k: int):
    """Returns (top_tok int64 [M, k], top_logp fp64 [M, k], candidates int64 [M, C]).  When short
    tiles leave a row fewer than k candidates, its remaining entries are token -1 with
    log-probability -inf (a reading: the pages do not meet the case)."""
    h, W = _f64(hidden), _f64(weight)
    cand = candidates(hidden, lr_b, lr_a, tile_tokens, k_tile)
    M = h.shape[0]
    tok = np.full((M, k), -1, dtype=np.int64)
    lp = np.full((M, k), -np.inf)
    for r in range(M):
        ids = [int(i) for i in cand[r] if i >= 0]
        logits = {i: float(W[i] @ h[r]) for i in ids}
        mx = max(logits.values())
        lse = mx + np.log(sum(np.exp(v - mx) for v in logits.values()))
        best = sorted(ids, key=lambda i: (-logits[i], i))[:k]
        tok[r, :len(best)] = best
        lp[r, :len(best)] = [logits[i] - lse for i in best]
    return tok, lp, cand
