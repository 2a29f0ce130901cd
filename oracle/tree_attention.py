"""Oracle: tree attention over a paged KV prefix (fp64).

Sources (web pages, by title and section):

* "rainlin.net/posts/eagle", section 四 (Tree Attention): the tree's nodes are flattened
  into one sequence; each node attends only to the tokens on its own root-to-node path,
  and one pass is equivalent to verifying every path separately.
* "lesty.tech — EAGLE-2 vs. Medusa", section 5: a chain is the ordinary causal mask;
  section 8 (Speculative PagedAttention): the tree's K/V live in blocks of the same paged
  sequence after the committed prefix.

Definition used here, per batch b, query head h (KV head h // g), tree node i:
keys are the L_b prefix positions (through the block table) plus tree position
L_b + t for every t with mask bit (i, t) set; s_j = scale * <q, k_j>;
p = softmax(s) over those keys; out = sum_j p_j v_j; lse = log sum_j exp(s_j).
Everything is computed in fp64 from the exact input values.

Reading: there is no positional encoding here (RoPE happens upstream at position
L_b + depth); the paged layout is [num_blocks, Hkv, block_size, d].

Pins (tests/test_oracle_tree_attention.py): brute force per node over the gathered
root path (no mask, no paging), the chain case against torch's causal
``scaled_dot_product_attention`` in fp64, m = 1 against plain decode attention, and GQA
head mapping against ``repeat_interleave`` + SDPA.  No numeric attention output is
printed on the pages, so absolute values are pinned only through these equivalences.
"""
from __future__ import annotations

import numpy as np


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor: exact widening to fp64
        import torch
        return x.detach().to(torch.float64).cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def gather_sequence(cache, table_row, n: int) -> np.ndarray:
    """Logical positions 0..n-1 of one sequence from a paged cache -> fp64 [n, Hkv, d].

    Only the gathered rows are widened to fp64 (exactly), so large caches stay in their
    storage type."""
    bs = cache.shape[2]
    pos = np.arange(n)
    blocks = np.asarray(table_row)[pos // bs]
    if np.any(blocks < 0) or np.any(blocks >= cache.shape[0]):
        raise ValueError("block table entry out of range")
    if hasattr(cache, "detach"):
        import torch
        rows = cache[torch.from_numpy(blocks), :, torch.from_numpy(pos % bs), :]
        return _f64(rows)
    return np.asarray(cache[blocks, :, pos % bs, :], dtype=np.float64)


def tree_attention(q, k_cache, v_cache, block_table, prefix_len, mask, scale: float,
                   select=None):
    """Tree attention in fp64.

    q [B, m, Hq, d]; k_cache/v_cache [NB, Hkv, bs, d]; block_table [B, max_blocks];
    prefix_len [B]; mask: boolean [B, m, m] (ancestor-or-self).
    ``select``: optional iterable of (b, i, h) to compute only those outputs.
    Returns (out [B, m, Hq, d] fp64, lse [B, m, Hq] fp64); unselected entries are NaN.
    """
    qd = _f64(q)
    kc, vc = k_cache, v_cache
    table = np.asarray(block_table).astype(np.int64)
    plen = np.asarray(prefix_len).astype(np.int64)
    mask = np.asarray(mask, dtype=bool)
    B, m, Hq, d = qd.shape
    Hkv = kc.shape[1]
    g = Hq // Hkv
    out = np.full((B, m, Hq, d), np.nan)
    lse = np.full((B, m, Hq), np.nan)
    want = None
    if select is not None:
        want = {}
        for (b, i, h) in select:
            want.setdefault(int(b), set()).add((int(i), int(h)))
    for b in range(B):
        if want is not None and b not in want:
            continue
        L = int(plen[b])
        n = L + m
        Kb = gather_sequence(kc, table[b], n)    # [n, Hkv, d]
        Vb = gather_sequence(vc, table[b], n)
        allowed = np.zeros((m, n), dtype=bool)
        allowed[:, :L] = True
        allowed[:, L:] = mask[b]
        for h in range(Hq):
            nodes = range(m) if want is None else sorted(i for (i, hh) in want[b] if hh == h)
            nodes = list(nodes)
            if not nodes:
                continue
            kh = h // g
            s = (qd[b, nodes, h, :] @ Kb[:, kh, :].T) * scale          # [len(nodes), n]
            s = np.where(allowed[nodes], s, -np.inf)
            smax = s.max(axis=1, keepdims=True)
            e = np.exp(s - smax)
            z = e.sum(axis=1, keepdims=True)
            out[b, nodes, h, :] = (e @ Vb[:, kh, :]) / z
            lse[b, nodes, h] = (smax + np.log(z))[:, 0]
    return out, lse
