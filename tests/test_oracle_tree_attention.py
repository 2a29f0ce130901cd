"""Pins of the oracle's tree attention (CPU only).

The pages print no attention numbers; the oracle is pinned through equivalences the
pages state: one tree pass == attending along each root path separately (rainlin.net,
section 四), a chain == ordinary causal attention (lesty.tech, section 5), one node ==
plain decode attention, and GQA sharing of KV heads.
"""
import math

import numpy as np
import torch
import torch.nn.functional as F

from oracle import ancestor_mask, tree_attention


def _random_tree(rng, m):
    return [-1] + [int(rng.integers(0, i)) for i in range(1, m)]


def _make(rng, B, Hq, Hkv, d, prefix, m, bs=4, parents=None):
    """Contiguous per-sequence K/V first, then scattered into a shuffled paged cache, so
    the brute force below never touches the block table."""
    n = [prefix[b] + m for b in range(B)]
    nblk = [math.ceil(x / bs) for x in n]
    NB = sum(nblk) + 3
    perm = rng.permutation(NB)
    table = -np.ones((B, max(nblk)), dtype=np.int64)
    kc = rng.normal(size=(NB, Hkv, bs, d))
    vc = rng.normal(size=(NB, Hkv, bs, d))
    Kc, Vc = [], []
    off = 0
    for b in range(B):
        table[b, : nblk[b]] = perm[off: off + nblk[b]]
        off += nblk[b]
        Kb = rng.normal(size=(n[b], Hkv, d))
        Vb = rng.normal(size=(n[b], Hkv, d))
        for p in range(n[b]):
            kc[table[b, p // bs], :, p % bs] = Kb[p]
            vc[table[b, p // bs], :, p % bs] = Vb[p]
        Kc.append(Kb)
        Vc.append(Vb)
    q = rng.normal(size=(B, m, Hq, d))
    if parents is None:
        parents = [_random_tree(rng, m) for _ in range(B)]
    mask = np.stack([ancestor_mask(p) for p in parents])
    return q, kc, vc, table, np.array(prefix), mask, parents, Kc, Vc


def test_brute_force_per_root_path():
    """Each node == single-query attention over prefix ++ its root path (root -> node)."""
    rng = np.random.default_rng(0)
    B, Hq, Hkv, d, m = 2, 4, 2, 8, 7
    prefix = [5, 9]
    q, kc, vc, table, plen, mask, parents, Kc, Vc = _make(rng, B, Hq, Hkv, d, prefix, m)
    scale = 1.0 / math.sqrt(d)
    out, lse = tree_attention(q, kc, vc, table, plen, mask, scale)
    g = Hq // Hkv
    for b in range(B):
        L = prefix[b]
        for i in range(m):
            path, n = [], i
            while n != -1:
                path.append(n)
                n = parents[b][n]
            path.reverse()
            pos = list(range(L)) + [L + t for t in path]
            for h in range(Hq):
                kh = h // g
                s = [scale * sum(q[b, i, h, c] * Kc[b][p, kh, c] for c in range(d)) for p in pos]
                mx = max(s)
                e = [math.exp(x - mx) for x in s]
                z = sum(e)
                ref = [sum(e[j] * Vc[b][pos[j], kh, c] for j in range(len(pos))) / z for c in range(d)]
                np.testing.assert_allclose(out[b, i, h], ref, rtol=0, atol=1e-12)
                assert abs(lse[b, i, h] - (mx + math.log(z))) < 1e-12


def test_chain_equals_causal_sdpa():
    """Chain tree == causal attention over prefix + chain (torch SDPA, fp64)."""
    rng = np.random.default_rng(1)
    B, Hq, Hkv, d, m, L = 1, 4, 4, 16, 6, 11
    par = [[-1] + list(range(m - 1))]
    q, kc, vc, table, plen, mask, _, Kc, Vc = _make(rng, B, Hq, Hkv, d, [L], m, parents=par)
    scale = 1.0 / math.sqrt(d)
    out, _ = tree_attention(q, kc, vc, table, plen, mask, scale)
    n = L + m
    qf = np.zeros((Hq, n, d))
    qf[:, L:, :] = q[0].transpose(1, 0, 2)
    qf[:, :L, :] = rng.normal(size=(Hq, L, d))
    ref = F.scaled_dot_product_attention(torch.tensor(qf)[None], torch.tensor(Kc[0].transpose(1, 0, 2))[None],
                                         torch.tensor(Vc[0].transpose(1, 0, 2))[None], is_causal=True,
                                         scale=scale)[0]
    np.testing.assert_allclose(out[0].transpose(1, 0, 2), ref[:, L:, :].numpy(), atol=1e-12, rtol=0)


def test_single_node_is_decode_attention_gqa():
    """m = 1 == plain decode attention; GQA heads h share KV head h // g (repeat_interleave)."""
    rng = np.random.default_rng(2)
    B, Hq, Hkv, d, m, L = 2, 8, 2, 16, 1, 13
    q, kc, vc, table, plen, mask, _, Kc, Vc = _make(rng, B, Hq, Hkv, d, [L, L + 4], m)
    scale = 0.3
    out, _ = tree_attention(q, kc, vc, table, plen, mask, scale)
    for b in range(B):
        K = torch.tensor(Kc[b]).permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)
        V = torch.tensor(Vc[b]).permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)
        Q = torch.tensor(q[b]).permute(1, 0, 2)  # [Hq, 1, d]
        ref = F.scaled_dot_product_attention(Q[None], K[None], V[None], scale=scale)[0]
        np.testing.assert_allclose(out[b, 0], ref[:, 0, :].numpy(), atol=1e-12, rtol=0)


def test_select_subset_matches_full():
    rng = np.random.default_rng(3)
    q, kc, vc, table, plen, mask, _, _, _ = _make(rng, 2, 4, 1, 8, [3, 7], 5)
    full, lf = tree_attention(q, kc, vc, table, plen, mask, 0.5)
    sel = [(0, 1, 2), (1, 4, 0), (1, 0, 3)]
    part, lp = tree_attention(q, kc, vc, table, plen, mask, 0.5, select=sel)
    for (b, i, h) in sel:
        np.testing.assert_allclose(part[b, i, h], full[b, i, h], rtol=0, atol=1e-14)
        assert abs(lp[b, i, h] - lf[b, i, h]) < 1e-14


def test_zero_prefix():
    rng = np.random.default_rng(4)
    q, kc, vc, table, plen, mask, parents, Kc, Vc = _make(rng, 1, 1, 1, 4, [0], 3, parents=[[-1, 0, 0]])
    out, _ = tree_attention(q, kc, vc, table, plen, mask, 1.0)
    np.testing.assert_allclose(out[0, 0, 0], Vc[0][0, 0], atol=1e-15)  # the root sees only itself
