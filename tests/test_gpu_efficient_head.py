"""GPU two-stage efficient draft head and tree_build_from_topk vs the oracle.

Integer-valued inputs keep u = B h exact in bf16 and every score and logit exact in fp32, so
the candidate sets and the top-k must match the fp64 oracle exactly (ties -> lower id on both
sides); the log-probabilities (fp32 logsumexp) match within 1e-5.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_tree_eagle_gb300 as ts
from gpu_helpers import dev, lib

pytestmark = pytest.mark.gpu


def _inputs(seed, M, V, d, rank, b_density=1.0):
    g = torch.Generator().manual_seed(seed)
    h = torch.randint(-1, 2, (M, d), generator=g)
    B = torch.randint(-1, 2, (rank, d), generator=g)
    if b_density < 1.0:
        B = B * (torch.rand(rank, d, generator=g) < b_density)
    A = torch.randint(-2, 3, (V, rank), generator=g)
    W = torch.randint(-2, 3, (V, d), generator=g)
    return [t.to(torch.bfloat16) for t in (h, B, A, W)]


CASES = [dict(M=7, V=3000, d=128, rank=32, tile_tokens=256, k_tile=3, k=10),
         dict(M=130, V=10000, d=64, rank=16, tile_tokens=512, k_tile=8, k=16),
         dict(M=1, V=256, d=8, rank=8, tile_tokens=256, k_tile=1, k=1),
         dict(M=33, V=5000, d=96, rank=24, tile_tokens=1024, k_tile=4, k=8),
         dict(M=80, V=128256, d=4096, rank=256, tile_tokens=1024, k_tile=2, k=10, b_density=1 / 64),
         # 1024 candidates: the largest set the warp-per-row top-k takes; 1256: one CTA per row
         dict(M=9, V=32768, d=64, rank=16, tile_tokens=256, k_tile=8, k=16),
         dict(M=6, V=40000, d=64, rank=16, tile_tokens=256, k_tile=8, k=12),
         # a one-id last tile: 9 candidates for k = 16, the last 7 entries are -1 / -inf
         dict(M=3, V=257, d=64, rank=16, tile_tokens=256, k_tile=8, k=16)]


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: f"M{c['M']}_V{c['V']}_d{c['d']}_r{c['rank']}_T{c['tile_tokens']}_kt{c['k_tile']}")
def test_integer_inputs_match_the_oracle(cfg):
    cfg = dict(cfg)
    dens = cfg.pop("b_density", 1.0)
    M, V, d, rank = cfg["M"], cfg["V"], cfg["d"], cfg["rank"]
    T, kt, k = cfg["tile_tokens"], cfg["k_tile"], cfg["k"]
    h, B, A, W = _inputs(M + V, M, V, d, rank, dens)
    lib()
    status = ts.new_status(dev())
    out = ts.efficient_head(h.to(dev()), B.to(dev()), A.to(dev()), W.to(dev()), tile_tokens=T, k_tile=kt, k=k,
                            with_candidates=True, status=status)
    ts.check_status(status)
    tok, lp, cand = oracle.efficient_head(h, B, A, W, T, kt, k)
    np.testing.assert_array_equal(out["candidates"].cpu().numpy(), cand)
    np.testing.assert_array_equal(out["top_tok"].cpu().numpy(), tok)
    np.testing.assert_allclose(out["top_logp"].cpu().numpy(), lp, rtol=0, atol=1e-5)


def _rows_from_lists(tok, lp, V):
    """Full draft rows holding only the listed (token, log-prob) pairs (-inf elsewhere)."""
    B, R, k = tok.shape
    rows = np.full((B, R, V), -np.inf, dtype=np.float32)
    for b in range(B):
        for r in range(R):
            rows[b, r, tok[b, r]] = lp[b, r]
    return rows


def test_tree_from_topk_equals_tree_from_rows():
    """Row lists from the oracle's row top-k of full draft rows give the same tree as the
    full-row build on the GPU."""
    B, k, depth, m, V = 3, 6, 5, 40, 4000
    R = 1 + (depth - 1) * k
    g = torch.Generator().manual_seed(21)
    logp = torch.log_softmax(torch.randn(B, R, V, generator=g) * 2, dim=-1).contiguous()
    roots = torch.tensor([1, 2, 3], dtype=torch.int32)
    ln = logp.numpy()
    tok = np.zeros((B, R, k), dtype=np.int32)
    lp = np.zeros((B, R, k), dtype=np.float32)
    for b in range(B):
        for r in range(R):
            tok[b, r], lp[b, r] = oracle.row_topk(ln[b, r], k)
    lib()
    status = ts.new_status(dev())
    a = ts.tree_build_from_topk(torch.from_numpy(tok).to(dev()), torch.from_numpy(lp).to(dev()),
                                roots.to(dev()), k, depth, m, status=status)
    bt = ts.tree_build(logp.to(dev()), roots.to(dev()), k, depth, m, status=status)
    ts.check_status(status)
    for key in ("tokens", "parents", "depth", "mask", "values", "node_row"):
        assert torch.equal(a[key], bt[key]), key


def test_unsorted_row_is_reported():
    B, k, depth, m = 1, 3, 2, 4
    R = 1 + (depth - 1) * k
    tok = torch.arange(R * k, dtype=torch.int32).view(1, R, k)
    lp = torch.tensor([[-1.0, -2.0, -3.0]] * R).view(1, R, k).clone()
    lp[0, 2, 1] = -0.5                          # row 2 out of order
    lib()
    status = ts.new_status(dev())
    ts.tree_build_from_topk(tok.to(dev()), lp.to(dev()), torch.zeros(1, dtype=torch.int32, device=dev()), k, depth,
                            m, status=status)
    assert int(status.item()) == -6


def test_efficient_head_feeds_the_tree():
    """Draft rows through the efficient head, then tree_build_from_topk: the same tree as the
    oracle builds from full rows holding the head's lists."""
    Bs, k, depth, m, V, d, rank = 2, 4, 4, 20, 6000, 64, 16
    R = 1 + (depth - 1) * k
    h, B, A, W = _inputs(5, Bs * R, V, d, rank)
    lib()
    status = ts.new_status(dev())
    out = ts.efficient_head(h.to(dev()), B.to(dev()), A.to(dev()), W.to(dev()), tile_tokens=512, k_tile=4, k=k,
                            status=status)
    roots = torch.tensor([7, 8], dtype=torch.int32)
    tree = ts.tree_build_from_topk(out["top_tok"].view(Bs, R, k).contiguous(), out["top_logp"].view(Bs, R, k).contiguous(),
                                   roots.to(dev()), k, depth, m, status=status)
    ts.check_status(status)
    tok = out["top_tok"].view(Bs, R, k).cpu().numpy()
    lp = out["top_logp"].view(Bs, R, k).cpu().numpy()
    ref = oracle.tree_build(_rows_from_lists(tok, lp, V), roots.numpy(), k, depth, m)
    for key in ("tokens", "parents", "depth", "node_row"):
        np.testing.assert_array_equal(tree[key].cpu().numpy(), ref[key])
    np.testing.assert_array_equal(tree["mask"].cpu().numpy().view(np.uint64), ref["mask_words"])
    np.testing.assert_array_equal(tree["values"].cpu().numpy(), ref["values"])
