"""Pins of the two-stage efficient-head oracle ("jialefu.github.io — EAGLE-4 efficient LM head")."""
import math

import numpy as np
import pytest
import torch

import oracle


def _case(seed, M=3, d=16, rank=8, V=40):
    g = torch.Generator().manual_seed(seed)
    h = torch.randint(-2, 3, (M, d), generator=g).to(torch.bfloat16)
    B = torch.randint(-1, 2, (rank, d), generator=g).to(torch.bfloat16)
    A = torch.randint(-2, 3, (V, rank), generator=g).to(torch.bfloat16)
    W = torch.randint(-2, 3, (V, d), generator=g).to(torch.bfloat16)
    return h, B, A, W


@pytest.mark.parametrize("seed", range(3))
def test_every_id_a_candidate_gives_the_exact_full_vocabulary_topk(seed):
    h, B, A, W = _case(seed)
    V, k = W.shape[0], 5
    tok, lp, cand = oracle.efficient_head(h, B, A, W, tile_tokens=8, k_tile=8, k=k)
    logits = h.double().numpy() @ W.double().numpy().T
    for r in range(h.shape[0]):
        order = sorted(range(V), key=lambda i: (-logits[r, i], i))[:k]
        assert list(tok[r]) == order
        lse = math.log(sum(math.exp(x) for x in logits[r]))
        np.testing.assert_allclose(lp[r], [logits[r, i] - lse for i in order], rtol=0, atol=1e-12)


def test_candidate_sets_by_explicit_tile_loops():
    h, B, A, W = _case(7, V=37)
    cand = oracle.efficient_head(h, B, A, W, tile_tokens=10, k_tile=3, k=4)[2]
    hn, Bn, An = h.double().numpy(), B.double().numpy(), A.double().numpy()
    u = hn @ Bn.T                               # small integers: exact in bf16
    scores = u @ An.T
    for r in range(h.shape[0]):
        for t, (lo, hi) in enumerate([(0, 10), (10, 20), (20, 30), (30, 37)]):
            best = []
            for i in range(lo, hi):             # insertion by (score desc, id asc)
                best.append(i)
                best.sort(key=lambda j: (-scores[r, j], j))
                best = best[:3]
            assert list(cand[r, 3 * t:3 * t + 3]) == best


def test_short_tile_and_ties():
    h = torch.tensor([[1.0, 0.0]]).to(torch.bfloat16)
    B = torch.tensor([[1.0, 0.0], [0.0, 1.0]]).to(torch.bfloat16)
    A = torch.tensor([[1.0, 0.0]] * 5).to(torch.bfloat16)        # every score 1: ties -> lower id
    W = torch.tensor([[1.0, 0.0], [2.0, 0.0], [2.0, 0.0], [0.0, 0.0], [5.0, 0.0]]).to(torch.bfloat16)
    tok, lp, cand = oracle.efficient_head(h, B, A, W, tile_tokens=4, k_tile=2, k=3)
    assert list(cand[0]) == [0, 1, 4, -1]                          # tile [4] keeps its one id
    assert list(tok[0]) == [4, 1, 0]          # logits 5, 2, 1; id 2 (logit 2) is not a candidate


def test_fewer_candidates_than_k_pad_with_minus_one_and_minus_inf():
    """Three candidates for k = 4: the three by logit (5, 2, 1) with log-probabilities from the
    closed-form logsumexp over exactly those three logits, then one padding entry."""
    h = torch.tensor([[1.0, 0.0]]).to(torch.bfloat16)
    B = torch.tensor([[1.0, 0.0], [0.0, 1.0]]).to(torch.bfloat16)
    A = torch.tensor([[1.0, 0.0]] * 5).to(torch.bfloat16)
    W = torch.tensor([[1.0, 0.0], [2.0, 0.0], [2.0, 0.0], [0.0, 0.0], [5.0, 0.0]]).to(torch.bfloat16)
    tok, lp, _ = oracle.efficient_head(h, B, A, W, tile_tokens=4, k_tile=2, k=4)
    assert list(tok[0]) == [4, 1, 0, -1]
    lse = math.log(math.exp(5) + math.exp(2) + math.exp(1))
    np.testing.assert_allclose(lp[0, :3], [5 - lse, 2 - lse, 1 - lse], rtol=0, atol=1e-12)
    assert lp[0, 3] == -math.inf


def test_one_tile_is_global_topk_on_the_low_rank_scores():
    h, B, A, W = _case(11, V=30)
    cand = oracle.efficient_head(h, B, A, W, tile_tokens=64, k_tile=6, k=2)[2]
    u = h.double().numpy() @ B.double().numpy().T
    scores = u @ A.double().numpy().T
    for r in range(h.shape[0]):
        assert list(cand[r]) == sorted(range(30), key=lambda i: (-scores[r, i], i))[:6]
