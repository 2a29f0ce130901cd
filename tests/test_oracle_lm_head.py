"""Pins of the LM-head argmax oracle: explicit loops, first-index ties, and composition with
the acceptance walk."""
import numpy as np
import pytest

import oracle


def _loops(h, w):
    M, K = h.shape
    N = w.shape[0]
    out = np.zeros((M, N))
    for r in range(M):
        for n in range(N):
            acc = 0.0
            for k in range(K):
                acc += float(h[r, k]) * float(w[n, k])
            out[r, n] = acc
    return out


@pytest.mark.parametrize("seed", range(3))
def test_matches_explicit_loops(seed):
    rng = np.random.default_rng(seed)
    h = rng.integers(-3, 4, size=(4, 9)).astype(np.float64)
    w = rng.integers(-3, 4, size=(13, 9)).astype(np.float64)
    ref = _loops(h, w)
    idx, mx = oracle.lm_head_argmax(h, w)
    for r in range(4):
        best = max(range(13), key=lambda n: (ref[r, n], -n))
        assert idx[r] == best and mx[r] == ref[r, best]


def test_ties_go_to_the_first_index():
    h = np.array([[1.0, 2.0], [0.0, 0.0]])
    w = np.array([[0.0, 1.0], [1.0, 0.5], [2.0, 0.0], [1.0, 0.5]])   # row 0: logits 2, 2, 2, 2
    idx, mx = oracle.lm_head_argmax(h, w)
    assert list(idx) == [0, 0] and list(mx) == [2.0, 0.0]


def test_composition_with_the_acceptance_walk():
    """Accepting with the LM head's argmax == accepting with the argmax of explicit logits."""
    rng = np.random.default_rng(4)
    B, m, K, V = 2, 6, 5, 7
    h = rng.integers(-2, 3, size=(B * m, K)).astype(np.float64)
    w = rng.integers(-2, 3, size=(V, K)).astype(np.float64)
    parents = np.array([[-1, 0, 0, 1, 1, 3], [-1, 0, 1, 2, 3, 4]])
    idx, _ = oracle.lm_head_argmax(h, w)
    amax = idx.reshape(B, m)
    tokens = np.zeros((B, m), dtype=np.int64)
    for b in range(B):            # every child carries its parent's argmax: the deepest node wins
        for i in range(1, m):
            tokens[b, i] = amax[b, parents[b, i]]
    tokens[0, 2] = (amax[0, 0] + 1) % V   # except one sibling
    logits = _loops(h, w).reshape(B, m, V)
    a1 = oracle.accept_longest_path(tokens, parents, amax)
    a2 = oracle.accept_longest_path(tokens, parents, oracle.target_argmax(logits))
    for x, y in zip(a1, a2):
        np.testing.assert_array_equal(x, y)
    assert int(a1[0][1]) == m           # chain sequence: all nodes accepted


def test_error_bound_covers_fp32_accumulation():
    rng = np.random.default_rng(9)
    h = rng.standard_normal((3, 256)).astype(np.float32)
    w = rng.standard_normal((50, 256)).astype(np.float32)
    exact = oracle.lm_head_logits(h, w)
    approx = np.zeros_like(exact)
    for r in range(3):            # a different order: reversed fp32 accumulation
        for n in range(50):
            acc = np.float32(0)
            for k in range(255, -1, -1):
                acc = np.float32(acc + np.float32(h[r, k]) * np.float32(w[n, k]))
            approx[r, n] = acc
    bound = oracle.fp32_error_bound(h, w)
    assert (np.abs(approx - exact).max(axis=1) <= bound).all()
