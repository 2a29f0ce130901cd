"""Pins of the oracle's stochastic tree acceptance (CPU only).

What is pinned comes from the mathematics the page states, not from the oracle's own
formulas: the emitted token must be distributed as the target p (lossless), the
one-candidate chain must reproduce the page's printed acceptance probability and residual,
and the T -> 0 limit must reduce to the greedy longest-path acceptance (another routine).
"""
import numpy as np
import pytest
from scipy.stats import chisquare

from oracle import accept_longest_path, accept_sample
from oracle.accept_sample import accept_sample_one, softmax_t


def _draw_without_replacement(rng, q, n):
    """n distinct ids drawn one after another from q, each draw renormalised over the rest."""
    q = q.copy()
    out = []
    for _ in range(n):
        x = int(rng.choice(len(q), p=q / q.sum()))
        out.append(x)
        q[x] = 0.0
    return out


# a small tree: root 0 -> {1, 2, 3}; 1 -> {4, 5}; 2 -> {6}; 4 -> {7}
PARENTS = np.array([-1, 0, 0, 0, 1, 1, 2, 4])
NODE_ROW = np.array([0, 1, 2, -1, 3, -1, -1, -1])   # rows the children of 0, 1, 2, 4 were drawn from
V = 6


def _tree_dists(seed, T):
    rng = np.random.default_rng(seed)
    logits = rng.normal(0, 1.5, size=(len(PARENTS), V))
    draft = rng.normal(0, 1.5, size=(4, V))
    draft = draft - np.log(np.exp(draft).sum(1, keepdims=True))
    return logits, draft


def _emitted(alen, path, bonus, tokens, i):
    """Token number i (1-based) emitted by the step: a kept draft, else the bonus, else None."""
    if i < alen:
        return int(tokens[path[i]])
    if i == alen:
        return int(bonus)
    return None


def _sample_tokens(rng, q_mode, draft):
    """Tokens of the tree: children drawn from q without replacement (draft mode), or a
    fixed choice (point mode: the proposal is deterministic)."""
    tok = np.zeros(len(PARENTS), dtype=np.int64)
    for u, row in enumerate(NODE_ROW):
        kids = [c for c in range(len(PARENTS)) if PARENTS[c] == u]
        if not kids:
            continue
        if q_mode == "draft":
            ids = _draw_without_replacement(rng, np.exp(draft[row]), len(kids))
        else:
            ids = [(3 * u + 2 * j + 1) % V for j in range(len(kids))]   # distinct siblings
        tok[kids] = ids
    return tok


@pytest.mark.parametrize("q_mode,T", [("point", 1.0), ("point", 0.7), ("draft", 1.0), ("draft", 1.6)])
def test_first_and_second_tokens_follow_the_target(q_mode, T):
    """Lossless: token 1 ~ p(root); token 2 given that token 1 was child 1's draft ~ p(node 1)."""
    logits, draft = _tree_dists(7, T)
    rng = np.random.default_rng(11)
    N = 12000
    first = np.zeros(V)
    second = np.zeros(V)
    for _ in range(N):
        tok = _sample_tokens(rng, q_mode, draft)
        u = rng.random(len(PARENTS))
        a, path, y, _, _ = accept_sample_one(logits, tok, PARENTS, u, T, q_mode, draft, NODE_ROW)
        first[_emitted(a, path, y, tok, 1)] += 1
        if a >= 2 and path[1] == 1:
            second[_emitted(a, path, y, tok, 2)] += 1
    p0 = softmax_t(logits[0], T)
    p1 = softmax_t(logits[1], T)
    assert chisquare(first, p0 * N).pvalue > 1e-4
    assert second.sum() > 1000
    assert chisquare(second, p1 * second.sum()).pvalue > 1e-4


def test_draft_proposals_with_fixed_children_are_not_lossless():
    """The draft-mode rule relies on the children being drawn from q: with fixed children the
    first token is visibly off p, which the chi-square test above would catch."""
    logits, draft = _tree_dists(7, 1.0)
    rng = np.random.default_rng(3)
    tok = _sample_tokens(np.random.default_rng(0), "point", draft)
    N = 12000
    first = np.zeros(V)
    for _ in range(N):
        a, path, y, _, _ = accept_sample_one(logits, tok, PARENTS, rng.random(len(PARENTS)), 1.0, "draft", draft,
                                          NODE_ROW)
        first[_emitted(a, path, y, tok, 1)] += 1
    assert chisquare(first, softmax_t(logits[0], 1.0) * N).pvalue < 1e-6


def _grid(G):
    return (np.arange(G) + 0.5) / G


@pytest.mark.parametrize("q_mode", ["point", "draft"])
def test_one_candidate_chain_reproduces_the_page_formulas(q_mode):
    """Root -> one child x: P(keep) = min(1, p(x)/q(x)); a rejected step draws from
    max(0, p - q) / (1 - sum min(p, q)).  Integrated over midpoint grids of the uniforms."""
    G = 4000
    rng = np.random.default_rng(5)
    lg = rng.normal(0, 1, size=(2, V))
    d = rng.normal(0, 1, size=(1, V))
    d = d - np.log(np.exp(d).sum())
    p = softmax_t(lg[0], 1.0)
    q = np.exp(d[0]) / np.exp(d[0]).sum()
    x = int(np.argmax(q - p))                          # a token the draft over-proposes: P(keep) < 1
    tok = np.array([0, x])
    par = np.array([-1, 0])
    nr = np.array([0, -1])
    qq = np.zeros(V)
    qq[x] = 1.0
    qx = q if q_mode == "draft" else qq
    kept = 0
    for r in _grid(G):
        a, _, _, _, _ = accept_sample_one(lg, tok, par, np.array([0.5, r]), 1.0, q_mode, d, nr)
        kept += a == 2
    assert abs(kept / G - min(1.0, p[x] / qx[x])) <= 1.0 / G
    # residual: the child is rejected for r = 0.999999; sweep the bonus uniform
    hist = np.zeros(V)
    for r0 in _grid(G):
        a, _, y, _, _ = accept_sample_one(lg, tok, par, np.array([r0, 0.999999]), 1.0, q_mode, d, nr)
        assert a == 1
        hist[y] += 1
    expect = np.maximum(0.0, p - qx) / (1.0 - np.minimum(p, qx).sum())
    np.testing.assert_allclose(hist / G, expect, atol=1.0 / G)


def test_kept_child_takes_the_walk_down():
    """p == q everywhere: every first child is kept (r * q(x) < p(x) for all r < 1)."""
    lg = np.log(np.array([[0.1, 0.2, 0.3, 0.4]] * 4))
    d = lg[:3].copy()
    par = np.array([-1, 0, 1, 1])
    tok = np.array([0, 2, 1, 3])
    nr = np.array([0, 1, -1, -1])
    a, path, y, _, _ = accept_sample_one(lg, tok, par, np.array([0.3, 0.99, 0.99, 0.5]), 1.0, "draft", d, nr)
    assert a == 3 and path == [0, 1, 2]


def test_zero_target_mass_rejects_every_candidate():
    lg = np.array([[0.0, 0.0, -np.inf, -np.inf], [0.0, 0.0, 0.0, 0.0], [0.0, 0.0, 0.0, 0.0]])
    par = np.array([-1, 0, 0])
    tok = np.array([0, 2, 3])
    for mode in ("point", "draft"):
        d = np.log(np.array([[0.1, 0.1, 0.4, 0.4]]))
        a, path, y, _, _ = accept_sample_one(lg, tok, par, np.array([0.75, 0.0, 0.0]), 1.0, mode, d,
                                          np.array([0, -1, -1]))
        assert a == 1 and y == 1                     # residual is p itself here: [0.5, 0.5, 0, 0]


def test_low_temperature_is_greedy():
    """T -> 0 with point proposals: p is one-hot at the argmax, so a child is kept iff it is its
    parent's argmax and the bonus is the argmax at the kept node — the greedy routine."""
    rng = np.random.default_rng(2)
    B, m, Vv = 6, 30, 50
    logits = rng.permutation(np.arange(B * m * Vv)).reshape(B, m, Vv) * 0.01
    amax = logits.argmax(-1)
    parents = np.zeros((B, m), dtype=np.int64)
    tokens = np.zeros((B, m), dtype=np.int64)
    for b in range(B):
        parents[b, 0] = -1
        used = {}
        for i in range(1, m):
            p = int(rng.integers(0, i))
            parents[b, i] = p
            want = amax[b, p] if rng.random() < 0.6 else int(rng.integers(0, Vv))
            while want in used.setdefault(p, set()):
                want = (want + 1) % Vv
            used[p].add(want)
            tokens[b, i] = want
    alen, apath, bonus, _, _ = accept_sample(logits, tokens, parents, rng.random((B, m)), 1e-6, "point")
    ref = accept_longest_path(tokens, parents, amax)
    np.testing.assert_array_equal(alen, ref[0])
    np.testing.assert_array_equal(apath, ref[1])
    np.testing.assert_array_equal(bonus, ref[2])
    assert (alen > 2).any()


def test_margin_is_the_distance_to_the_nearest_threshold():
    lg = np.log(np.array([[0.25, 0.25, 0.5], [1 / 3, 1 / 3, 1 / 3]]))
    par = np.array([-1, 0])
    tok = np.array([0, 2])
    a, _, _, mg, mb = accept_sample_one(lg, tok, par, np.array([0.1, 0.45]), 1.0, "point")
    assert a == 2 and abs(mg - 0.05) < 1e-12   # trial: |0.45 - 0.5|
    assert abs(mb - 0.1) < 1e-12               # bonus at node 1: 0.1 in [0, 1/3)
    a, _, y, mg, mb = accept_sample_one(lg, tok, par, np.array([0.3, 0.6]), 1.0, "point")
    assert a == 1 and y == 0 and abs(mg - 0.1) < 1e-12      # trial: |0.6 - 0.5|
    assert abs(mb - 0.2) < 1e-12                            # residual [.5, .5, 0]: 0.3 in [0, 0.5)
    _, _, _, mg, _ = accept_sample_one(lg[:1], tok[:1], par[:1], np.array([0.3]), 1.0, "point")
    assert mg == np.inf


def test_bad_parents_raise():
    with pytest.raises(ValueError):
        accept_sample_one(np.zeros((2, 3)), [0, 1], [0, 0], [0.5, 0.5], 1.0)
    with pytest.raises(ValueError):
        accept_sample_one(np.zeros((2, 3)), [0, 1], [-1, 0], [0.5, 0.5], 1.0, "draft", np.zeros((1, 3)),
                          [-1, -1])
