"""GPU stochastic tree acceptance (multi-round rejection sampling) vs the oracle.

Every trial and the final draw are floating-point decisions.  The GPU computes p in fp32
(fp64 running sums for the inverse CDF), the oracle in fp64.  So a sequence is compared
exactly (length, path, drawn token) when every trial the oracle took lies more than
TRIAL_TOL from its threshold and the draw's target more than BONUS_TOL (of the total mass)
from the drawn token's cumulative bounds.  The few others must still be valid outcomes.
TRIAL_TOL covers the fp32 normaliser (sum of up to 2^17 terms, relative error ~1e-6,
amplified at most ~10x when most of the mass has been rejected); BONUS_TOL covers fp32
element values summed in fp64 (relative ~1e-9 of the total).

Independently of the oracle, a chi-square test checks that the GPU's emitted tokens follow
the target distribution.
"""
import numpy as np
import pytest
import torch
from scipy.stats import chisquare

import oracle
import speculative_decoding_tree_eagle_gb300 as ts
import workloads
from gpu_helpers import dev, lib

pytestmark = pytest.mark.gpu

TRIAL_TOL = 1e-4
BONUS_TOL = 1e-7


def _random_trees(rng, B, m, V, max_kids=4):
    """Parents [B, m] (parents precede children, at most max_kids children each) and tokens
    with distinct siblings."""
    parents = np.zeros((B, m), dtype=np.int32)
    tokens = np.zeros((B, m), dtype=np.int32)
    for b in range(B):
        parents[b, 0] = -1
        tokens[b, 0] = rng.integers(0, V)
        kids = {}
        for i in range(1, m):
            while True:
                p = int(rng.integers(max(0, i - 8), i))       # recent parents: deep trees
                if len(kids.setdefault(p, [])) < max_kids:
                    break
            while True:
                t = int(rng.integers(0, V))
                if t not in [tokens[b, c] for c in kids[p]]:
                    break
            kids[p].append(i)
            parents[b, i] = p
            tokens[b, i] = t
    return parents, tokens


def _sharpen(rng, logits, parents, tokens):
    """Give one child of every node a logit ln(V) + U(-2, 3) above the row, so that the walk
    keeps it with probability ~0.1..0.9 and trees are walked several levels deep."""
    B, m, V = logits.shape
    for b in range(B):
        for u in range(m):
            kids = np.nonzero(parents[b] == u)[0]
            if len(kids):
                c = kids[rng.integers(len(kids))]
                logits[b, u, tokens[b, c]] = np.log(V) + rng.uniform(-2, 3)
    return logits


def _valid(path, alen, parents, bonus, V):
    if alen < 1 or path[0] != 0 or not (0 <= bonus < V):
        return False
    return all(parents[path[i]] == path[i - 1] for i in range(1, alen)) and (path[alen:] == -1).all()


def _run(logits, tokens, parents, uniforms, T, mode, draft=None, node_row=None, expect_ok=True):
    lib()
    status = ts.new_status(dev())
    d = lambda x: None if x is None else torch.as_tensor(x).to(dev())
    out = ts.tree_accept_sample(d(logits), d(tokens), d(parents), d(uniforms), T, q_mode=mode, draft_logp=d(draft),
                                node_row=d(node_row), status=status)
    torch.cuda.synchronize()
    if expect_ok:
        ts.check_status(status)
    return {k: v.cpu().numpy() for k, v in out.items()}, int(status.item())


def _compare(got, ref, parents, V, min_frac=0.85):
    alen, apath, bonus, mg, mb = ref
    ok = (mg > TRIAL_TOL) & (mb > BONUS_TOL)
    if min_frac is not None:
        assert ok.mean() >= min_frac, ok.mean()
    for b in range(len(alen)):
        if ok[b]:
            assert got["accept_len"][b] == alen[b], b
            np.testing.assert_array_equal(got["accept_path"][b], apath[b], err_msg=str(b))
            assert got["bonus"][b] == bonus[b], b
        else:
            assert _valid(got["accept_path"][b], got["accept_len"][b], parents[b], got["bonus"][b], V), b
    return ok


CASES = [dict(dt=torch.float32, B=16, m=40, V=1000, T=1.0),
         dict(dt=torch.float32, B=8, m=64, V=32000, T=0.7),
         dict(dt=torch.float32, B=4, m=33, V=4097, T=1.3),           # V odd: scalar loads
         dict(dt=torch.bfloat16, B=8, m=64, V=128256, T=1.0),
         dict(dt=torch.bfloat16, B=3, m=256, V=2000, T=1.0),          # largest tree
         dict(dt=torch.bfloat16, B=2, m=20, V=1003, T=2.0),           # bf16, V % 8 != 0
         dict(dt=torch.bfloat16, B=8, m=24, V=140000, T=1.0)]         # beyond one cluster: streaming kernel


@pytest.mark.parametrize("mode", ["point", "draft"])
@pytest.mark.parametrize("cfg", CASES, ids=lambda c: f"{str(c['dt'])[6:]}_B{c['B']}_m{c['m']}_V{c['V']}_T{c['T']}")
def test_random_trees_match_the_oracle(cfg, mode):
    B, m, V, T, dt = cfg["B"], cfg["m"], cfg["V"], cfg["T"], cfg["dt"]
    rng = np.random.default_rng(B * 1000 + m + V)
    parents, tokens = _random_trees(rng, B, m, V)
    logits = _sharpen(rng, rng.normal(0, 1, size=(B, m, V)).astype(np.float32), parents, tokens)
    lt = torch.from_numpy(logits).to(dt)
    uniforms = rng.random((B, m)).astype(np.float32)
    draft = node_row = None
    if mode == "draft":
        draft = torch.log_softmax(torch.from_numpy(rng.normal(0, 2, size=(B, m, V)).astype(np.float32)), -1).numpy()
        node_row = np.tile(rng.permutation(m).astype(np.int32), (B, 1))
    got, _ = _run(lt, tokens, parents, uniforms, T, mode, draft, node_row)
    ref = oracle.accept_sample(lt.float().numpy(), tokens, parents, uniforms, T, mode, draft, node_row)
    ok = _compare(got, ref, parents, V)
    if B >= 8:
        assert (ref[0][ok] > 2).any()                    # some walks went two levels deep


@pytest.mark.parametrize("mode", ["point", "draft"])
@pytest.mark.parametrize("name", ["llama2_7b", "llama3_8b_gqa", "llama2_70b_gqa"])
def test_workload_trees_from_tree_build(name, mode):
    """ts_tree_build's tree (tokens, parents, node_row) on the workload's draft rows, target
    logits with a sharpened child per node; T = 1."""
    w = workloads.WORKLOADS[name]
    inp = workloads.generate(w, with_attention=False)
    lib()
    status = ts.new_status(dev())
    tree = ts.tree_build(inp["draft_logp"].to(dev()), inp["root_tokens"].to(dev()), w.k, w.depth, w.m, status=status)
    ts.check_status(status)
    tokens = tree["tokens"].cpu().numpy()
    parents = tree["parents"].cpu().numpy()
    node_row = tree["node_row"].cpu().numpy()
    rng = np.random.default_rng(w.seed)
    logits = _sharpen(rng, inp["logits"].float().numpy().copy(), parents, tokens)
    lt = torch.from_numpy(logits).to(inp["logits"].dtype)
    draft = inp["draft_logp"].numpy() if mode == "draft" else None
    oks = []
    for _ in range(max(1, 8 // w.B)):                   # several uniform draws for small batches
        uniforms = rng.random((w.B, w.m)).astype(np.float32)
        got, _ = _run(lt, tokens, parents, uniforms, 1.0, mode, draft, node_row if mode == "draft" else None)
        ref = oracle.accept_sample(lt.float().numpy(), tokens, parents, uniforms, 1.0, mode, draft, node_row)
        oks.append(_compare(got, ref, parents, w.V, min_frac=None))
    assert np.concatenate(oks).mean() >= 0.75


def _gumbel_top(rng, logq, n, size):
    """n ids drawn without replacement from q, `size` times (the Gumbel top-n construction)."""
    g = logq[None, :] - np.log(-np.log(rng.random((size, len(logq)))))
    return np.argsort(-g, axis=1)[:, :n]


@pytest.mark.parametrize("mode,T", [("point", 1.0), ("point", 0.6), ("draft", 1.0), ("draft", 1.5)])
def test_emitted_tokens_follow_the_target(mode, T):
    """20000 sequences on one small tree: token 1 ~ p(root); token 2, given that token 1 was
    child 1's draft, ~ p(node 1).  Draft mode draws each sequence's children from q without
    replacement.  No oracle involved."""
    B, V = 20000, 12
    parents1 = np.array([-1, 0, 0, 0, 1, 1, 2, 4], dtype=np.int32)
    node_row1 = np.array([0, 1, 2, -1, 3, -1, -1, -1], dtype=np.int32)
    m = len(parents1)
    rng = np.random.default_rng(99)
    lg1 = rng.normal(0, 1.2, size=(m, V)).astype(np.float32)
    lg1[0, 1] = lg1[0].max() + 1.0     # point mode: child 1 carries token 1, kept often enough
    d1 = torch.log_softmax(torch.from_numpy(rng.normal(0, 1.2, size=(4, V)).astype(np.float32)), -1).numpy()
    tokens = np.zeros((B, m), dtype=np.int32)
    for u, row in enumerate(node_row1):
        kids = np.nonzero(parents1 == u)[0]
        if not len(kids):
            continue
        if mode == "draft":
            tokens[:, kids] = _gumbel_top(rng, d1[row].astype(np.float64), len(kids), B)
        else:
            tokens[:, kids] = [(3 * u + 2 * j + 1) % V for j in range(len(kids))]
    logits = np.broadcast_to(lg1, (B, m, V)).copy()
    parents = np.tile(parents1, (B, 1))
    uniforms = rng.random((B, m)).astype(np.float32)
    draft = np.broadcast_to(d1, (B, 4, V)).copy() if mode == "draft" else None
    node_row = np.tile(node_row1, (B, 1)) if mode == "draft" else None
    got, _ = _run(logits, tokens, parents, uniforms, T, mode, draft, node_row)
    alen, path, bonus = got["accept_len"], got["accept_path"], got["bonus"]
    first = np.where(alen >= 2, tokens[np.arange(B), np.maximum(path[:, 1], 0)], bonus)
    p0 = oracle.softmax_t(lg1[0], T)
    assert chisquare(np.bincount(first, minlength=V), p0 * B).pvalue > 1e-4
    sel = (alen >= 2) & (path[:, 1] == 1)
    second = np.where(alen[sel] >= 3, tokens[sel][np.arange(sel.sum()), np.maximum(path[sel][:, 2], 0)], bonus[sel])
    assert sel.sum() > 1000
    assert chisquare(np.bincount(second, minlength=V), oracle.softmax_t(lg1[1], T) * sel.sum()).pvalue > 1e-4


def test_low_temperature_equals_the_greedy_kernel():
    """T -> 0 with point proposals keeps exactly the greedy path: same result as ts_tree_accept."""
    B, m, V = 8, 60, 5000
    rng = np.random.default_rng(4)
    parents, tokens = _random_trees(rng, B, m, V)
    # distinct logits 0.01 apart: at T = 1e-4 every runner-up has mass 2^-144 -> 0 in fp32
    logits = (np.stack([rng.permutation(V) for _ in range(B * m)]).reshape(B, m, V) * 0.01).astype(np.float32)
    amax = logits.argmax(-1)
    for b in range(B):                          # plant: half the nodes carry their parent's argmax
        for i in range(1, m):
            sib = tokens[b][parents[b] == parents[b, i]]
            if rng.random() < 0.5 and amax[b, parents[b, i]] not in sib:
                tokens[b, i] = amax[b, parents[b, i]]
    got, _ = _run(logits, tokens, parents, rng.random((B, m)).astype(np.float32), 1e-4, "point")
    lib()
    g = ts.tree_accept(torch.from_numpy(logits).to(dev()), torch.from_numpy(tokens).to(dev()),
                       torch.from_numpy(parents).to(dev()))
    np.testing.assert_array_equal(got["accept_len"], g["accept_len"].cpu().numpy())
    np.testing.assert_array_equal(got["accept_path"], g["accept_path"].cpu().numpy())
    np.testing.assert_array_equal(got["bonus"], g["bonus"].cpu().numpy())
    assert (got["accept_len"] > 2).any()


def test_root_only_and_edge_uniforms():
    """m = 1: the step only draws.  r = 0 keeps any child with mass and draws the first id with
    mass; ids whose logit is -inf are never drawn."""
    V = 300
    lg = np.full((1, 1, V), -np.inf, dtype=np.float32)
    lg[0, 0, [7, 100, 299]] = [0.0, 1.0, 2.0]
    got, _ = _run(lg, np.zeros((1, 1), np.int32), np.full((1, 1), -1, np.int32), np.zeros((1, 1), np.float32), 1.0,
                  "point")
    assert got["accept_len"][0] == 1 and got["bonus"][0] == 7 and got["accept_path"][0, 0] == 0
    got, _ = _run(lg, np.zeros((1, 1), np.int32), np.full((1, 1), -1, np.int32),
                  np.full((1, 1), np.float32(1) - np.float32(2 ** -24)), 1.0, "point")
    assert got["bonus"][0] == 299
    lg2 = np.zeros((1, 3, V), dtype=np.float32)
    got, _ = _run(lg2, np.array([[0, 5, 6]], np.int32), np.array([[-1, 0, 0]], np.int32),
                  np.array([[0.5, 0.0, 0.0]], np.float32), 1.0, "point")
    assert got["accept_len"][0] == 2 and got["accept_path"][0, 1] == 1


def test_duplicate_sibling_tokens():
    """Two siblings with one token: after the first is rejected its mass is gone, so the
    second is rejected too (both modes), as in the oracle."""
    V = 64
    rng = np.random.default_rng(8)
    lg = rng.normal(0, 1, size=(2, 4, V)).astype(np.float32)
    lg[:, 0, 9] = -30.0                                  # the duplicated token has almost no target mass
    tokens = np.array([[0, 9, 9, 3]] * 2, np.int32)
    parents = np.array([[-1, 0, 0, 0]] * 2, np.int32)
    uniforms = np.array([[0.3, 0.999, 0.0, 0.999], [0.6, 0.999, 0.0, 0.0]], np.float32)
    d = torch.log_softmax(torch.from_numpy(rng.normal(0, 1, size=(2, 4, V)).astype(np.float32)), -1).numpy()
    nr = np.array([[0, -1, -1, -1]] * 2, np.int32)
    for mode in ("point", "draft"):
        got, _ = _run(lg, tokens, parents, uniforms, 1.0, mode, d if mode == "draft" else None,
                      nr if mode == "draft" else None)
        ref = oracle.accept_sample(lg, tokens, parents, uniforms, 1.0, mode, d, nr)
        np.testing.assert_array_equal(got["accept_len"], ref[0])
        np.testing.assert_array_equal(got["accept_path"], ref[1])
        if mode == "point":     # r = 0 keeps the third child (in draft mode its residual mass may be 0)
            assert got["accept_len"][1] == 2 and got["accept_path"][1, 1] == 3


@pytest.mark.parametrize("case", ["bad_parent", "root_parent", "bad_token", "bad_row"])
def test_bad_trees_are_reported(case):
    V, m = 50, 4
    lg = np.zeros((2, m, V), np.float32)
    tokens = np.array([[0, 1, 2, 3]] * 2, np.int32)
    parents = np.array([[-1, 0, 0, 1]] * 2, np.int32)
    d = np.log(np.full((2, 2, V), 1.0 / V, np.float32))
    nr = np.array([[0, 1, -1, -1]] * 2, np.int32)
    if case == "bad_parent":
        parents[0, 3] = 3
    elif case == "root_parent":
        parents[0, 0] = 0
    elif case == "bad_token":
        tokens[0, 2] = V
    else:
        nr[0, 1] = 2
    got, st = _run(lg, tokens, parents, np.full((2, m), 0.5, np.float32), 1.0, "draft", d, nr, expect_ok=False)
    assert st == -6
    assert got["accept_len"][0] == 0 and got["bonus"][0] == -1 and (got["accept_path"][0] == -1).all()
    assert got["accept_len"][1] >= 1 and 0 <= got["bonus"][1] < V


def test_row_without_mass_is_reported():
    V = 40
    lg = np.zeros((1, 2, V), np.float32)
    lg[0, 0] = -np.inf
    _, st = _run(lg, np.array([[0, 3]], np.int32), np.array([[-1, 0]], np.int32), np.full((1, 2), 0.5, np.float32),
                 1.0, "point", expect_ok=False)
    assert st == -6


@pytest.mark.parametrize("mode", ["point", "draft"])
def test_a_node_with_more_than_32_children(mode):
    """A star-shaped level (100 children under the root, 40 under the first child): the trials
    run in groups of 32 lanes and the children past the 32nd are fetched separately."""
    B, V = 6, 3000
    rng = np.random.default_rng(17)
    par = [-1] + [0] * 100 + [1] * 40 + list(range(101, 131))
    m = len(par)
    parents = np.tile(np.array(par, np.int32), (B, 1))
    tokens = np.zeros((B, m), np.int32)
    for b in range(B):
        for u in set(par[1:]):
            kids = [c for c in range(m) if par[c] == u]
            tokens[b, kids] = rng.choice(V, size=len(kids), replace=False)
    logits = rng.normal(0, 1, size=(B, m, V)).astype(np.float32)
    for b in range(B):                       # the kept child sits late in the sibling order
        logits[b, 0, tokens[b, 70 + b]] = np.log(V) + 2.0
        logits[b, 1, tokens[b, 101 + 35]] = np.log(V) + 1.0
    uniforms = rng.random((B, m)).astype(np.float32)
    draft = node_row = None
    if mode == "draft":
        draft = torch.log_softmax(torch.from_numpy(rng.normal(0, 1, size=(B, m, V)).astype(np.float32)), -1).numpy()
        node_row = np.tile(np.arange(m, dtype=np.int32), (B, 1))
    got, _ = _run(logits, tokens, parents, uniforms, 1.0, mode, draft, node_row)
    ref = oracle.accept_sample(logits, tokens, parents, uniforms, 1.0, mode, draft, node_row)
    ok = _compare(got, ref, parents, V, min_frac=0.8)
    assert (ref[0][ok] >= 2).any()


@pytest.mark.parametrize("V", [5, 33, 511])
def test_tiny_vocabularies(V):
    B, m = 8, 6
    rng = np.random.default_rng(V)
    parents = np.tile(np.array([-1, 0, 0, 1, 1, 2], np.int32), (B, 1))
    tokens = np.zeros((B, m), np.int32)
    for b in range(B):
        tokens[b, 1:3] = rng.choice(V, size=2, replace=False)
        tokens[b, 3:5] = rng.choice(V, size=2, replace=False)
        tokens[b, 5] = rng.integers(V)
    logits = rng.normal(0, 1.5, size=(B, m, V)).astype(np.float32)
    uniforms = rng.random((B, m)).astype(np.float32)
    for mode in ("point", "draft"):
        draft = torch.log_softmax(torch.from_numpy(rng.normal(0, 1, size=(B, m, V)).astype(np.float32)), -1).numpy()
        node_row = np.tile(np.arange(m, dtype=np.int32), (B, 1))
        got, _ = _run(logits, tokens, parents, uniforms, 1.0, mode, draft if mode == "draft" else None,
                      node_row if mode == "draft" else None)
        ref = oracle.accept_sample(logits, tokens, parents, uniforms, 1.0, mode, draft, node_row)
        _compare(got, ref, parents, V, min_frac=0.75)


def test_many_sequences():
    """300 sequences (300 clusters of 8 CTAs at V = 32000): several waves of clusters."""
    B, m, V = 300, 12, 32000
    rng = np.random.default_rng(5)
    parents, tokens = _random_trees(rng, B, m, V)
    logits = _sharpen(rng, rng.normal(0, 1, size=(B, m, V)).astype(np.float32), parents, tokens)
    lt = torch.from_numpy(logits).to(torch.bfloat16)
    uniforms = rng.random((B, m)).astype(np.float32)
    got, _ = _run(lt, tokens, parents, uniforms, 1.0, "point")
    ref = oracle.accept_sample(lt.float().numpy(), tokens, parents, uniforms, 1.0, "point")
    _compare(got, ref, parents, V, min_frac=0.9)
