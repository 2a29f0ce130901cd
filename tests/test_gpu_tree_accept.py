"""GPU tree_accept vs the fp64 oracle: bit-exact argmax, accept_len, accept_path, bonus."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_tree_eagle_gb300 as ts
import workloads
from gpu_helpers import dev, full_workload, lib, oracle_tree

pytestmark = pytest.mark.gpu


def _compare(logits_cpu: torch.Tensor, tokens, parents, logits_gpu=None):
    lib()
    status = ts.new_status(dev())
    lg = logits_gpu if logits_gpu is not None else logits_cpu.to(dev())
    tok = torch.as_tensor(np.asarray(tokens), dtype=torch.int32).to(dev())
    par = torch.as_tensor(np.asarray(parents), dtype=torch.int32).to(dev())
    got = ts.tree_accept(lg, tok, par, status=status)
    ts.check_status(status)
    amax = oracle.target_argmax(logits_cpu)
    lens, paths, bonus = oracle.accept_longest_path(np.asarray(tokens), np.asarray(parents), amax)
    np.testing.assert_array_equal(got["argmax"].cpu().numpy(), amax)
    np.testing.assert_array_equal(got["accept_len"].cpu().numpy(), lens)
    np.testing.assert_array_equal(got["accept_path"].cpu().numpy(), paths)
    np.testing.assert_array_equal(got["bonus"].cpu().numpy(), bonus)
    return got, lens


def test_tiny_fixed_tree_fp32():
    w, inp, tree = full_workload("tiny")
    _compare(inp["logits"], tree["tokens"], tree["parents"])


def test_hand_planted_worked_tree_fp32():
    """Plant It->is, is->a, a->good: accepted path [It, is, a, good], len 4."""
    w, inp, tree = full_workload("tiny")
    tokens = tree["tokens"]
    logits = inp["logits"].clone()
    for u, v in ((0, 1), (1, 3), (3, 6)):
        logits[0, u, int(tokens[0, v])] = logits[0, u].max() + 1.0
    got, lens = _compare(logits, tokens, tree["parents"])
    assert lens[0] == 4 and got["accept_path"][0, :4].tolist() == [0, 1, 3, 6]


@pytest.mark.parametrize("name", ["llama2_7b", "llama3_8b_gqa", "llama2_70b_gqa", "long_context_m8",
                                  "long_context_m128"])
@pytest.mark.parametrize("frac", [None, 1.0])
def test_workloads_full_size(name, frac):
    """Full-size logits; frac=None is the workload's own planting, 1.0 plants every sequence."""
    w = workloads.WORKLOADS[name]
    inp = workloads.generate(w, with_attention=False)
    tree = oracle_tree(inp, w)
    tok = torch.from_numpy(tree["tokens"])
    par = torch.from_numpy(tree["parents"])
    logits = workloads.plant_paths(w, inp["logits"], tok, par, frac=frac)
    got, lens = _compare(logits, tree["tokens"], tree["parents"])
    if frac == 1.0:
        assert (lens > 1).all()


@pytest.mark.parametrize("V,dtype", [(1000, torch.bfloat16), (1003, torch.bfloat16), (77, torch.float32),
                                     (4099, torch.float32), (128256, torch.bfloat16), (32000, torch.float32)])
def test_shapes_and_ties(V, dtype):
    """Quantised logits give many equal maxima: the lowest index must win."""
    g = torch.Generator().manual_seed(V)
    B, m = 3, 17
    logits = torch.round(torch.randn(B, m, V, generator=g) * 2).to(dtype)
    parents = np.array([[-1] + [int(torch.randint(0, i, (1,), generator=g)) for i in range(1, m)]
                        for _ in range(B)])
    tokens = np.array([[int(torch.randint(0, 5, (1,), generator=g)) for _ in range(m)] for _ in range(B)])
    _compare(logits, tokens, parents)


def test_unaligned_logits_scalar_path():
    B, m, V = 2, 9, 2048
    logits = torch.randn(B, m, V, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    flat = torch.empty(B * m * V + 1, dtype=torch.bfloat16, device=dev())
    gpu = flat[1:].view(B, m, V)
    gpu.copy_(logits.to(dev()))
    parents = np.tile(np.array([-1, 0, 0, 1, 1, 2, 3, 5, 7]), (B, 1))
    tokens = np.tile(np.arange(9), (B, 1))
    _compare(logits, tokens, parents, logits_gpu=gpu)


def test_duplicate_sibling_tokens_longest_wins():
    V = 64
    logits = torch.zeros(1, 4, V)
    logits[0, 0, 5] = 1.0  # root predicts 5
    logits[0, 2, 6] = 1.0  # node 2 predicts 6
    logits[0, 3, 9] = 1.0
    got, lens = _compare(logits, [[0, 5, 5, 6]], [[-1, 0, 0, 2]])
    assert lens[0] == 3 and got["accept_path"][0].tolist() == [0, 2, 3, -1]


def test_root_only_and_max_nodes():
    _compare(torch.randn(2, 1, 300), [[3], [4]], [[-1], [-1]])
    m = 256
    g = torch.Generator().manual_seed(2)
    par = [-1] + [i - 1 for i in range(1, m)]   # a chain of 256
    tok = [0] + [int(x) for x in torch.randint(0, 50, (m - 1,), generator=g)]
    logits = torch.randn(1, m, 50, generator=g)
    for i in range(1, 200):                      # make the first 199 links match
        logits[0, i - 1, tok[i]] = 10.0
    got, lens = _compare(logits, [tok], [par])
    assert lens[0] >= 200


def test_bad_parents_reported():
    lib()
    status = ts.new_status(dev())
    logits = torch.randn(2, 4, 100, device=dev())
    tok = torch.zeros(2, 4, dtype=torch.int32, device=dev())
    par = torch.tensor([[-1, 0, 0, 1], [-1, 0, 3, 1]], dtype=torch.int32, device=dev())  # 2nd: parent after child
    got = ts.tree_accept(logits, tok, par, status=status)
    assert int(status.item()) == -6
    assert got["accept_len"].tolist()[1] == 0 and got["bonus"].tolist()[1] == -1
    assert got["accept_path"][1].tolist() == [-1, -1, -1, -1]


@pytest.mark.parametrize("V,dtype", [(1000, torch.bfloat16), (4099, torch.float32), (128256, torch.bfloat16)])
def test_nan_logits_are_never_the_argmax(V, dtype):
    """Rows with NaN entries (before, at and after the maximum, a row of NaN only, NaN beside
    -inf only): the argmax is the first largest non-NaN entry, -1 for a row of NaN only."""
    lib()
    g = torch.Generator().manual_seed(V + 3)
    B, m = 2, 9
    logits = torch.round(torch.randn(B, m, V, generator=g) * 2)
    nan, inf = float("nan"), float("inf")
    logits[0, 0, : V // 2] = nan                 # NaN before the maximum
    mx = int(logits[0, 1].argmax())
    logits[0, 1, mx] = nan                       # NaN where the maximum was
    logits[0, 2, -5:] = nan                      # NaN at the end
    logits[0, 3] = nan                           # nothing but NaN
    logits[0, 4] = -inf
    logits[0, 4, ::3] = nan                      # -inf and NaN only
    logits[1, ::2, 7] = nan
    logits = logits.to(dtype)
    parents = np.tile(np.array([-1, 0, 0, 1, 1, 2, 3, 5, 7]), (B, 1))
    tokens = np.tile(np.arange(9), (B, 1))
    status = ts.new_status(dev())
    got = ts.tree_accept(logits.to(dev()), torch.as_tensor(tokens, dtype=torch.int32, device=dev()),
                         torch.as_tensor(parents, dtype=torch.int32, device=dev()), status=status)
    ts.check_status(status)
    amax = oracle.target_argmax_ignoring_nan(logits)
    assert amax[0, 3] == -1
    np.testing.assert_array_equal(got["argmax"].cpu().numpy(), amax)
    lens, paths, bonus = oracle.accept_longest_path(tokens, parents, amax)
    np.testing.assert_array_equal(got["accept_len"].cpu().numpy(), lens)
    np.testing.assert_array_equal(got["accept_path"].cpu().numpy(), paths)
    np.testing.assert_array_equal(got["bonus"].cpu().numpy(), bonus)
