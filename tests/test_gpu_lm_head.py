"""GPU fused LM-head argmax vs the oracle.

Small-integer inputs make every fp32 partial sum exact, so the argmax (ties -> first index)
and the maximum must match the fp64 oracle exactly.  For Gaussian inputs the chosen logit
must lie within the fp32 accumulation bound of the row maximum, and the index must match
wherever the top-2 gap exceeds twice that bound.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_tree_eagle_gb300 as ts
from gpu_helpers import dev, lib

pytestmark = pytest.mark.gpu


def _ints(shape, seed, lo=-3, hi=3):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(lo, hi + 1, shape, generator=g).to(torch.bfloat16)


def _run(h, w):
    lib()
    status = ts.new_status(dev())
    out = ts.lm_head_argmax(h.to(dev()), w.to(dev()), status=status)
    ts.check_status(status)
    return out["argmax"].cpu().numpy(), out["max_logit"].cpu().numpy()


# (M, N, K): one and several row tiles, vocabulary tails, K tails, tiny and large K
SHAPES = [(5, 1000, 64), (130, 777, 200), (256, 513, 8), (1, 256, 128), (60, 32000, 4096), (300, 5003, 136)]


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_integer_inputs_are_exact(M, N, K):
    h = _ints((M, K), M * 7 + N)
    w = _ints((N, K), N * 3 + K)
    got_i, got_v = _run(h, w)
    ref_i, ref_v = oracle.lm_head_argmax(h, w)
    np.testing.assert_array_equal(got_i, ref_i)
    np.testing.assert_array_equal(got_v.astype(np.float64), ref_v)


def test_ties_across_vocabulary_tiles_go_to_the_first_index():
    M, N, K = 70, 1300, 96
    h = _ints((M, K), 1)
    w = _ints((N, K), 2, lo=-1, hi=1)
    big = (h.float().sign() * 3).to(torch.bfloat16)          # logit 3 * sum|h| beats every +-1 row
    for r0, cols in ((0, (17, 300)), (1, (255, 256)), (2, (1299, 40)), (3, (512, 513, 1024))):
        for c in cols:
            w[c] = big[r0]
    got_i, _ = _run(h, w)
    ref_i, _ = oracle.lm_head_argmax(h, w)
    np.testing.assert_array_equal(got_i, ref_i)
    assert got_i[0] == 17 and got_i[1] == 255 and got_i[2] == 40 and got_i[3] == 512


@pytest.mark.parametrize("M,N,K", [(60, 32000, 4096), (64, 50000, 4096)])
def test_gaussian_inputs_within_the_fp32_bound(M, N, K):
    g = torch.Generator().manual_seed(M + N)
    h = torch.randn(M, K, generator=g).to(torch.bfloat16)
    w = (torch.randn(N, K, generator=g) * 0.05).to(torch.bfloat16)
    got_i, got_v = _run(h, w)
    logits = oracle.lm_head_logits(h, w)
    ref_i = np.argmax(logits, axis=1)
    ref_v = logits[np.arange(M), ref_i]
    tol = oracle.fp32_error_bound(h, w)
    chosen = logits[np.arange(M), got_i]
    assert (chosen >= ref_v - 2 * tol).all()
    assert (np.abs(got_v - ref_v) <= tol).all()
    top2 = np.sort(logits, axis=1)[:, -2]
    clear = ref_v - top2 > 2 * tol
    np.testing.assert_array_equal(got_i[clear], ref_i[clear])


def test_tree_accept_from_hidden_states():
    """The fused path feeds the acceptance walk: same result as the oracle walk on the
    oracle's argmax (integer inputs, so the argmax is exact)."""
    B, m, K, V = 3, 60, 256, 2048
    h = _ints((B, m, K), 5)
    w = _ints((V, K), 6)
    amax, _ = oracle.lm_head_argmax(h.view(B * m, K), w)
    amax = amax.reshape(B, m)
    rng = np.random.default_rng(1)
    parents = np.zeros((B, m), dtype=np.int32)
    tokens = np.zeros((B, m), dtype=np.int32)
    for b in range(B):
        parents[b, 0] = -1
        for i in range(1, m):
            p = int(rng.integers(0, i))
            parents[b, i] = p
            # half the nodes carry their parent's argmax, so accepted paths are long
            tokens[b, i] = amax[b, p] if rng.random() < 0.5 else (amax[b, p] + 1 + i) % V
    lib()
    status = ts.new_status(dev())
    out = ts.tree_accept_hidden(h.to(dev()), w.to(dev()), torch.from_numpy(tokens).to(dev()),
                                torch.from_numpy(parents).to(dev()), status=status)
    ts.check_status(status)
    ref = oracle.accept_longest_path(tokens, parents, amax)
    np.testing.assert_array_equal(out["argmax"].cpu().numpy(), amax)
    np.testing.assert_array_equal(out["accept_len"].cpu().numpy(), ref[0])
    np.testing.assert_array_equal(out["accept_path"].cpu().numpy(), ref[1])
    np.testing.assert_array_equal(out["bonus"].cpu().numpy(), ref[2])
    assert (ref[0] > 1).any()
