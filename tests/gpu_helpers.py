"""Helpers shared by the GPU parity tests (imported by test files only)."""
from __future__ import annotations

import functools
import math

import numpy as np
import torch

import oracle
import speculative_decoding_tree_eagle_gb300 as ts
import workloads
from speculative_decoding_tree_eagle_gb300 import build as tsbuild

BF16_ABS, BF16_REL = 2e-2, 1e-2      # |err| <= 2e-2 or <= 1e-2 |ref|  (bf16 in, fp32 accumulate)
F32_ABS = 1e-5                       # fp32 inputs


@functools.lru_cache(maxsize=None)
def lib():
    tsbuild.build()
    return ts.library()


def dev():
    return torch.device("cuda:0")


def to_dev(d):
    return {k: (v.to(dev()) if torch.is_tensor(v) else v) for k, v in d.items()}


def words_i64(words_u64: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(words_u64).view(np.int64)).to(dev())


def assert_attention_close(out_gpu: torch.Tensor, ref: np.ndarray, dtype: torch.dtype, where=None):
    got = out_gpu.detach().double().cpu().numpy()
    if where is not None:
        got = np.stack([got[b, i, h] for (b, i, h) in where])
        ref = np.stack([ref[b, i, h] for (b, i, h) in where])
    assert np.isfinite(got).all(), "non-finite attention output"
    diff = np.abs(got - ref)
    if dtype == torch.float32:
        assert diff.max() <= F32_ABS, f"max abs error {diff.max()}"
    else:
        ok = (diff <= BF16_ABS) | (diff <= BF16_REL * np.abs(ref))
        assert ok.all(), f"{(~ok).sum()} elements out of tolerance, max abs error {diff.max()}"


def oracle_tree(inp, w):
    return oracle.tree_build(inp["draft_logp"].numpy(), inp["root_tokens"].numpy(), w.k, w.depth, w.m)


@functools.lru_cache(maxsize=4)
def full_workload(name: str):
    """Inputs + oracle tree of a named workload (cached across the test module)."""
    w = workloads.WORKLOADS[name]
    inp = workloads.generate(w)
    if w.fixed_tree:
        par = inp["tree_parents"].numpy()
        mask = np.stack([oracle.ancestor_mask(p) for p in par])
        tree = dict(tokens=inp["tree_tokens"].numpy(), parents=par, mask=mask,
                    mask_words=np.stack([oracle.mask_to_words(mb) for mb in mask]))
    else:
        tree = oracle_tree(inp, w)
    return w, inp, tree


def sample_rows(w, rng, n=48):
    """(b, i, h) triples: corners plus random ones."""
    pts = {(0, 0, 0), (w.B - 1, w.m - 1, w.Hq - 1), (0, w.m - 1, 0), (w.B - 1, 0, w.Hq - 1)}
    while len(pts) < n:
        pts.add((int(rng.integers(w.B)), int(rng.integers(w.m)), int(rng.integers(w.Hq))))
    return sorted(pts)


def scale_of(w):
    return 1.0 / math.sqrt(w.d)
