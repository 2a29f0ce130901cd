"""Oracle: per-row argmax of the target LM head (TEST INFRASTRUCTURE ONLY).

Sources (web pages, by title and section):

* "jialefu.github.io — EAGLE-4 efficient LM head", section "A variant based on local Top-k":
  the selection is fused with the vocabulary-tile matrix multiplication; for the greedy
  check only the top-1 of each row is needed.
* "lesty.tech — EAGLE-2 vs. Medusa", section 4: the greedy acceptance compares each draft
  token with the base model's argmax.

Definition: logits[r, n] = sum_k hidden[r, k] * weight[n, k] in fp64 from the exact bf16
inputs (a library matrix product is the step); argmax[r] = the first n of the row maximum
(numpy's argmax returns the first maximum); max_logit[r] = that value.  The kernel
accumulates in fp32 in the tensor cores' order, so the decision is taken in the same
precision only when every partial sum is exact in fp32 (small-integer inputs, as the exact
tests use); otherwise its choice is checked against this definition within the fp32
accumulation error bound.

Pins (tests/test_oracle_lm_head.py): explicit triple loops on tiny inputs, ties to the first
index, and the composition with the acceptance walk equals the acceptance walk on the
explicitly computed logits.
"""
from __future__ import annotations

import numpy as np


def _as_f64(x):
    if hasattr(x, "detach"):
        import torch
        return x.detach().to(torch.float64).cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def lm_head_logits(hidden, weight) -> np.ndarray:
    """[M, K] x [N, K] -> fp64 [M, N]."""
    return _as_f64(hidden) @ _as_f64(weight).T


def lm_head_argmax(hidden, weight):
    """Returns (argmax int64 [M], max_logit fp64 [M])."""
    logits = lm_head_logits(hidden, weight)
    idx = np.argmax(logits, axis=1)
    return idx.astype(np.int64), logits[np.arange(logits.shape[0]), idx]


def fp32_error_bound(hidden, weight) -> np.ndarray:
    """Per-row bound on |fp32-accumulated logit - exact logit| for any summation order:
    K * 2^-23 * max_n sum_k |h_k w_nk| (each of the K additions rounds once, relative 2^-24,
    doubled for safety)."""
    h = np.abs(_as_f64(hidden))
    w = np.abs(_as_f64(weight))
    K = h.shape[1]
    return K * 2.0 ** -23 * (h @ w.T).max(axis=1)
