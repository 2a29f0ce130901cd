"""fp64 CPU oracle for the tree-verify hot path — TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously-correct numpy restatements of what the pages define:

* :mod:`oracle.tree_build`   — EAGLE-2 dynamic draft tree (expansion, rerank,
  flatten) and the ancestor mask ("rainlin.net/posts/eagle", sections 7.1, 7.2
  and 四; "lesty.tech EAGLE-2 vs. Medusa", section 5).
* :mod:`oracle.tree_attention` — tree attention over a paged KV prefix
  ("rainlin.net/posts/eagle", section 四 Tree Attention; "lesty.tech", sections 5 and 8).
* :mod:`oracle.tree_accept`  — greedy acceptance of the longest matching root path
  ("lesty.tech", section 4; "rainlin.net/posts/eagle", sections 3.2 and 四).
* :mod:`oracle.kv_commit`    — keep the accepted path's K/V rows and release the rejected
  scratch pages ("lesty.tech", section 8).
* :mod:`oracle.lm_head`      — the target LM head's per-row argmax ("jialefu.github.io —
  EAGLE-4 efficient LM head", local Top-k section; "lesty.tech", section 4).
* :mod:`oracle.efficient_head` — the draft's two-stage efficient LM head (low-rank scores,
  local top-k per vocabulary tile, exact logits of the candidates; same page).
* :mod:`oracle.accept_sample` — verification at T > 0 by multi-round rejection sampling
  ("lesty.tech", section 4).
* :mod:`oracle.tree_prune`   — cost-aware pruning of the tree before verification (same
  page, EAGLE-Harness section; "rainlin.net/posts/eagle", sections 7.1 and 六).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding) never imports, links or calls it, and it shares no code with
the product: the only common module is the seeded input generator
``workloads`` (no method arithmetic there).

Parity status of each function is stated in its module header.
"""
from .tree_build import row_topk, tree_build, ancestor_mask, mask_to_words, words_to_mask  # noqa: F401
from .tree_attention import tree_attention  # noqa: F401
from .tree_accept import target_argmax, target_argmax_ignoring_nan, accept_longest_path  # noqa: F401
from .kv_commit import kv_commit  # noqa: F401
from .lm_head import lm_head_logits, lm_head_argmax, fp32_error_bound  # noqa: F401
from .efficient_head import candidates, efficient_head  # noqa: F401
from .accept_sample import accept_sample, softmax_t  # noqa: F401
from .tree_prune import tree_prune  # noqa: F401
