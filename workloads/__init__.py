"""Seeded synthetic inputs for the tree-verify hot path.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no top-k, no tree construction, no attention, no argmax).
Both the fp64 CPU oracle (through the tests) and the CUDA path are fed from
here, so they see the same bits.

Recipe (one CPU ``torch.Generator`` per workload, seed ``20260 + index``, the
long-context sub-cases add ``10 * m``; tensors are drawn in this fixed order):

1. draft logits ``sigma * N(0,1)`` of shape ``[B, 1 + (depth-1)*k, V]``,
   turned into fp32 log-probabilities (the stand-in for the draft model's
   softmax output: confidence = draft softmax probability),
2. root tokens ``[B]`` uniform over the vocabulary,
3. prefix lengths ``[B]`` (fixed, or uniform in a range),
4. the physical-block permutation of the paged KV cache (identity or shuffled),
5. Q ``[B, m, Hq, d]`` ~ N(0,1),
6. K cache and 7. V cache ``[num_blocks, Hkv, block_size, d]`` ~ N(0,1),
8. target logits ``[B, m, V]`` ~ N(0,1),
9. (tiny workload only) distinct random token ids for the fixed 8-node tree.

Values are drawn in fp32 and cast with ``.to(torch.bfloat16)`` (round to
nearest even) for the bf16 workloads.  Planting a matching root path into the
target logits needs the draft tree, so it is a separate call
(:func:`plant_paths`) with its own generator (seed ``+ 7``).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional

import torch

BLOCK_SIZE = 16

# The worked 8-node tree printed on "rainlin.net/posts/eagle", section 四
# (Tree Attention): flattened order It, is, has, a, the, to, good, be.
PAGE_TREE_WORDS = ["It", "is", "has", "a", "the", "to", "good", "be"]
PAGE_TREE_PARENTS = [-1, 0, 0, 1, 1, 2, 3, 5]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    B: int
    Hq: int
    Hkv: int
    d: int
    prefix: tuple          # (lo, hi) inclusive; lo == hi for a fixed length
    m: int                 # tree nodes including the root
    V: int                 # vocabulary
    k: int                 # draft top-k
    depth: int             # draft layers below the root
    dtype: str             # "f32" or "bf16" for Q/K/V and target logits
    sigma: float           # std of the draft logits
    shuffled: bool         # shuffled physical block table
    plant_frac: float = 0.0
    fixed_tree: bool = False
    seed_extra: int = 0

    @property
    def seed(self) -> int:
        return 20260 + self.index + self.seed_extra

    @property
    def g(self) -> int:
        return self.Hq // self.Hkv

    @property
    def rows(self) -> int:
        """Draft rows fed to tree construction: the root row + k per later layer."""
        return 1 + (self.depth - 1) * self.k

    @property
    def max_prefix(self) -> int:
        return self.prefix[1]


def _long_context(m: int) -> Workload:
    chain = m == 8
    return Workload(name=f"long_context_m{m}", index=4, B=4, Hq=32, Hkv=8, d=128,
                    prefix=(32768, 32768), m=m, V=128256,
                    k=1 if chain else 10, depth=7 if chain else 8,
                    dtype="bf16", sigma=2.0, shuffled=True, seed_extra=10 * m)


WORKLOADS: Dict[str, Workload] = {
    # The pages' 8-node tree, one head, fp32 (tiny case the oracle runs in ms).
    "tiny": Workload(name="tiny", index=0, B=1, Hq=1, Hkv=1, d=64, prefix=(16, 16), m=8,
                     V=1000, k=2, depth=3, dtype="f32", sigma=1.0, shuffled=False,
                     fixed_tree=True),
    # Llama-2-7B-shaped single layer (MHA), dynamic tree k=10, depth 6, m=60.
    "llama2_7b": Workload(name="llama2_7b", index=1, B=1, Hq=32, Hkv=32, d=128,
                          prefix=(2048, 2048), m=60, V=32000, k=10, depth=6,
                          dtype="bf16", sigma=2.0, shuffled=False),
    # Llama-3-8B-shaped GQA, batch 8, ragged prefixes 1024..8192, paged + shuffled.
    "llama3_8b_gqa": Workload(name="llama3_8b_gqa", index=2, B=8, Hq=32, Hkv=8, d=128,
                              prefix=(1024, 8192), m=64, V=128256, k=10, depth=7,
                              dtype="bf16", sigma=2.0, shuffled=True),
    # Llama-2-70B-shaped GQA single layer, 30% of sequences get a planted path.
    "llama2_70b_gqa": Workload(name="llama2_70b_gqa", index=3, B=16, Hq=64, Hkv=8, d=128,
                               prefix=(4096, 4096), m=60, V=32000, k=8, depth=6,
                               dtype="bf16", sigma=2.0, shuffled=True, plant_frac=0.3),
    "long_context_m8": _long_context(8),
    "long_context_m32": _long_context(32),
    "long_context_m64": _long_context(64),
    "long_context_m128": _long_context(128),
}


def custom(name: str = "custom", **kw) -> Workload:
    """A workload with explicit sizes (used for small parity cases and edge cases)."""
    base = dict(index=100, B=1, Hq=4, Hkv=1, d=128, prefix=(40, 40), m=8, V=4096, k=2,
                depth=3, dtype="bf16", sigma=2.0, shuffled=True)
    base.update(kw)
    return Workload(name=name, **base)


def _draw_draft_logp(gen: torch.Generator, w: Workload) -> torch.Tensor:
    logits = torch.randn(w.B, w.rows, w.V, generator=gen, dtype=torch.float32) * w.sigma
    # log-probabilities of the draft distribution (input preparation, fp32)
    return torch.log_softmax(logits, dim=-1).contiguous()


def generate(w: Workload, with_attention: bool = True, with_logits: bool = True) -> Dict[str, torch.Tensor]:
    """All inputs of one verify step of workload ``w`` as CPU tensors (deterministic).

    Keys: ``draft_logp`` fp32 [B,R,V]; ``root_tokens`` int32 [B]; ``prefix_len`` int32 [B];
    ``block_table`` int32 [B, max_blocks] (-1 padded); ``num_blocks``; ``q`` [B,m,Hq,d];
    ``k_cache``/``v_cache`` [num_blocks,Hkv,16,d]; ``logits`` [B,m,V]; for the tiny workload
    also ``tree_tokens``/``tree_parents`` int32 [1,8] (the pages' fixed tree).
    Skipped tensors (``with_attention``/``with_logits`` False) are still drawn from the
    generator so that later tensors do not depend on the flags.
    """
    gen = torch.Generator().manual_seed(w.seed)
    fdt = torch.float32 if w.dtype == "f32" else torch.bfloat16
    out: Dict[str, torch.Tensor] = {}
    out["draft_logp"] = _draw_draft_logp(gen, w)
    out["root_tokens"] = torch.randint(0, w.V, (w.B,), generator=gen, dtype=torch.int64).to(torch.int32)
    lo, hi = w.prefix
    if lo == hi:
        prefix = torch.full((w.B,), lo, dtype=torch.int32)
    else:
        prefix = torch.randint(lo, hi + 1, (w.B,), generator=gen, dtype=torch.int64).to(torch.int32)
    out["prefix_len"] = prefix
    nblk = [math.ceil((int(prefix[b]) + w.m) / BLOCK_SIZE) for b in range(w.B)]
    num_blocks = sum(nblk)
    perm = torch.randperm(num_blocks, generator=gen) if w.shuffled else torch.arange(num_blocks)
    # table width covers the largest prefix the workload allows (the kernels' host-side bound)
    max_blocks = max(max(nblk), math.ceil((hi + w.m) / BLOCK_SIZE))
    table = torch.full((w.B, max_blocks), -1, dtype=torch.int32)
    off = 0
    for b in range(w.B):
        table[b, :nblk[b]] = perm[off:off + nblk[b]].to(torch.int32)
        off += nblk[b]
    out["block_table"] = table
    out["num_blocks"] = torch.tensor(num_blocks)
    qshape = (w.B, w.m, w.Hq, w.d)
    kvshape = (num_blocks, w.Hkv, BLOCK_SIZE, w.d)
    if with_attention:
        out["q"] = torch.randn(qshape, generator=gen, dtype=torch.float32).to(fdt)
        out["k_cache"] = torch.randn(kvshape, generator=gen, dtype=torch.float32).to(fdt)
        out["v_cache"] = torch.randn(kvshape, generator=gen, dtype=torch.float32).to(fdt)
    else:
        for shape in (qshape, kvshape, kvshape):
            _skip(gen, shape)
    lshape = (w.B, w.m, w.V)
    if with_logits:
        out["logits"] = torch.randn(lshape, generator=gen, dtype=torch.float32).to(fdt)
    else:
        _skip(gen, lshape)
    if w.fixed_tree:
        ids = torch.randperm(w.V, generator=gen)[: len(PAGE_TREE_PARENTS)].to(torch.int32)
        out["tree_tokens"] = ids.view(1, -1).repeat(w.B, 1)
        out["tree_parents"] = torch.tensor(PAGE_TREE_PARENTS, dtype=torch.int32).view(1, -1).repeat(w.B, 1)
    return out


def _skip(gen: torch.Generator, shape) -> None:
    # advance the generator exactly as a draw of this shape would
    torch.randn(shape, generator=gen, dtype=torch.float32)


def plant_paths(w: Workload, logits: torch.Tensor, tokens: torch.Tensor, parents: torch.Tensor,
                frac: Optional[float] = None) -> torch.Tensor:
    """Plant a matching root-to-leaf path into ``round(frac * B)`` seeded sequences.

    For each chosen sequence a leaf is picked uniformly; along its root path every
    edge (u -> v) gets ``logits[b, u, tokens[b, v]] = max(logits[b, u, :]) + 1`` so that
    the target model "agrees" with the draft along that branch.  Returns a new tensor.
    ``tokens``/``parents`` are the draft tree ([B, m] int tensors, CPU).
    """
    frac = w.plant_frac if frac is None else frac
    gen = torch.Generator().manual_seed(w.seed + 7)
    out = logits.clone()
    nplant = int(round(frac * w.B))
    if nplant == 0:
        return out
    seqs = torch.randperm(w.B, generator=gen)[:nplant].tolist()
    for b in sorted(seqs):
        par = parents[b].tolist()
        m = len(par)
        is_parent = [False] * m
        for i in range(1, m):
            is_parent[par[i]] = True
        leaves = [i for i in range(m) if not is_parent[i]]
        leaf = leaves[int(torch.randint(0, len(leaves), (1,), generator=gen))]
        v = leaf
        while par[v] != -1:
            u = par[v]
            row = out[b, u].float()
            out[b, u, int(tokens[b, v])] = (row.max() + 1.0).to(out.dtype)
            v = u
    return out
