"""GPU kv_commit vs the oracle: caches, block table, prefix lengths and freed pages, bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_tree_eagle_gb300 as ts
import workloads
from gpu_helpers import dev, lib

pytestmark = pytest.mark.gpu


def _case(seed, B, Hkv, d, bs, m, dtype, a_max=None):
    rng = np.random.default_rng(seed)
    L = rng.integers(0, 3 * bs, size=B)
    need = [-(-(int(l) + m) // bs) for l in L]
    max_blocks = max(need) + 2
    num_blocks = sum(need) + 3
    perm = rng.permutation(num_blocks)
    table = np.full((B, max_blocks), -1, dtype=np.int32)
    o = 0
    for b in range(B):
        table[b, :need[b]] = perm[o:o + need[b]]
        o += need[b]
    k = torch.randn(num_blocks, Hkv, bs, d, generator=torch.Generator().manual_seed(seed)).to(dtype)
    v = torch.randn(num_blocks, Hkv, bs, d, generator=torch.Generator().manual_seed(seed + 1)).to(dtype)
    a = rng.integers(1, (a_max or m) + 1, size=B).astype(np.int32)
    path = np.full((B, m), -1, dtype=np.int32)
    for b in range(B):
        rest = np.sort(rng.choice(np.arange(1, m), size=int(a[b]) - 1, replace=False))
        path[b, :a[b]] = np.concatenate([[0], rest])
    return k, v, table, L.astype(np.int32), path, a


def _run(k, v, table, L, path, a, m, bs):
    lib()
    g = dict(k=k.to(dev()), v=v.to(dev()), table=torch.from_numpy(table).to(dev()),
             plen=torch.from_numpy(L).to(dev()), path=torch.from_numpy(path).to(dev()),
             alen=torch.from_numpy(a).to(dev()))
    status = ts.new_status(dev())
    out = ts.kv_commit(g["k"], g["v"], g["table"], g["plen"], g["path"], g["alen"], status=status)
    torch.cuda.synchronize()
    ref = oracle.kv_commit(k.float().numpy() if k.dtype != torch.bfloat16 else k.view(torch.int16).numpy(),
                           v.float().numpy() if v.dtype != torch.bfloat16 else v.view(torch.int16).numpy(),
                           table, L, path, a, m, bs)
    return g, out, status, ref


def _compare(g, out, ref, dtype):
    rk, rv, rt, rl, rf, rc, bad = ref
    gk = g["k"].cpu().view(torch.int16).numpy() if dtype == torch.bfloat16 else g["k"].cpu().numpy()
    gv = g["v"].cpu().view(torch.int16).numpy() if dtype == torch.bfloat16 else g["v"].cpu().numpy()
    np.testing.assert_array_equal(gk, rk)
    np.testing.assert_array_equal(gv, rv)
    np.testing.assert_array_equal(g["table"].cpu().numpy(), rt)
    np.testing.assert_array_equal(g["plen"].cpu().numpy(), rl)
    np.testing.assert_array_equal(out["freed_count"].cpu().numpy(), rc)
    np.testing.assert_array_equal(out["freed_blocks"].cpu().numpy(), rf)
    return bad


CASES = [dict(B=3, Hkv=2, d=128, bs=16, m=60, dtype=torch.bfloat16),
         dict(B=2, Hkv=8, d=128, bs=16, m=64, dtype=torch.bfloat16, a_max=8),
         dict(B=4, Hkv=32, d=128, bs=16, m=60, dtype=torch.bfloat16, a_max=7),
         dict(B=2, Hkv=2, d=64, bs=4, m=20, dtype=torch.bfloat16),
         dict(B=2, Hkv=3, d=96, bs=32, m=40, dtype=torch.float32),
         dict(B=3, Hkv=1, d=6, bs=8, m=30, dtype=torch.float32),       # 24-byte rows: 4-byte columns
         dict(B=1, Hkv=2, d=128, bs=16, m=256, dtype=torch.bfloat16)]  # paths up to 256 rows


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: f"B{c['B']}_H{c['Hkv']}_d{c['d']}_bs{c['bs']}_m{c['m']}_{str(c['dtype'])[6:]}")
def test_random_paths_match_the_oracle(cfg):
    cfg = dict(cfg)
    dtype, bs, m = cfg.pop("dtype"), cfg["bs"], cfg["m"]
    for seed in range(3):
        k, v, table, L, path, a = _case(seed, dtype=dtype, **cfg)
        g, out, status, ref = _run(k, v, table, L, path, a, m, bs)
        ts.check_status(status)
        assert not _compare(g, out, ref, dtype).any()


def test_a_source_that_is_also_a_later_destination():
    """path [0, 2, 5]: row 2 moves to 1 and row 5 moves to 2, so row 2 must be read first."""
    k, v, table, L, path, a = _case(7, B=1, Hkv=4, d=128, bs=16, m=8, dtype=torch.bfloat16)
    path[0, :] = -1
    path[0, :3] = [0, 2, 5]
    a[0] = 3
    g, out, status, ref = _run(k, v, table, L, path, a, 8, 16)
    ts.check_status(status)
    _compare(g, out, ref, torch.bfloat16)


@pytest.mark.parametrize("case", ["len0", "len_over_m", "not_root", "not_increasing", "bad_page", "negative_prefix",
                                  "huge_prefix"])
def test_contract_breaks_are_reported_and_leave_the_sequence_untouched(case):
    k, v, table, L, path, a = _case(3, B=2, Hkv=2, d=128, bs=16, m=12, dtype=torch.bfloat16)
    if case == "len0":
        a[0] = 0
    elif case == "len_over_m":
        a[0] = 13
    elif case == "not_root":
        a[0] = 3
        path[0, :3] = [1, 2, 3]
    elif case == "not_increasing":
        a[0] = 3
        path[0, :3] = [0, 4, 2]
    elif case == "bad_page":
        table[0, int(L[0]) // 16] = 1000
    elif case == "negative_prefix":
        L[0] = -4
    else:
        L[0] = 2**31 - 5
    g, out, status, ref = _run(k, v, table, L, path, a, 12, 16)
    assert int(status.item()) == -6
    bad = _compare(g, out, ref, torch.bfloat16)
    assert bad[0] and not bad[1]


def test_after_a_full_verify_step():
    """tree_build -> tree_attention -> tree_accept -> kv_commit on the Llama-2-70B-shaped GQA
    workload (30% of the sequences get a planted accepted path); the commit matches the oracle
    applied to the same caches, table and accepted paths."""
    w = workloads.WORKLOADS["llama2_70b_gqa"]
    inp = workloads.generate(w)
    lib()
    d = {n: inp[n].to(dev()) for n in ("draft_logp", "root_tokens", "q", "k_cache", "v_cache", "block_table",
                                        "prefix_len")}
    status = ts.new_status(dev())
    tree = ts.tree_build(d["draft_logp"], d["root_tokens"], w.k, w.depth, w.m, status=status)
    logits = workloads.plant_paths(w, inp["logits"], tree["tokens"].cpu(), tree["parents"].cpu()).to(dev())
    ts.tree_attention(d["q"], d["k_cache"], d["v_cache"], d["block_table"], d["prefix_len"],
                      tree["mask"], max_prefix=w.max_prefix, status=status)
    acc = ts.tree_accept(logits, tree["tokens"], tree["parents"], status=status)
    ts.check_status(status)
    a = acc["accept_len"].cpu().numpy()
    assert (a > 1).any()
    path = acc["accept_path"].cpu().numpy()
    k0 = d["k_cache"].cpu().view(torch.int16).numpy()
    v0 = d["v_cache"].cpu().view(torch.int16).numpy()
    t0 = d["block_table"].cpu().numpy()
    L0 = d["prefix_len"].cpu().numpy()
    out = ts.kv_commit(d["k_cache"], d["v_cache"], d["block_table"], d["prefix_len"], acc["accept_path"],
                       acc["accept_len"], status=status)
    ts.check_status(status)
    rk, rv, rt, rl, rf, rc, bad = oracle.kv_commit(k0, v0, t0, L0, path, a, w.m, workloads.BLOCK_SIZE)
    assert not bad.any()
    np.testing.assert_array_equal(d["k_cache"].cpu().view(torch.int16).numpy(), rk)
    np.testing.assert_array_equal(d["v_cache"].cpu().view(torch.int16).numpy(), rv)
    np.testing.assert_array_equal(d["block_table"].cpu().numpy(), rt)
    np.testing.assert_array_equal(d["prefix_len"].cpu().numpy(), rl)
    np.testing.assert_array_equal(out["freed_count"].cpu().numpy(), rc)
    np.testing.assert_array_equal(out["freed_blocks"].cpu().numpy(), rf)
