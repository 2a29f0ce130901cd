"""ts_tree_accept_noalloc — the tree_accept variant for callers that cannot allocate.

Callers such as a serving engine that gives all free device memory to its KV-cache pool,
or a plugin whose host framework owns every allocation, cannot hand the library a
workspace.  The no-allocation entry point keeps its scratch in a fixed array inside the
library; these checks call it through the C ABI and compare it with the workspace-taking
entry point on two calls in a row and at the array's exact limit (outputs are integers,
so they must agree exactly).  The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import speculative_decoding_tree_eagle_gb300 as ts
from speculative_decoding_tree_eagle_gb300 import build as tsbuild

pytestmark = pytest.mark.gpu

TS_BF16, TS_ERR_UNSUPPORTED = 1, -2


def _lib():
    tsbuild.build()
    L = ts.library()
    P, I = ctypes.c_void_p, ctypes.c_int
    L.ts_tree_accept_noalloc.restype = I
    L.ts_tree_accept_noalloc.argtypes = [P, I, P, P, I, I, I, P, P, P, P, P, P]
    return L


def _case(seed, B, m, V):
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn(B, m, V, generator=g).to(torch.bfloat16)
    parents = torch.tensor([[-1] + [int(torch.randint(0, i, (1,), generator=g)) for i in range(1, m)]
                            for _ in range(B)], dtype=torch.int32)
    tokens = torch.randint(0, V, (B, m), generator=g, dtype=torch.int32)
    for b in range(B):  # make some root paths match so the accepted paths are non-trivial
        for i in range(1, m):
            if int(torch.randint(0, 2, (1,), generator=g)):
                logits[b, parents[b, i], tokens[b, i]] = 100.0
    return logits.cuda(), tokens.cuda(), parents.cuda()


def _outs(B, m):
    return [torch.full(s, -7, dtype=torch.int32, device="cuda") for s in ((B, m), (B,), (B, m), (B,))]


def test_noalloc_matches_workspace_entry_point_twice():
    L = _lib()
    stream = torch.cuda.current_stream().cuda_stream
    for seed, (B, m, V) in ((1, (4, 60, 32000)), (2, (8, 64, 128256))):
        logits, tokens, parents = _case(seed, B, m, V)
        status_a, status_b = ts.new_status(), ts.new_status()
        ref = ts.tree_accept(logits, tokens, parents, status=status_a)
        got = _outs(B, m)
        rc = L.ts_tree_accept_noalloc(logits.data_ptr(), TS_BF16, tokens.data_ptr(), parents.data_ptr(),
                                      B, m, V, *[t.data_ptr() for t in got], status_b.data_ptr(), stream)
        assert rc == 0, ts.status_string(rc)
        torch.cuda.synchronize()
        assert int(status_a.item()) == 0 and int(status_b.item()) == 0
        for key, t in zip(("argmax", "accept_len", "accept_path", "bonus"), got):
            np.testing.assert_array_equal(t.cpu().numpy(), ref[key].cpu().numpy(), err_msg=key)
        assert (got[1].cpu().numpy() > 1).any()


def test_noalloc_rejects_requests_beyond_its_scratch():
    L = _lib()
    B, m, V = 512, 256, 4096   # 131072 rows x 1 segment x 8 bytes + 256 > 1 MiB
    dummy = torch.zeros(1, dtype=torch.int32, device="cuda")
    p = dummy.data_ptr()
    rc = L.ts_tree_accept_noalloc(p, TS_BF16, p, p, B, m, V, p, p, p, p, None, None)
    assert rc == TS_ERR_UNSUPPORTED


def test_noalloc_at_its_exact_limit():
    """The largest request the 1 MiB array holds (131040 rows of one segment: 8 bytes each
    plus 256 bytes of alignment) runs and matches the workspace entry point; one more row
    is rejected."""
    L = _lib()
    stream = torch.cuda.current_stream().cuda_stream
    B, m, V = 546, 240, 2048  # 131040 rows; V = 2048 is one segment per row
    g = torch.Generator(device="cuda").manual_seed(11)
    logits = torch.randn(B, m, V, generator=g, device="cuda").to(torch.bfloat16)
    parents = (torch.rand(B, m, generator=g, device="cuda") * torch.arange(m, device="cuda")).floor().to(torch.int32)
    parents[:, 0] = -1
    tokens = logits.float().argmax(-1).to(torch.int32).gather(1, parents.clamp(min=0).long()).to(torch.int32)
    status_a, status_b = ts.new_status(), ts.new_status()
    ref = ts.tree_accept(logits, tokens, parents, status=status_a)
    got = _outs(B, m)
    rc = L.ts_tree_accept_noalloc(logits.data_ptr(), TS_BF16, tokens.data_ptr(), parents.data_ptr(),
                                  B, m, V, *[t.data_ptr() for t in got], status_b.data_ptr(), stream)
    assert rc == 0, ts.status_string(rc)
    torch.cuda.synchronize()
    assert int(status_a.item()) == 0 and int(status_b.item()) == 0
    for key, t in zip(("argmax", "accept_len", "accept_path", "bonus"), got):
        np.testing.assert_array_equal(t.cpu().numpy(), ref[key].cpu().numpy(), err_msg=key)
    assert (got[1].cpu().numpy() > 1).any()
    p = logits.data_ptr()
    rc = L.ts_tree_accept_noalloc(p, TS_BF16, p, p, B, m + 1, V, p, p, p, p, None, None)
    assert rc == TS_ERR_UNSUPPORTED
