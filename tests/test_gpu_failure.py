"""Failure detection on the GPU without a fault: a bounded wait that nothing completes gives
up after its limit, reports TS_ERR_TIMEOUT through the status word and returns; the context
stays usable for the next call."""
import time

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_tree_eagle_gb300 as ts
from gpu_helpers import dev, lib

pytestmark = pytest.mark.gpu

TS_ERR_TIMEOUT = -5


def _run(mode):
    L = lib()
    status = ts.new_status(dev())
    result = torch.full((2,), -1, dtype=torch.int32, device=dev())
    t0 = time.time()
    rc = L.ts_selftest_bounded_wait(mode, result.data_ptr(), status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return rc, int(status.item()), result.cpu().tolist(), time.time() - t0


def test_a_wait_that_nothing_completes_times_out_and_reports():
    rc, st, res, dt = _run(0)
    assert rc == 0
    assert st == TS_ERR_TIMEOUT
    assert res == [0, 0]              # one wait gave up, the other left on the abort flag
    assert 1.5 < dt < 30.0            # the 2 s limit, not a hang
    # the context is still usable: a verification step afterwards is correct
    g = torch.Generator().manual_seed(1)
    logits = torch.randn(2, 8, 500, generator=g)
    parents = torch.tensor([[-1, 0, 0, 1, 1, 2, 3, 5]] * 2, dtype=torch.int32)
    tokens = torch.randint(0, 500, (2, 8), generator=g).to(torch.int32)
    status = ts.new_status(dev())
    out = ts.tree_accept(logits.to(dev()), tokens.to(dev()), parents.to(dev()), status=status)
    ts.check_status(status)
    ref = oracle.accept_longest_path(tokens.numpy(), parents.numpy(), oracle.target_argmax(logits))
    np.testing.assert_array_equal(out["bonus"].cpu().numpy(), ref[2])


def test_a_completed_wait_returns_at_once():
    rc, st, res, dt = _run(1)
    assert rc == 0 and st == 0 and res == [1, 1] and dt < 1.5
