"""Failure detection without a GPU fault: a bounded device wait that nothing
completes gives up, reports HS_DEVERR_TIMEOUT through the pool's error word,
and the context stays usable (a resolve step afterwards still matches)."""
import time

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    import __graft_entry__ as g
    g.build()
    import tiered_sparse_mla_gb300 as hs
    from harness import GpuWorkload
    w = W.WORKLOADS["tiny"].scaled(steps=1)
    gw = GpuWorkload(w)
    assert gw.pool.get_error() == 0
    t0 = time.perf_counter()
    gw.pool.check_bounded_wait(20000)  # 20 ms
    err = gw.pool.get_error()  # synchronises
    dt = time.perf_counter() - t0
    assert err == hs.HS_DEVERR_TIMEOUT
    assert 0.015 < dt < 5.0
    assert gw.pool.get_error() == 0  # cleared by the read
    # the context is still usable
    gw.resolve(0)
    torch.cuda.synchronize()
    assert gw.pool.get_error() == 0
    assert (gw.counts.cpu().numpy().sum(axis=1) == w.K).all()
    with pytest.raises(hs.HsError):
        gw.pool.check_bounded_wait(0)
    gw.pool.close()
