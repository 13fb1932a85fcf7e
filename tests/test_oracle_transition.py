"""Pins of the oracle's residency transitions (active copy, demotion), CPU only.

Each check is fixed by something other than the transition code itself: the
"tail" residency layout the workloads define, the page table's meaning as read
by the (separately pinned) resolve, and plain invariants."""
import numpy as np
import pytest
import torch

import workloads as W

PAGE = 64


@pytest.fixture(scope="module")
def O():
    import oracle
    oracle.build()
    return oracle


def _full_resident(O, w, with_host_arena=True):
    """Every page of every request resident (GPU blocks in request order), no
    host copies yet; the oracle's own writable host arena of one block per page."""
    P = w.pages
    page_gpu = np.arange(w.B * P, dtype=np.int32).reshape(w.B, P)
    page_host = np.full((w.B, P), -1, np.int32)
    hb = w.hot_rows // PAGE
    hot = (w.B * P + np.arange(w.B * hb, dtype=np.int32)).reshape(w.B, hb)
    n_gpu = w.B * P + w.B * hb
    fp8 = w.dtype == "fp8"
    rows = torch.zeros((n_gpu * PAGE, w.row_bytes), dtype=torch.uint8)
    sc = torch.zeros(n_gpu * PAGE) if fp8 else None
    W.fill_rows(w.dtype, rows, sc, W.row_seed(w, "gpu"))
    host = np.zeros((w.B * P * PAGE, w.row_bytes), np.uint8)
    hsc = np.zeros(w.B * P * PAGE, np.float32) if fp8 else None
    return O.OracleTiers(page_gpu=page_gpu, page_host=page_host, hot_blocks=hot,
                         ctx_len=np.full(w.B, w.ctx, np.int32), pool_rows=rows.numpy().copy(),
                         pool_scales=None if sc is None else sc.numpy().copy(), host_rows=host,
                         host_scales=hsc, hot_rows=w.hot_rows, max_ctx=w.ctx)


def _copy_finished(O, ot, w):
    """Active copy of every finished page (all but the last) to host block = page index."""
    reqs, pages, hbs = [], [], []
    for r in range(w.B):
        for p in range(w.pages - 1):
            reqs.append(r), pages.append(p), hbs.append(r * w.pages + p)
    return ot.active_copy(reqs, pages, hbs)


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_demotion_to_the_tail_gives_the_hybrid_layout(O, dtype):
    """Demoting a fully resident, actively copied request to its last T tokens
    leaves exactly the pages the workloads' hybrid ("tail") residency keeps."""
    w = W.WORKLOADS["hybrid"].scaled(B=3, ctx=16384, resident_tail=4096, hot_rows=512, K=256,
                                     dtype=dtype)
    ot = _full_resident(O, w)
    assert _copy_finished(O, ot, w) == 0
    before = ot.page_gpu.copy()
    freed, err = ot.demote(np.arange(w.B), np.full(w.B, w.resident_tail))
    assert err == 0
    want = w.resident_pages()
    for r in range(w.B):
        assert np.array_equal(ot.page_gpu[r] >= 0, want), r
        gone = np.nonzero((before[r] >= 0) & (ot.page_gpu[r] < 0))[0]
        assert np.array_equal(freed[r], before[r, gone])   # ascending page order
    # again: nothing left to free
    freed2, err2 = ot.demote(np.arange(w.B), np.full(w.B, w.resident_tail))
    assert err2 == 0 and all(len(f) == 0 for f in freed2)


def test_pages_without_host_copy_stay(O):
    w = W.WORKLOADS["hybrid"].scaled(B=2, ctx=8192, resident_tail=1024, hot_rows=512, K=128)
    ot = _full_resident(O, w)
    # copy only the even pages of request 0, nothing of request 1
    ev = np.arange(0, w.pages - 1, 2)
    assert ot.active_copy(np.zeros_like(ev), ev, ev) == 0
    freed, err = ot.demote([0, 1], [0, 0])
    assert err == 0
    assert np.array_equal(np.nonzero(ot.page_gpu[0] < 0)[0], ev)
    assert (ot.page_gpu[1] >= 0).all() and len(freed[1]) == 0


def test_active_copy_copies_rows_and_rejects_bad_triples(O):
    w = W.WORKLOADS["hybrid"].scaled(B=2, ctx=4096, resident_tail=1024, hot_rows=512, K=128,
                                     dtype="fp8")
    ot = _full_resident(O, w)
    assert ot.active_copy([1], [3], [7]) == 0
    gb = ot.page_gpu[1, 3]
    assert np.array_equal(ot.host_rows[7 * PAGE:8 * PAGE], ot.pool_rows[gb * PAGE:(gb + 1) * PAGE])
    assert np.array_equal(ot.host_scales[7 * PAGE:8 * PAGE], ot.pool_scales[gb * PAGE:(gb + 1) * PAGE])
    assert ot.page_host[1, 3] == 7 and (ot.page_host >= 0).sum() == 1
    host0 = ot.host_rows.copy()
    ot.page_gpu[0, 5] = -1
    bad = ot.active_copy([2, 0, 0, 0], [0, w.pages, 5, 1], [0, 0, 0, w.B * w.pages])
    assert bad == O.ERR_BAD_PAGE
    assert np.array_equal(ot.host_rows, host0) and (ot.page_host >= 0).sum() == 1
    _, err = ot.demote([5, 0], [0, -1])
    assert err == O.ERR_BAD_REQUEST | O.ERR_BAD_PAGE


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_demoted_rows_resolve_to_the_same_bytes(O, dtype):
    """After active copy and demotion, the resolve (pinned separately) serves
    every selected row with the bytes it had while resident: the copy went to
    the right host block and the table names it."""
    w = W.WORKLOADS["hybrid"].scaled(B=2, ctx=8192, resident_tail=1024, hot_rows=512, K=128,
                                     steps=3, tail=16, dtype=dtype)
    lists = list(W.topk_lists(w))
    ref = _full_resident(O, w)
    ot = _full_resident(O, w)
    assert _copy_finished(O, ot, w) == 0
    freed, err = ot.demote(np.arange(w.B), np.full(w.B, w.resident_tail))
    assert err == 0 and sum(len(f) for f in freed) > 0
    for s in range(w.steps):
        r0, g0, sc0, c0, e0 = ref.resolve(np.arange(w.B), lists[s])
        r1, g1, sc1, c1, e1 = ot.resolve(np.arange(w.B), lists[s])
        assert e0 == 0 and e1 == 0
        assert np.array_equal(g0, g1)
        if sc0 is not None:
            assert np.array_equal(sc0.view(np.uint32), sc1.view(np.uint32))
        assert c1[:, 2].sum() > 0 or s > 0   # misses after demotion
        assert (c0.sum(1) == c1.sum(1)).all()
