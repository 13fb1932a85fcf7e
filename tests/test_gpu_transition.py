"""GPU parity of the residency transitions (active copy, demotion) and of the
resolve that follows them, against the oracle (bit-exact)."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu
PAGE = 64


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()
    assert torch.cuda.is_available()


class _Full:
    """A fully resident pool (every page on the GPU, no host copies yet) with a
    host arena of one block per page, and the oracle's own copy of it. Both
    host arenas start with the same seeded random bytes (and scales), so that
    a write into a block that no transition names shows up as a difference."""

    def __init__(self, w):
        import oracle
        import tiered_sparse_mla_gb300 as hs
        self.w = w
        P, hb = w.pages, w.hot_rows // PAGE
        self.page_gpu = np.arange(w.B * P, dtype=np.int32).reshape(w.B, P)
        hot = (w.B * P + np.arange(w.B * hb, dtype=np.int32)).reshape(w.B, hb)
        fp8 = w.dtype == "fp8"
        self.pool = hs.Pool(dtype=hs.HS_FP8_E4M3_ROWSCALE if fp8 else hs.HS_BF16,
                            n_gpu_blocks=w.B * (P + hb), n_host_blocks=w.B * P,
                            max_requests=w.B, max_ctx=w.ctx, max_topk=w.K, hot_rows=w.hot_rows)
        for r in range(w.B):
            self.pool.request_init(r, w.ctx)
            self.pool.page_map_range(r, 0, self.page_gpu[r], np.full(P, -1, np.int32))
            self.pool.hot_lease(r, hot[r])
        W.fill_rows(w.dtype, self.pool.gpu_rows(), self.pool.gpu_scales(), W.row_seed(w, "gpu"))
        rng = np.random.default_rng(W.row_seed(w, "host"))
        host0 = rng.integers(0, 256, size=(w.B * P * PAGE, w.row_bytes), dtype=np.uint8)
        self.pool.host_rows()[:] = host0
        hsc0 = None
        if fp8:
            hsc0 = rng.random(w.B * P * PAGE, dtype=np.float32)
            self.pool.host_scales()[:] = hsc0
        torch.cuda.synchronize()
        sc = self.pool.gpu_scales()
        self.ot = oracle.OracleTiers(
            page_gpu=self.page_gpu.copy(), page_host=np.full((w.B, P), -1, np.int32),
            hot_blocks=hot, ctx_len=np.full(w.B, w.ctx, np.int32),
            pool_rows=self.pool.gpu_rows().cpu().numpy().copy(),
            pool_scales=None if sc is None else sc.cpu().numpy().copy(),
            host_rows=host0.copy(), host_scales=None if hsc0 is None else hsc0.copy(),
            hot_rows=w.hot_rows, max_ctx=w.ctx)
        dev = "cuda"
        self.req_ids = torch.arange(w.B, dtype=torch.int32, device=dev)
        self.resolved = torch.empty((w.B, w.K), dtype=torch.int32, device=dev)
        self.gathered = torch.empty((w.B, w.K, w.row_bytes), dtype=torch.uint8, device=dev)
        self.gscale = torch.empty((w.B, w.K), dtype=torch.float32, device=dev) if fp8 else None
        self.counts = torch.empty((w.B, 3), dtype=torch.int32, device=dev)

    def page_table(self):
        t = self.pool.tables()["page_table"]
        torch.cuda.synchronize()
        t = t.cpu().numpy()
        return t[..., 0], t[..., 1]

    def check_tables(self):
        g, h = self.page_table()
        assert np.array_equal(g, self.ot.page_gpu) and np.array_equal(h, self.ot.page_host)


def _i32(a):
    return torch.tensor(np.asarray(a, np.int32), device="cuda")


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_active_copy_demote_then_resolve(dtype):
    import tiered_sparse_mla_gb300 as hs
    from _mirror import compare_resolve
    w = W.WORKLOADS["hybrid"].scaled(B=3, ctx=16384, resident_tail=2048, hot_rows=512, K=256,
                                     steps=4, tail=32, dtype=dtype)
    f = _Full(w)
    # active copy of every finished page, host block = r * pages + p
    reqs = np.repeat(np.arange(w.B), w.pages - 1)
    pages = np.tile(np.arange(w.pages - 1), w.B)
    hbs = reqs * w.pages + pages
    hs.hs_active_copy(f.pool.handle, _i32(reqs), _i32(pages), _i32(hbs))
    assert f.pool.get_error() == 0
    assert f.ot.active_copy(reqs, pages, hbs) == 0
    f.check_tables()
    # the whole host arena: the copied blocks and, untouched, every other one
    assert np.array_equal(f.pool.host_rows(), f.ot.host_rows)
    if dtype == "fp8":
        assert np.array_equal(f.pool.host_scales().view(np.uint32),
                              f.ot.host_scales.view(np.uint32))
    # demotion: request 0 to the workload's tail, 1 to nothing, 2 keeps everything
    keep = np.array([w.resident_tail, 0, w.ctx], np.int32)
    freed = torch.full((w.B, w.pages), -7, dtype=torch.int32, device="cuda")
    nfreed = torch.empty(w.B, dtype=torch.int32, device="cuda")
    hs.hs_demote_cold_pages(f.pool.handle, _i32(np.arange(w.B)), _i32(keep), freed, nfreed)
    assert f.pool.get_error() == 0
    ofreed, err = f.ot.demote(np.arange(w.B), keep)
    assert err == 0
    nf = nfreed.cpu().numpy()
    fr = freed.cpu().numpy()
    for r in range(w.B):
        assert nf[r] == len(ofreed[r]) and np.array_equal(fr[r, :nf[r]], ofreed[r])
    assert nf[0] > 0 and nf[1] == w.pages - 1 and nf[2] == 0
    f.check_tables()
    # the resolve after the transitions, bit-exact (misses now come from the host copies)
    lists = list(W.topk_lists(w))
    tot = np.zeros(3, np.int64)
    for s in range(w.steps):
        t = torch.from_numpy(lists[s]).cuda()
        f.pool.resolve_topk(f.req_ids, t, f.resolved, f.gathered, f.gscale, f.counts)
        gerr = f.pool.get_error()
        out = f.ot.resolve(np.arange(w.B), lists[s], nthreads=4)
        compare_resolve(f, f.ot, *out, gerr, s)
        tot += out[3].sum(0)
    assert tot[2] > 0 and tot[0] > 0
    f.pool.close()


def test_transition_errors():
    import oracle
    import tiered_sparse_mla_gb300 as hs
    w = W.WORKLOADS["hybrid"].scaled(B=2, ctx=4096, resident_tail=1024, hot_rows=512, K=128)
    f = _Full(w)
    # page 5 of request 0 loses its GPU block first (host bookkeeping)
    f.pool.page_map(0, 5, -1, -1)
    f.ot.page_gpu[0, 5] = -1
    reqs, pages, hbs = [2, 0, 0, 0, 1], [0, w.pages, 5, 1, 2], [0, 0, 0, w.B * w.pages, 9]
    hs.hs_active_copy(f.pool.handle, _i32(reqs), _i32(pages), _i32(hbs))
    assert f.pool.get_error() == oracle.ERR_BAD_PAGE
    assert f.ot.active_copy(reqs, pages, hbs) == oracle.ERR_BAD_PAGE
    f.check_tables()   # only (1, 2) -> 9 applied
    freed = torch.empty((2, w.pages), dtype=torch.int32, device="cuda")
    nfreed = torch.empty(2, dtype=torch.int32, device="cuda")
    hs.hs_demote_cold_pages(f.pool.handle, _i32([7, 1]), _i32([0, -5]), freed, nfreed)
    assert f.pool.get_error() == oracle.ERR_BAD_REQUEST | oracle.ERR_BAD_PAGE
    assert (nfreed.cpu().numpy() == 0).all()
    f.check_tables()
    with pytest.raises(hs.HsError):
        hs.hs_active_copy(0, _i32([0]), _i32([0]), _i32([0]))
    f.pool.close()
