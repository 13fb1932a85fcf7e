"""GPU parity of the fused resolve kernel against the oracle (bit-exact).

Same seeded inputs on both sides; per step every resolved row id, every
gathered byte and scale, the (resident, hot, miss) counts, the device error
bits and the whole hot-buffer state (slot_tag, slot_stamp, pos_to_slot, clock)
must be identical. The GPU's extra LRU order must equal argsort(stamp, slot).
"""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _run(w, steps=None, nthreads=4, topk_override=None, in_place=False):
    from harness import GpuWorkload
    from _mirror import compare_resolve, oracle_mirror
    gw = GpuWorkload(w, in_place=in_place)
    ot = oracle_mirror(gw)
    lists = gw.topk_host if topk_override is None else topk_override
    n = len(lists) if steps is None else min(steps, len(lists))
    tot = np.zeros(3, np.int64)
    for s in range(n):
        t = torch.from_numpy(np.ascontiguousarray(lists[s])).cuda()
        gw.resolve(s, topk=t)
        err = gw.pool.get_error()
        out = ot.resolve(np.arange(w.B), lists[s], nthreads=nthreads)
        compare_resolve(gw, ot, *out, err, s)
        tot += out[3].sum(axis=0)
    gw.pool.close()
    return tot


SMALL = {
    "tiny": W.WORKLOADS["tiny"],
    "resident": W.WORKLOADS["resident"].scaled(B=3, ctx=16384, steps=3),
    "hybrid": W.WORKLOADS["hybrid"].scaled(B=3, ctx=65536, resident_tail=8192, steps=8),
    "hybrid_ragged": W.WORKLOADS["hybrid"].scaled(B=2, ctx=32768, resident_tail=4096, K=1000,
                                                   hot_rows=2048, tail=100, steps=6),
    "noresident": W.WORKLOADS["noresident"].scaled(B=4, ctx=65536, steps=5),
    "noresident_small_k": W.WORKLOADS["noresident"].scaled(B=5, ctx=4096, K=37, hot_rows=128,
                                                            steps=7),
    # more miss rows per CTA than its shared memory stages: the rest are read
    # from the host directly
    "noresident_bf16": W.WORKLOADS["noresident"].scaled(B=2, ctx=32768, dtype="bf16", steps=3),
    # a hot buffer of 8,192 slots: rank 0 ranks its LRU order in two chunks of
    # 4,096 (eight rows of 512 flags each)
    "noresident_big_hot": W.WORKLOADS["noresident"].scaled(B=2, ctx=65536, hot_rows=8192, steps=5),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_resolve_parity_small(name):
    tot = _run(SMALL[name])
    assert tot.sum() > 0


@pytest.mark.parametrize("name", list(SMALL))
def test_resolve_in_place_parity_small(name):
    """No gathered buffer: the same ids, counts and LRU state, and every
    resolved pool row holds the bytes the oracle gathered (misses copied from
    the host arena straight into their hot slots)."""
    tot = _run(SMALL[name], in_place=True)
    assert tot.sum() > 0


@pytest.mark.parametrize("name,steps", [("resident", 2), ("hybrid", 3), ("noresident", 2)])
def test_resolve_parity_full_size(name, steps):
    """The full-size workloads, first steps, every request compared."""
    tot = _run(W.WORKLOADS[name], steps=steps, nthreads=16)
    assert tot.sum() == W.WORKLOADS[name].B * W.WORKLOADS[name].K * steps


def _run_union(w, steps, in_place=False, nthreads=8, lists=None):
    """Per-token lists resolved as one union per request, against the oracle's
    union resolve of the same concatenated lists."""
    from harness import GpuWorkload
    from _mirror import compare_resolve, oracle_mirror
    gw = GpuWorkload(w, in_place=in_place, per_token=True, build_topk=lists is None)
    ot = oracle_mirror(gw)
    lists = gw.topk_host if lists is None else lists
    tot = np.zeros(3, np.int64)
    for s in range(steps):
        flat = np.ascontiguousarray(lists[s].reshape(w.B, -1))
        gw.resolve(s, topk=torch.from_numpy(flat).cuda())
        err = gw.pool.get_error()
        out = ot.resolve(np.arange(w.B), flat, nthreads=nthreads, union=True)
        compare_resolve(gw, ot, *out, err, s)
        tot += out[3].sum(axis=0)
    gw.pool.close()
    return tot


UNION = {
    "hybrid_mtp": W.WORKLOADS["hybrid"].scaled(B=3, ctx=65536, resident_tail=8192, steps=5),
    "hybrid_ragged": W.WORKLOADS["hybrid"].scaled(B=2, ctx=32768, resident_tail=4096, K=1000,
                                                   hot_rows=2048, tail=100, T=3, steps=4),
    "noresident_mtp": W.WORKLOADS["noresident"].scaled(B=3, ctx=65536, T=4, steps=4),
    "resident_mtp": W.WORKLOADS["resident"].scaled(B=2, ctx=16384, T=2, steps=3),
}


@pytest.mark.parametrize("name", list(UNION))
@pytest.mark.parametrize("in_place", [False, True])
def test_resolve_union_parity(name, in_place):
    """Per-token lists: every occurrence of a repeated position resolves to the
    same row, only the first takes an LRU slot; ids, counts, bytes and state
    bit-exact."""
    w = UNION[name]
    tot = _run_union(w, w.steps, in_place=in_place)
    assert tot.sum() > 0


def test_resolve_union_capacity_and_repeats():
    """A union whose distinct misses exceed the free slots: the same rejected
    entries (all occurrences of a rejected position) and error bits as the
    oracle; positions repeated inside one token's list are served once too."""
    w = W.WORKLOADS["noresident"].scaled(B=2, ctx=16384, K=200, hot_rows=256, T=3, steps=2)
    base = list(W.topk_lists(w))
    lists = np.stack([W.token_lists(w, b, s, fresh=0.5) for s, b in enumerate(base)])
    lists[0, 1, 2, :4] = [11, 11, 11, -1]   # repeats within one token's list, padding
    tot = _run_union(w, 2, lists=lists)
    assert tot.sum() > 0


@pytest.mark.parametrize("in_place", [False, True])
def test_resolve_union_full_size(in_place):
    """The MTP workload (16 requests x 1M context, 4 tokens x top-2048 lists,
    4096-row hot buffers), first steps, every request compared."""
    w = W.WORKLOADS["hybrid"]
    tot = _run_union(w, 2, in_place=in_place, nthreads=16)
    assert tot.sum() == w.B * w.T * w.K * 2


def test_resolve_error_paths():
    """Out-of-range, repeated and host-less positions, padding and a bad request id:
    the same -1 entries, counts and error bits as the oracle."""
    w = W.WORKLOADS["tiny"].scaled(B=3, steps=2)
    lay = W.layout(w)
    rng = np.random.default_rng(3)
    lists = np.stack(list(W.topk_lists(w)))
    bad = lists.copy()
    bad[0, 0, :5] = [-1, -7, w.ctx, w.ctx + 100, -1]
    bad[0, 1, 10:14] = [3, 3, 3, 5]            # position 3 misses three times
    bad[1, 2, 20:22] = [9, 9]
    from harness import GpuWorkload
    from _mirror import compare_resolve, oracle_mirror
    gw = GpuWorkload(w)
    # request 2, page 1: neither resident nor copied to host
    gw.pool.page_map(2, 1, -1, -1)
    ot = oracle_mirror(gw)
    ot.page_host[2, 1] = -1
    bad[0, 2, 30:33] = [64, 65, 127]
    for s in range(2):
        t = torch.from_numpy(bad[s]).cuda()
        gw.resolve(s, topk=t)
        err = gw.pool.get_error()
        out = ot.resolve(np.arange(w.B), bad[s])
        assert out[4] != 0
        compare_resolve(gw, ot, *out, err, s)
    # a request id outside the pool
    rid = torch.tensor([0, 7, 2], dtype=torch.int32, device="cuda")
    gw.pool.resolve_topk(rid, torch.from_numpy(lists[1]).cuda(), gw.resolved, gw.gathered,
                         gw.gscale, gw.counts)
    err = gw.pool.get_error()
    assert err & 8
    assert (gw.resolved[1] == -1).all() and (gw.counts[1] == 0).all()
    assert not gw.gathered[1].any()
    gw.pool.close()


def test_host_side_argument_errors():
    import tiered_sparse_mla_gb300 as hs
    w = W.WORKLOADS["tiny"]
    from harness import GpuWorkload
    gw = GpuWorkload(w, build_topk=False)
    big = torch.zeros((1, w.hot_rows + 64), dtype=torch.int32, device="cuda")
    res = torch.empty_like(big)
    gat = torch.empty((1, big.shape[1], w.row_bytes), dtype=torch.uint8, device="cuda")
    cnt = torch.empty((1, 3), dtype=torch.int32, device="cuda")
    with pytest.raises(hs.HsError) as e:
        gw.pool.resolve_topk(gw.req_ids, big, res, gat, None, cnt)
    assert e.value.status == hs.HS_ERR_CAPACITY
    lib = hs.load()
    t = torch.zeros((1, 8), dtype=torch.int32, device="cuda")
    st = lib.hs_resolve_topk(gw.pool.handle, 1, None, t.data_ptr(), 8, t.data_ptr(),
                             gat.data_ptr(), None, cnt.data_ptr(), None)
    assert st == hs.HS_ERR_INVALID_ARG
    st = lib.hs_resolve_topk(gw.pool.handle, 1, gw.req_ids.data_ptr(), t.data_ptr(), 8,
                             t.data_ptr(), gat.data_ptr() + 4, None, cnt.data_ptr(), None)
    assert st == hs.HS_ERR_INVALID_ARG
    # FP8 scale pointer given to a BF16 pool
    st = lib.hs_resolve_topk(gw.pool.handle, 1, gw.req_ids.data_ptr(), t.data_ptr(), 8,
                             t.data_ptr(), gat.data_ptr(), t.data_ptr(), cnt.data_ptr(), None)
    assert st == hs.HS_ERR_INVALID_ARG
    with pytest.raises(hs.HsError):
        gw.pool.page_map(0, 0, gw.pool.cfg.n_gpu_blocks, -1)
    with pytest.raises(hs.HsError):
        gw.pool.hot_lease(0, [0] * 3)
    assert gw.pool.get_error() == 0
    gw.pool.close()


def test_snapshot_restore_replays_identically():
    w = SMALL["hybrid"]
    from harness import GpuWorkload
    from _mirror import gpu_state
    gw = GpuWorkload(w)
    gw.resolve(0)
    snap = gw.pool.snapshot()
    outs = []
    for rep in range(2):
        if rep:
            gw.pool.restore(snap)
        for s in (1, 2, 3):
            gw.resolve(s)
        torch.cuda.synchronize()
        outs.append((gw.resolved.cpu().clone(), gw.gathered.cpu().clone(), gpu_state(gw)))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    for k in outs[0][2]:
        assert np.array_equal(outs[0][2][k], outs[1][2][k])
    gw.pool.close()


# ---------------------------------------------------------------- several layers, one launch
def _run_layers(w, L, steps, in_place=False, nthreads=8):
    """L layers (pools of the same shape, own seeds) resolved by one
    hs_resolve_topk_layers launch per step; every layer is compared with its
    own oracle exactly as a single-layer resolve is."""
    import tiered_sparse_mla_gb300 as hs
    from harness import GpuWorkload
    from _mirror import compare_resolve, oracle_mirror
    gws = [GpuWorkload(w.scaled(index=w.index + 100 * l), in_place=in_place) for l in range(L)]
    ots = [oracle_mirror(gw) for gw in gws]
    B, K, rb = w.B, w.K, w.row_bytes
    res = torch.empty((L, B, K), dtype=torch.int32, device="cuda")
    gat = None if in_place else torch.empty((L, B, K, rb), dtype=torch.uint8, device="cuda")
    gsc = (torch.empty((L, B, K), dtype=torch.float32, device="cuda")
           if (w.dtype == "fp8" and not in_place) else None)
    cnt = torch.empty((L, B, 3), dtype=torch.int32, device="cuda")
    for l, gw in enumerate(gws):  # per-layer views, read by compare_resolve
        gw.resolved, gw.counts = res[l], cnt[l]
        gw.gathered = None if gat is None else gat[l]
        gw.gscale = None if gsc is None else gsc[l]
    group = hs.hs_layer_group_create([gw.pool for gw in gws])
    tot = np.zeros(3, np.int64)
    try:
        for s in range(steps):
            topk = torch.stack([gw.topk[s] for gw in gws]).contiguous()
            hs.hs_resolve_topk_layers(group, gws[0].req_ids, topk, res, gat, gsc, cnt)
            for l, gw in enumerate(gws):
                err = gw.pool.get_error()
                out = ots[l].resolve(np.arange(B), gw.topk_host[s], nthreads=nthreads)
                compare_resolve(gw, ots[l], *out, err, s)
                tot += out[3].sum(axis=0)
    finally:
        hs.hs_layer_group_destroy(group)
        for gw in gws:
            gw.pool.close()
    return tot


@pytest.mark.parametrize("name", ["hybrid", "resident", "noresident_small_k"])
@pytest.mark.parametrize("in_place", [False, True])
def test_resolve_layers_parity(name, in_place):
    w = SMALL[name]
    tot = _run_layers(w, 3, min(w.steps, 4), in_place=in_place)
    assert tot.sum() > 0


def test_layer_group_argument_errors():
    import tiered_sparse_mla_gb300 as hs
    from harness import GpuWorkload
    a = GpuWorkload(W.WORKLOADS["tiny"], build_topk=False)
    b = GpuWorkload(W.WORKLOADS["tiny"].scaled(hot_rows=1024), build_topk=False)
    with pytest.raises(hs.HsError) as e:  # pools of different hot-buffer sizes
        hs.hs_layer_group_create([a.pool, b.pool])
    assert e.value.status == hs.HS_ERR_INVALID_ARG
    with pytest.raises(hs.HsError):
        hs.hs_layer_group_create([])
    a.pool.close()
    b.pool.close()


def test_host_arena_device_views_read_the_host_bytes():
    """hs_host_rows_device / hs_host_scales_device: the GPU's view of the pinned
    host arena (the addresses the resolve reads misses through) holds the same
    bytes as the CPU's view, read by a GPU kernel."""
    from harness import GpuWorkload
    w = W.WORKLOADS["hybrid"].scaled(B=2, ctx=32768, resident_tail=4096, H=16, steps=1)
    gw = GpuWorkload(w)
    host = gw.pool.host_rows()
    dev = gw.pool.host_rows_device()
    assert host is not None and dev is not None and dev.is_cuda
    assert tuple(dev.shape) == host.shape
    rng = np.random.default_rng(5)
    rows = np.sort(rng.choice(host.shape[0], size=256, replace=False))
    idx = torch.from_numpy(rows).cuda()
    got = dev.index_select(0, idx).cpu().numpy()  # a GPU gather over the mapping
    assert np.array_equal(got, host[rows])
    hs_, ds_ = gw.pool.host_scales(), gw.pool.host_scales_device()
    assert np.array_equal(ds_.index_select(0, idx).cpu().numpy(), hs_[rows])
    gw.pool.close()
