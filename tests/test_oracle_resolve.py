"""Pins for the oracle's resolve (CPU only).

The pages print no worked example, so the resolve oracle is pinned by:
hand-computed LRU scenarios (tests/golden/lru_cases.json), a third
formulation of the LRU rule written here in plain Python, agreement between the
oracle's two C formulations on random inputs, and the state invariants
(occupancy <= capacity; every selected row GPU-addressable after its step;
gathered rows byte-identical to their originals; pos_to_slot and tag mutual
inverses; no row used in a step evicted in that step).
"""
import json
import os

import numpy as np
import pytest

import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))
PAGE = 64


def _tiers(oracle, page_gpu, page_host, hot_blocks, ctx_len, hot_rows, rb, n_gpu_rows,
           n_host_rows, rng, fp8=False, max_ctx=None):
    host_rows = rng.integers(0, 256, size=(n_host_rows, rb), dtype=np.uint8)
    pool_rows = rng.integers(0, 256, size=(n_gpu_rows, rb), dtype=np.uint8)
    host_scales = rng.random(n_host_rows, dtype=np.float32) if fp8 else None
    pool_scales = rng.random(n_gpu_rows, dtype=np.float32) if fp8 else None
    return oracle.OracleTiers(
        page_gpu=np.atleast_2d(page_gpu), page_host=np.atleast_2d(page_host),
        hot_blocks=np.atleast_2d(hot_blocks), ctx_len=np.atleast_1d(ctx_len),
        pool_rows=pool_rows, pool_scales=pool_scales, host_rows=host_rows,
        host_scales=host_scales, hot_rows=hot_rows,
        max_ctx=max_ctx or int(np.max(ctx_len)))


def _golden():
    with open(os.path.join(HERE, "golden", "lru_cases.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("formulation", [0, 1])
@pytest.mark.parametrize("case", _golden(), ids=lambda c: c["name"])
def test_golden_lru(oracle_lib, case, formulation):
    rng = np.random.default_rng(5)
    n_pages = len(case["page_gpu"])
    remaps = [st["set_page_gpu"] for st in case["steps"] if "set_page_gpu" in st]
    n_gpu_rows = 64 * (1 + max(max(case["page_gpu"]), max(case["hot_blocks"]),
                               max([max(m) for m in remaps], default=-1)))
    ot = _tiers(oracle_lib, np.array([case["page_gpu"]]), np.array([case["page_host"]]),
                np.array([case["hot_blocks"]]), case["ctx_len"], case["hot_rows"], 32,
                n_gpu_rows, 64 * n_pages, rng, max_ctx=64 * n_pages)
    host0 = ot.host_rows.copy()
    page_gpu = list(case["page_gpu"])
    for st in case["steps"]:
        if "set_page_gpu" in st:
            page_gpu = st["set_page_gpu"]
            ot.page_gpu[0, :] = page_gpu
        topk = np.array([st["topk"]], np.int32)
        res, gat, _, cnt, err = ot.resolve([0], topk, formulation=formulation)
        assert res[0].tolist() == st["resolved"], st["note"]
        assert cnt[0].tolist() == st["counts"], st["note"]
        assert err == st["err"], st["note"]
        assert ot.tag[0].tolist() == st["tag"], st["note"]
        assert ot.stamp[0].tolist() == st["stamp"], st["note"]
        # pos_to_slot is the inverse of tag
        p2s = ot.pos_to_slot[0]
        for s_, t in enumerate(st["tag"]):
            if t >= 0:
                assert p2s[t] == s_
        assert int((p2s >= 0).sum()) == sum(t >= 0 for t in st["tag"])
        # gathered rows: the host original of every hot/miss row, the pool row of a resident one
        for j, p in enumerate(st["topk"]):
            r = st["resolved"][j]
            if r < 0:
                assert not gat[0, j].any()
                continue
            pg = p // PAGE
            if page_gpu[pg] >= 0:
                assert np.array_equal(gat[0, j], ot.pool_rows[r])
            else:
                hrow = case["page_host"][pg] * PAGE + p % PAGE
                assert np.array_equal(gat[0, j], host0[hrow])


def test_bad_request_id(oracle_lib):
    rng = np.random.default_rng(1)
    ot = _tiers(oracle_lib, np.array([[-1]]), np.array([[0]]), np.array([[0]]), 64, 4, 16,
                64, 64, rng)
    res, gat, _, cnt, err = ot.resolve([3], np.array([[1, 2]], np.int32))
    assert err == oracle_lib.ERR_BAD_REQUEST
    assert res.tolist() == [[-1, -1]] and cnt.tolist() == [[0, 0, 0]]
    assert not gat.any() and ot.clock[0] == 0


def _python_lru_step(state, topk, ctx_len, page_gpu, page_host, C):
    """Third formulation, written independently in plain Python: keep the hot
    buffer as a dict slot -> (stamp, tag); after hits are stamped, repeatedly
    pick min((stamp, slot)) among slots not used this step for the next miss."""
    tag, stamp = state["tag"], state["stamp"]
    state["clock"] += 1
    c = state["clock"]
    where = {t: s for s, t in enumerate(tag) if t >= 0}
    resolved = [None] * len(topk)
    misses = []
    for j, p in enumerate(topk):
        if p == -1 or p < 0 or p >= ctx_len:
            resolved[j] = ("none",)
        elif page_gpu[p // PAGE] >= 0:
            resolved[j] = ("res", p)
        elif p in where:
            stamp[where[p]] = c
            resolved[j] = ("hot", where[p])
        elif page_host[p // PAGE] < 0:
            resolved[j] = ("none",)
        else:
            misses.append((p, j))
    seen = set()
    for p, j in sorted(misses):
        if p in seen:
            resolved[j] = ("none",)
            continue
        seen.add(p)
        cands = [(stamp[s], s) for s in range(C) if stamp[s] < c]
        if not cands:
            resolved[j] = ("none",)
            continue
        _, v = min(cands)
        if tag[v] >= 0:
            del where[tag[v]]
        tag[v], stamp[v] = p, c
        where[p] = v
        resolved[j] = ("hot", v)
    return resolved


def _random_case(rng):
    n_pages = int(rng.integers(1, 5))
    ctx = n_pages * PAGE - int(rng.integers(0, 40))
    C = int(rng.integers(2, 12))
    K = int(rng.integers(1, C + 1))
    kinds = rng.integers(0, 3, size=n_pages)  # 0 resident, 1 host, 2 neither
    page_gpu = np.where(kinds == 0, np.arange(n_pages), -1).astype(np.int32)
    page_host = np.where(kinds == 1, np.arange(n_pages), -1).astype(np.int32)
    return n_pages, ctx, C, K, page_gpu, page_host


@pytest.mark.parametrize("seed", range(40))
def test_three_formulations_agree(oracle_lib, seed):
    rng = np.random.default_rng(1000 + seed)
    n_pages, ctx, C, K, page_gpu, page_host = _random_case(rng)
    hot_block = n_pages  # leased after the page blocks
    mk = lambda: _tiers(oracle_lib, page_gpu[None], page_host[None], np.array([[hot_block]]),
                        ctx, C, 16, 64 * (n_pages + 1), 64 * n_pages,
                        np.random.default_rng(seed), max_ctx=64 * n_pages)
    a, b = mk(), mk()
    py = {"tag": [-1] * C, "stamp": [-1] * C, "clock": 0}
    # a small working set so that hits, misses, evictions and repeats all occur
    universe = rng.choice(64 * n_pages + 8, size=min(64 * n_pages, 3 * C), replace=False) - 4
    for step in range(12):
        topk = rng.choice(universe, size=K, replace=True).astype(np.int32)
        topk[rng.random(K) < 0.1] = -1
        ra = a.resolve([0], topk[None], formulation=0)
        rb = b.resolve([0], topk[None], formulation=1)
        for x, y in zip(ra, rb):
            if isinstance(x, np.ndarray):
                assert np.array_equal(x, y)
            else:
                assert x == y
        assert np.array_equal(a.tag, b.tag) and np.array_equal(a.stamp, b.stamp)
        assert np.array_equal(a.pos_to_slot, b.pos_to_slot)
        assert np.array_equal(a.pool_rows, b.pool_rows)
        pres = _python_lru_step(py, topk.tolist(), ctx, page_gpu, page_host, C)
        assert a.tag[0].tolist() == py["tag"] and a.stamp[0].tolist() == py["stamp"]
        for j, pr in enumerate(pres):
            got = int(ra[0][0, j])
            if pr[0] == "none":
                assert got == -1
            elif pr[0] == "res":
                p = pr[1]
                assert got == page_gpu[p // PAGE] * PAGE + p % PAGE
            else:
                assert got == hot_block * PAGE + pr[1]


def _check_invariants(ot, w, lay, topk, res, gat, gsc, before):
    """The state invariants after one resolve step of request batch 0..B-1."""
    B, K = topk.shape
    for b in range(B):
        tag, stamp, p2s = ot.tag[b], ot.stamp[b], ot.pos_to_slot[b]
        c = ot.clock[b]
        occupied = tag >= 0
        assert occupied.sum() <= w.hot_rows
        # pos_to_slot and tag are mutual inverses
        assert np.array_equal(np.sort(np.nonzero(p2s >= 0)[0]), np.sort(tag[occupied]))
        assert np.array_equal(p2s[tag[occupied]], np.nonzero(occupied)[0])
        # rows hot before this step and selected in it are still in the same slot
        btag = before["tag"][b]
        sel = set(topk[b][topk[b] >= 0].tolist())
        for s in np.nonzero(btag >= 0)[0]:
            if int(btag[s]) in sel and lay.page_gpu[b, btag[s] // PAGE] < 0:
                assert tag[s] == btag[s] and stamp[s] == c
        for j in range(K):
            p = int(topk[b, j])
            if p < 0:
                continue
            r = int(res[b, j])
            assert r >= 0  # every selected row is GPU-addressable after the step
            g = lay.page_gpu[b, p // PAGE]
            if g >= 0:
                assert r == g * PAGE + p % PAGE
                orig = before["pool"][r]
                orig_s = before["pool_s"][r] if gsc is not None else None
            else:
                s = p2s[p]
                assert s >= 0 and stamp[s] == c
                hrow = lay.page_host[b, p // PAGE] * PAGE + p % PAGE
                orig = ot.host_rows[hrow]
                orig_s = ot.host_scales[hrow] if gsc is not None else None
            assert np.array_equal(gat[b, j], orig)
            assert np.array_equal(ot.pool_rows[r], orig)
            if gsc is not None:
                assert gsc[b, j] == orig_s


@pytest.mark.parametrize("name,kw", [
    ("tiny", {}),
    ("hybrid", dict(B=2, ctx=16384, resident_tail=4096, hot_rows=512, K=256, steps=6, tail=32)),
    ("noresident", dict(B=3, ctx=8192, hot_rows=512, K=256, steps=5)),
])
def test_invariants_on_workloads(oracle_lib, name, kw):
    import torch
    w = W.WORKLOADS[name].scaled(**kw)
    lay = W.layout(w)
    fp8 = w.dtype == "fp8"
    pool = torch.zeros((lay.n_gpu_blocks * PAGE, w.row_bytes), dtype=torch.uint8)
    host = torch.zeros((lay.n_host_blocks * PAGE, w.row_bytes), dtype=torch.uint8)
    ps = torch.zeros(pool.shape[0]) if fp8 else None
    hs = torch.zeros(host.shape[0]) if fp8 else None
    W.fill_rows(w.dtype, pool, ps, W.row_seed(w, "gpu"))
    W.fill_rows(w.dtype, host, hs, W.row_seed(w, "host"))
    ot = oracle_lib.OracleTiers(
        page_gpu=lay.page_gpu, page_host=lay.page_host, hot_blocks=lay.hot_blocks,
        ctx_len=np.full(w.B, w.ctx, np.int32), pool_rows=pool.numpy().copy(),
        pool_scales=None if ps is None else ps.numpy().copy(), host_rows=host.numpy(),
        host_scales=None if hs is None else hs.numpy(), hot_rows=w.hot_rows, max_ctx=w.ctx)
    total = np.zeros(3, np.int64)
    for topk in W.topk_lists(w):
        before = {"tag": ot.tag.copy(), "pool": ot.pool_rows.copy(),
                  "pool_s": None if ps is None else ot.pool_scales.copy()}
        res, gat, gsc, cnt, err = ot.resolve(np.arange(w.B), topk, nthreads=2)
        assert err == 0
        assert (cnt.sum(axis=1) == w.K).all()
        total += cnt.sum(axis=0)
        _check_invariants(ot, w, lay, topk, res, gat, gsc, before)
    if name == "tiny":
        assert total[0] > 0 and total[1] > 0 and total[2] > 0
    else:
        assert total[1] > 0 and total[2] > 0


# ---------------------------------------------------------------- union of lists
@pytest.mark.parametrize("seed", range(30))
def test_union_reduces_to_deduplicated_resolve(oracle_lib, seed):
    """Union mode (per-token MTP lists sharing one hot state): resolving a list
    with repeated positions equals resolving it with every repeat blanked (the
    pinned single-list rule), then giving each repeat its first occurrence's
    row. The hot state ends identical, and no repeat error is raised."""
    rng = np.random.default_rng(2000 + seed)
    n_pages, ctx, C, K, page_gpu, page_host = _random_case(rng)
    hot_block = n_pages
    mk = lambda: _tiers(oracle_lib, page_gpu[None], page_host[None], np.array([[hot_block]]),
                        ctx, C, 16, 64 * (n_pages + 1), 64 * n_pages,
                        np.random.default_rng(seed), max_ctx=64 * n_pages)
    u, d = mk(), mk()
    universe = rng.choice(64 * n_pages + 8, size=min(64 * n_pages, 3 * C), replace=False) - 4
    for step in range(12):
        # a few lists over a small working set, concatenated: repeats are common
        topk = rng.choice(universe, size=K, replace=True).astype(np.int32)
        topk[rng.random(K) < 0.1] = -1
        first = {}
        rep = np.zeros(K, bool)
        for j, p in enumerate(topk.tolist()):
            if p == -1:
                continue
            if p in first:
                rep[j] = True
            else:
                first[p] = j
        blank = topk.copy()
        blank[rep] = -1
        ru, gu, _, cu, eu = u.resolve([0], topk[None], union=True)
        rd, gd, _, cd, ed = d.resolve([0], blank[None])
        want = rd[0].copy()
        for j in np.nonzero(rep)[0]:
            want[j] = rd[0][first[int(topk[j])]]
        assert np.array_equal(ru[0], want)
        assert eu == ed and not (eu & 2)
        assert cu.sum() == cd.sum() + int((want[rep] >= 0).sum())
        for a, b in ((u.tag, d.tag), (u.stamp, d.stamp), (u.pos_to_slot, d.pos_to_slot),
                     (u.clock, d.clock), (u.pool_rows, d.pool_rows)):
            assert np.array_equal(a, b)
        # every occurrence of a position names one row, and its bytes are gathered
        for j in range(K):
            if ru[0, j] >= 0:
                assert ru[0, j] == ru[0, first[int(topk[j])]]
                assert np.array_equal(gu[0, j], u.pool_rows[ru[0, j]])


def test_token_lists_properties():
    """Per-token lists: token 0 keeps the step's list, later tokens replace
    about 10% of it, every list holds distinct positions up to its token's own."""
    w = W.WORKLOADS["hybrid"].scaled(B=3, ctx=32768, resident_tail=4096, steps=2)
    for s, base in enumerate(W.topk_lists(w)):
        tl = W.token_lists(w, base, s)
        assert tl.shape == (w.B, w.T, w.K) and tl.dtype == np.int32
        assert np.array_equal(tl[:, 0], base)
        for b in range(w.B):
            for t in range(w.T):
                assert len(np.unique(tl[b, t])) == w.K
                assert tl[b, t].min() >= 0 and tl[b, t].max() < w.ctx
                if t:
                    assert (tl[b, t] != base[b]).sum() == round(0.1 * w.K)
        assert np.array_equal(tl, W.token_lists(w, base, s))  # seeded


def test_union_of_token_lists_on_workload(oracle_lib):
    """The union resolve of an MTP step's per-token lists: every entry resolves
    (the distinct positions fit the hot buffer), every occurrence of a position
    names one row, and the hot buffer holds each distinct missing position once."""
    import torch
    w = W.WORKLOADS["hybrid"].scaled(B=2, ctx=16384, resident_tail=2048, hot_rows=512, K=128,
                                     steps=4, tail=16)
    lay = W.layout(w)
    pool = torch.zeros((lay.n_gpu_blocks * PAGE, w.row_bytes), dtype=torch.uint8)
    host = torch.zeros((lay.n_host_blocks * PAGE, w.row_bytes), dtype=torch.uint8)
    ps, hs = torch.zeros(pool.shape[0]), torch.zeros(host.shape[0])
    W.fill_rows(w.dtype, pool, ps, W.row_seed(w, "gpu"))
    W.fill_rows(w.dtype, host, hs, W.row_seed(w, "host"))
    ot = oracle_lib.OracleTiers(
        page_gpu=lay.page_gpu, page_host=lay.page_host, hot_blocks=lay.hot_blocks,
        ctx_len=np.full(w.B, w.ctx, np.int32), pool_rows=pool.numpy().copy(),
        pool_scales=ps.numpy().copy(), host_rows=host.numpy(), host_scales=hs.numpy(),
        hot_rows=w.hot_rows, max_ctx=w.ctx)
    for s, base in enumerate(W.topk_lists(w)):
        flat = W.token_lists(w, base, s).reshape(w.B, -1)
        res, gat, gsc, cnt, err = ot.resolve(np.arange(w.B), flat, union=True)
        assert err == 0 and (cnt.sum(axis=1) == w.T * w.K).all()
        for b in range(w.B):
            row_of = {}
            for p, r in zip(flat[b].tolist(), res[b].tolist()):
                assert r >= 0 and row_of.setdefault(p, r) == r
            tags = ot.tag[b][ot.tag[b] >= 0]
            assert len(np.unique(tags)) == len(tags)
            assert np.array_equal(gat[b], ot.pool_rows[res[b]])
            assert np.array_equal(gsc[b].view(np.uint32), ot.pool_scales[res[b]].view(np.uint32))


@pytest.mark.parametrize("seed", range(20))
def test_union_with_more_distinct_misses_than_slots(oracle_lib, seed):
    """A union longer than the hot buffer whose distinct missing positions
    outnumber the free slots: the positions beyond the capacity are rejected
    with every one of their occurrences (none takes another position's row),
    exactly as the single-list rule rejects them once repeats are blanked."""
    rng = np.random.default_rng(3000 + seed)
    n_pages = int(rng.integers(2, 5))
    ctx = n_pages * PAGE
    C = int(rng.integers(2, 10))
    K = int(rng.integers(C + 1, 3 * C + 1))
    page_gpu = np.full(n_pages, -1, np.int32)
    page_host = np.arange(n_pages, dtype=np.int32)   # every row misses unless hot
    hot_block = n_pages
    mk = lambda: _tiers(oracle_lib, page_gpu[None], page_host[None], np.array([[hot_block]]),
                        ctx, C, 16, 64 * (n_pages + 1), 64 * n_pages,
                        np.random.default_rng(seed), max_ctx=ctx)
    u, d = mk(), mk()
    universe = rng.choice(ctx, size=min(ctx, 2 * K), replace=False)
    rejected_seen = 0
    for step in range(8):
        topk = rng.choice(universe, size=K, replace=True).astype(np.int32)
        first, rep = {}, np.zeros(K, bool)
        for j, p in enumerate(topk.tolist()):
            if p in first:
                rep[j] = True
            else:
                first[p] = j
        blank = topk.copy()
        blank[rep] = -1
        ru, _, _, cu, eu = u.resolve([0], topk[None], union=True)
        rd, _, _, cd, ed = d.resolve([0], blank[None])
        want = rd[0].copy()
        for j in np.nonzero(rep)[0]:
            want[j] = rd[0][first[int(topk[j])]]
        assert np.array_equal(ru[0], want)
        assert eu == ed and not (eu & 2)
        assert cu.sum() == cd.sum() + int((want[rep] >= 0).sum())
        rejected_seen += int((want < 0).sum())
        for a, b in ((u.tag, d.tag), (u.stamp, d.stamp), (u.pos_to_slot, d.pos_to_slot)):
            assert np.array_equal(a, b)
    assert rejected_seen > 0  # the case does overflow


def _golden_union():
    with open(os.path.join(HERE, "golden", "union_cases.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("formulation", [0, 1])
@pytest.mark.parametrize("case", _golden_union(), ids=lambda c: c["name"])
def test_golden_union(oracle_lib, case, formulation):
    """Hand-computed unions of per-token lists (tests/golden/union_cases.json)."""
    rng = np.random.default_rng(6)
    n_pages = len(case["page_gpu"])
    n_gpu_rows = 64 * (1 + max(max(case["page_gpu"]), max(case["hot_blocks"])))
    ot = _tiers(oracle_lib, np.array([case["page_gpu"]]), np.array([case["page_host"]]),
                np.array([case["hot_blocks"]]), case["ctx_len"], case["hot_rows"], 32,
                n_gpu_rows, 64 * n_pages, rng, max_ctx=64 * n_pages)
    host0 = ot.host_rows.copy()
    for st in case["steps"]:
        topk = np.array([st["topk"]], np.int32)
        res, gat, _, cnt, err = ot.resolve([0], topk, formulation=formulation, union=True)
        assert res[0].tolist() == st["resolved"], st["note"]
        assert cnt[0].tolist() == st["counts"], st["note"]
        assert err == st["err"], st["note"]
        assert ot.tag[0].tolist() == st["tag"], st["note"]
        assert ot.stamp[0].tolist() == st["stamp"], st["note"]
        for j, p in enumerate(st["topk"]):
            r = st["resolved"][j]
            if r < 0:
                assert not gat[0, j].any()
            elif case["page_gpu"][p // PAGE] >= 0:
                assert np.array_equal(gat[0, j], ot.pool_rows[r])
            else:
                assert np.array_equal(gat[0, j], host0[case["page_host"][p // PAGE] * PAGE + p % PAGE])
