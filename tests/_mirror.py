"""Test helpers: the oracle's own copy of a GPU workload, and comparisons."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as W

PAGE = 64


def oracle_mirror(gw) -> oracle.OracleTiers:
    """Oracle tiers built from the same seeded inputs as a GpuWorkload: the pool
    rows are copied once at setup (before any step); the host arena is the same
    read-only pinned memory. From then on the oracle evolves on its own."""
    w, lay = gw.w, gw.lay
    pool_rows = gw.pool.gpu_rows().cpu().numpy().copy()
    ps = gw.pool.gpu_scales()
    host = gw.pool.host_rows()
    hs_ = gw.pool.host_scales()
    if host is None:
        host = np.zeros((PAGE, w.row_bytes), np.uint8)
        hs_ = np.zeros(PAGE, np.float32) if w.dtype == "fp8" else None
    return oracle.OracleTiers(
        page_gpu=lay.page_gpu, page_host=lay.page_host, hot_blocks=lay.hot_blocks,
        ctx_len=np.full(w.B, w.ctx, np.int32), pool_rows=pool_rows,
        pool_scales=None if ps is None else ps.cpu().numpy().copy(), host_rows=host,
        host_scales=hs_, hot_rows=w.hot_rows, max_ctx=w.ctx)


def gpu_state(gw) -> dict:
    t = gw.pool.tables()
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in t.items()
            if k in ("slot_tag", "slot_stamp", "lru_order", "pos_to_slot", "clock")}


def check_lru_order(state):
    """The GPU keeps lru_order = slots sorted by (stamp, slot)."""
    for r in range(state["slot_stamp"].shape[0]):
        st = state["slot_stamp"][r]
        want = np.lexsort((np.arange(len(st)), st))
        assert np.array_equal(state["lru_order"][r], want), f"lru_order of request {r}"


def compare_resolve(gw, ot, res_o, gat_o, gsc_o, cnt_o, err_o, err_gpu, step, rows=None):
    """Bit-exact comparison of one step (all requests, or `rows` request indices)."""
    res = gw.resolved.cpu().numpy()
    cnt = gw.counts.cpu().numpy()
    sel = slice(None) if rows is None else rows
    assert np.array_equal(res[sel], res_o[sel]), f"resolved differs at step {step}"
    assert np.array_equal(cnt[sel], cnt_o[sel]), f"counts differ at step {step}"
    if gw.gathered is not None:
        gat = gw.gathered.cpu().numpy()
        assert np.array_equal(gat[sel], gat_o[sel]), f"gathered rows differ at step {step}"
        if gsc_o is not None:
            gsc = gw.gscale.cpu().numpy()
            assert np.array_equal(gsc[sel].view(np.uint32), gsc_o[sel].view(np.uint32))
    else:
        # rows stay in the pool: every resolved row id must hold the bytes (and
        # scale) the oracle gathered for that entry
        rows = gw.pool.gpu_rows().cpu().numpy()
        r = res[sel]
        ok = r >= 0
        assert np.array_equal(rows[r[ok]], gat_o[sel][ok]), f"pool rows differ at step {step}"
        assert not gat_o[sel][~ok].any(), "absent entries gather zeros"
        if gsc_o is not None:
            sc = gw.pool.gpu_scales().cpu().numpy()
            assert np.array_equal(sc[r[ok]].view(np.uint32), gsc_o[sel][ok].view(np.uint32))
    assert err_gpu == err_o, f"error bits {err_gpu} vs oracle {err_o} at step {step}"
    st = gpu_state(gw)
    assert np.array_equal(st["clock"], ot.clock)
    assert np.array_equal(st["slot_tag"], ot.tag), f"slot_tag differs at step {step}"
    assert np.array_equal(st["slot_stamp"], ot.stamp), f"slot_stamp differs at step {step}"
    assert np.array_equal(st["pos_to_slot"], ot.pos_to_slot), f"pos_to_slot differs at step {step}"
    check_lru_order(st)


def attention_errors(out_gpu, lse_gpu, out_ref, lse_ref):
    """Per query row: relative L2 error of out, absolute error of lse."""
    o = out_gpu.float().cpu().numpy().reshape(-1, 512).astype(np.float64)
    lg = lse_gpu.float().cpu().numpy().reshape(-1).astype(np.float64)
    den = np.maximum(np.linalg.norm(out_ref, axis=1), 1e-6)
    rel = np.linalg.norm(o - out_ref, axis=1) / den
    fin = np.isfinite(lse_ref)
    assert np.array_equal(fin, np.isfinite(lg)), "empty rows must give lse = -inf"
    dl = np.abs(lg[fin] - lse_ref[fin])
    return rel, dl
