"""GPU parity of sparse MLA decode against the float64 oracle.

Tolerance (per query row (request, token, head)):
  ||out - out_ref||_2 / max(||out_ref||_2, 1e-6) <= 2e-2 for BF16 rows, 5e-2 for FP8
  |lse - lse_ref| <= 1e-2
The oracle attends over its own resolve's gathered rows (the resolve is
bit-exact, so both sides see the same bytes, but no oracle input comes from
the GPU).
"""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "fp8": 5e-2}
LSE_TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()
    assert torch.cuda.is_available()


def _bits(q):
    return q.cpu().view(torch.int16).numpy().view(np.uint16)


def _decode_case(w, steps, sample_rows=None, nthreads=8, topk_override=None, in_place=False):
    import oracle
    from harness import GpuWorkload
    from _mirror import attention_errors, oracle_mirror
    gw = GpuWorkload(w, in_place=in_place)
    ot = oracle_mirror(gw)
    lists = gw.topk_host if topk_override is None else topk_override
    worst = (0.0, 0.0)
    for s in range(steps):
        t = torch.from_numpy(np.ascontiguousarray(lists[s])).cuda()
        q = W.make_q(w, s, device="cuda")
        gw.resolve(s, topk=t)
        gw.decode(s, q, topk=t)
        torch.cuda.synchronize()
        assert gw.pool.get_error() == 0
        res, gat, gsc, _, err = ot.resolve(np.arange(w.B), lists[s], nthreads=nthreads)
        assert err == 0
        sel = None
        if sample_rows is not None:
            rng = np.random.default_rng(100 + s)
            n = w.B * w.T * w.H
            idx = np.sort(rng.choice(n, size=min(sample_rows, n), replace=False))
            sel = np.stack([idx // (w.T * w.H), (idx // w.H) % w.T, idx % w.H], 1).astype(np.int32)
        o_ref, l_ref = oracle.sparse_mla_decode(_bits(q), gat, gsc, res, lists[s],
                                                np.full(w.B, w.ctx, np.int32), w.sm_scale,
                                                sel=sel, nthreads=nthreads)
        out, lse = gw.out, gw.lse
        if sel is not None:
            out = gw.out[sel[:, 0], sel[:, 1], sel[:, 2]]
            lse = gw.lse[sel[:, 0], sel[:, 1], sel[:, 2]]
        rel, dl = attention_errors(out, lse, o_ref, l_ref)
        assert rel.max() <= TOL[w.dtype], f"step {s}: max rel err {rel.max():.3e}"
        assert dl.size == 0 or dl.max() <= LSE_TOL, f"step {s}: max lse err {dl.max():.3e}"
        worst = (max(worst[0], rel.max()), max(worst[1], dl.max() if dl.size else 0.0))
    gw.pool.close()
    return worst


SMALL = {
    "tiny": (W.WORKLOADS["tiny"], 3),
    "resident": (W.WORKLOADS["resident"].scaled(B=2, ctx=16384, H=64, steps=2), 2),
    "hybrid_mtp": (W.WORKLOADS["hybrid"].scaled(B=2, ctx=32768, resident_tail=4096, H=32,
                                                 steps=3), 3),
    "hybrid_ragged": (W.WORKLOADS["hybrid"].scaled(B=2, ctx=16384, resident_tail=2048, K=1000,
                                                    hot_rows=2048, tail=100, H=24, T=3,
                                                    steps=2), 2),
    "noresident": (W.WORKLOADS["noresident"].scaled(B=3, ctx=32768, H=16, steps=2), 2),
    # BF16 rows, K = 1000: eight splits of 128 keys, the last one's second tile
    # holds 40 keys (keys 32-39 valid in the half the second copying warp takes)
    "resident_ragged": (W.WORKLOADS["resident"].scaled(B=2, ctx=16384, H=64, K=1000, tail=100,
                                                       steps=2), 2),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_decode_parity_small(name):
    w, steps = SMALL[name]
    _decode_case(w, steps)


@pytest.mark.parametrize("name,steps,rows", [("resident", 1, 256), ("hybrid", 1, 256),
                                             ("noresident", 1, 256)])
def test_decode_parity_full_size_sampled(name, steps, rows):
    """Full-size workloads: sampled query rows, computed one by one by the oracle."""
    _decode_case(W.WORKLOADS[name], steps, sample_rows=rows, nthreads=16)


def test_decode_edge_cases():
    """Empty lists (lse = -inf, out = 0), a single valid entry, and the MTP causal
    rule excluding every entry for the early draft tokens."""
    w = W.WORKLOADS["tiny"].scaled(B=3, T=4, H=8, steps=1)
    lists = np.stack(list(W.topk_lists(w)))
    lists[0, 0, :] = -1                            # request 0: nothing selected
    lists[0, 1, :] = -1
    lists[0, 1, 7] = 4000                          # request 1: one valid entry
    lists[0, 2, :] = -1                            # request 2: the last three positions only;
    lists[0, 2, :3] = [w.ctx - 1, w.ctx - 2, w.ctx - 3]  # token 0 (position L-4) sees none
    _decode_case(w, 1, topk_override=lists)


# ---------------------------------------------------------------- rows read in place
@pytest.mark.parametrize("name", list(SMALL))
def test_decode_in_place_parity_small(name):
    """No gathered buffer: attention gathers the rows from the pool by row id."""
    w, steps = SMALL[name]
    _decode_case(w, steps, in_place=True)


@pytest.mark.parametrize("name", ["resident", "hybrid"])
def test_decode_in_place_full_size_sampled(name):
    _decode_case(W.WORKLOADS[name], 1, sample_rows=256, nthreads=16, in_place=True)


def test_decode_in_place_edge_cases():
    w = W.WORKLOADS["tiny"].scaled(B=3, T=4, H=8, steps=1)
    lists = np.stack(list(W.topk_lists(w)))
    lists[0, 0, :] = -1
    lists[0, 1, :] = -1
    lists[0, 1, 7] = 4000
    lists[0, 2, :] = -1
    lists[0, 2, :3] = [w.ctx - 1, w.ctx - 2, w.ctx - 3]
    _decode_case(w, 1, topk_override=lists, in_place=True)


@pytest.mark.parametrize("name", ["resident", "resident_ragged", "hybrid_ragged", "noresident"])
def test_decode_in_place_matches_gathered_bitwise(name):
    """The same rows reach the same tiles either way, so the outputs are identical."""
    from harness import GpuWorkload
    w, _ = SMALL[name]
    ga, gb = GpuWorkload(w), GpuWorkload(w, in_place=True)
    for s in range(2):
        q = W.make_q(w, s, device="cuda")
        for gw in (ga, gb):
            gw.resolve(s)
            gw.decode(s, q)
        torch.cuda.synchronize()
        assert ga.pool.get_error() == 0 and gb.pool.get_error() == 0
        assert torch.equal(ga.resolved, gb.resolved)
        assert torch.equal(ga.out.view(torch.int16), gb.out.view(torch.int16)), f"out differs, step {s}"
        assert torch.equal(ga.lse.view(torch.int32), gb.lse.view(torch.int32)), f"lse differs, step {s}"
    ga.pool.close()
    gb.pool.close()


# ---------------------------------------------------------------- one list per query token
def _per_token_case(w, steps, sample_rows=None, nthreads=8, in_place=False, lists=None):
    """Union resolve + per-token decode on the GPU; on the oracle side the union
    resolve, then each (request, token) attends over its own list as a
    one-token batch entry whose context ends at its position L - T + t."""
    import oracle
    from harness import GpuWorkload
    from _mirror import attention_errors, oracle_mirror
    gw = GpuWorkload(w, in_place=in_place, per_token=True, build_topk=lists is None)
    ot = oracle_mirror(gw)
    lists = gw.topk_host if lists is None else lists
    B, T, H, K = w.B, w.T, w.H, w.K
    L1 = (w.ctx - T + 1 + np.tile(np.arange(T), B)).astype(np.int32)  # per list (b, t)
    for s in range(steps):
        t = torch.from_numpy(np.ascontiguousarray(lists[s])).cuda()
        q = W.make_q(w, s, device="cuda")
        gw.resolve(s, topk=t)
        gw.decode(s, q, topk=t)
        torch.cuda.synchronize()
        assert gw.pool.get_error() == 0
        flat = np.ascontiguousarray(lists[s].reshape(B, T * K))
        res, gat, gsc, _, err = ot.resolve(np.arange(B), flat, nthreads=nthreads, union=True)
        assert err == 0
        sel = None
        if sample_rows is not None:
            rng = np.random.default_rng(200 + s)
            n = B * T * H
            idx = np.sort(rng.choice(n, size=min(sample_rows, n), replace=False))
            sel = np.stack([idx // H, np.zeros_like(idx), idx % H], 1).astype(np.int32)
        o_ref, l_ref = oracle.sparse_mla_decode(
            _bits(q).reshape(B * T, 1, H, -1), gat.reshape(B * T, K, -1),
            None if gsc is None else gsc.reshape(B * T, K), res.reshape(B * T, K),
            lists[s].reshape(B * T, K), L1, w.sm_scale, sel=sel, nthreads=nthreads)
        out, lse = gw.out, gw.lse
        if sel is not None:
            bt = sel[:, 0]
            out = gw.out[bt // T, bt % T, sel[:, 2]]
            lse = gw.lse[bt // T, bt % T, sel[:, 2]]
        rel, dl = attention_errors(out, lse, o_ref, l_ref)
        assert rel.max() <= TOL[w.dtype], f"step {s}: max rel err {rel.max():.3e}"
        assert dl.size == 0 or dl.max() <= LSE_TOL, f"step {s}: max lse err {dl.max():.3e}"
    gw.pool.close()


PER_TOKEN = {
    "hybrid_mtp": (W.WORKLOADS["hybrid"].scaled(B=2, ctx=32768, resident_tail=4096, H=32,
                                                 steps=3), 3),
    "hybrid_ragged": (W.WORKLOADS["hybrid"].scaled(B=2, ctx=16384, resident_tail=2048, K=1000,
                                                    hot_rows=2048, tail=100, H=24, T=3,
                                                    steps=2), 2),
    "resident_bf16": (W.WORKLOADS["resident"].scaled(B=2, ctx=16384, H=64, T=2, steps=2), 2),
}


@pytest.mark.parametrize("name", list(PER_TOKEN))
@pytest.mark.parametrize("in_place", [False, True])
def test_decode_per_token_parity_small(name, in_place):
    w, steps = PER_TOKEN[name]
    _per_token_case(w, steps, in_place=in_place)


@pytest.mark.parametrize("in_place", [False, True])
def test_decode_per_token_full_size_sampled(in_place):
    """16 requests x 1M context, 4 tokens with their own top-2048 lists, 128 heads."""
    _per_token_case(W.WORKLOADS["hybrid"], 1, sample_rows=256, nthreads=16, in_place=in_place)


def test_decode_per_token_edge_cases():
    """A token whose own list is empty, one with a single entry, and lists
    holding positions after a token's own position (masked for it only)."""
    w = W.WORKLOADS["tiny"].scaled(B=2, T=4, H=8, steps=1)
    base = next(iter(W.topk_lists(w)))
    lists = W.token_lists(w, base, 0)[None].copy()
    lists[0, 0, 1, :] = -1                         # request 0, token 1: nothing
    lists[0, 0, 2, :] = -1
    lists[0, 0, 2, 5] = 1000                       # token 2: one entry
    lists[0, 1, 0, :3] = [w.ctx - 1, w.ctx - 2, w.ctx - 3]  # after token 0 (L - 4): masked
    _per_token_case(w, 1, lists=lists)
