"""The multi-turn agent mix (residency moving full -> hybrid -> none, context
growing every step, MTP3, FP8): GPU resolve bit-exact against the oracle on
every step, attention within tolerance on sampled steps."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__ as g
    g.build()
    assert torch.cuda.is_available()


def _bits(q):
    return q.cpu().view(torch.int16).numpy().view(np.uint16)


def _run(w, attn_every, attn_rows=None, state_every=1, gathered_every=1, nthreads=16):
    import oracle
    from harness import GpuAgent
    from _mirror import attention_errors, check_lru_order, gpu_state
    ga = GpuAgent(w)
    lay = ga.lay
    ot = oracle.OracleTiers(
        page_gpu=np.full((w.B, w.pages), -1, np.int32), page_host=lay.page_host,
        hot_blocks=lay.hot_blocks, ctx_len=np.full(w.B, w.first, np.int32),
        pool_rows=ga.pool.gpu_rows().cpu().numpy().copy(),
        pool_scales=ga.pool.gpu_scales().cpu().numpy().copy(), host_rows=ga.pool.host_rows(),
        host_scales=ga.pool.host_scales(), hot_rows=w.hot_rows, max_ctx=w.ctx)
    states_seen = set()
    tot = np.zeros(3, np.int64)
    worst = 0.0
    for n, st in enumerate(W.agent_steps(w)):
        ga.apply(st)
        ot.page_gpu[:] = st.page_gpu
        ot.ctx_len[:] = st.ctx
        states_seen |= set(st.state.tolist())
        topk = torch.from_numpy(st.topk).cuda()
        ga.resolve(topk)
        attn = n % attn_every == 0 or n == w.steps - 1
        if attn:
            q = W.make_q(w, n, device="cuda")
            ga.decode(q, topk)
        torch.cuda.synchronize()
        assert ga.pool.get_error() == 0
        res, gat, gsc, cnt, err = ot.resolve(np.arange(w.B), st.topk, nthreads=nthreads)
        assert err == 0
        assert np.array_equal(ga.resolved.cpu().numpy(), res), f"step {n}"
        assert np.array_equal(ga.counts.cpu().numpy(), cnt), f"step {n}"
        tot += cnt.sum(0)
        if n % gathered_every == 0:
            assert np.array_equal(ga.gathered.cpu().numpy(), gat), f"step {n}"
            assert np.array_equal(ga.gscale.cpu().numpy().view(np.uint32), gsc.view(np.uint32))
        if n % state_every == 0 or n == w.steps - 1:
            s = gpu_state(ga)
            assert np.array_equal(s["slot_tag"], ot.tag) and np.array_equal(s["slot_stamp"], ot.stamp)
            assert np.array_equal(s["pos_to_slot"], ot.pos_to_slot) and np.array_equal(s["clock"], ot.clock)
            check_lru_order(s)
        if attn:
            sel = None
            if attn_rows is not None:
                rng = np.random.default_rng(n)
                idx = np.sort(rng.choice(w.B * w.T * w.H, size=attn_rows, replace=False))
                sel = np.stack([idx // (w.T * w.H), (idx // w.H) % w.T, idx % w.H], 1).astype(np.int32)
            o_ref, l_ref = oracle.sparse_mla_decode(_bits(q), gat, gsc, res, st.topk, st.ctx,
                                                    w.sm_scale, sel=sel, nthreads=nthreads)
            out, lse = ga.out, ga.lse
            if sel is not None:
                out, lse = out[sel[:, 0], sel[:, 1], sel[:, 2]], lse[sel[:, 0], sel[:, 1], sel[:, 2]]
            rel, dl = attention_errors(out, lse, o_ref, l_ref)
            assert rel.max() <= 5e-2 and (dl.size == 0 or dl.max() <= 1e-2), f"step {n}"
            worst = max(worst, rel.max())
    ga.pool.close()
    return tot, states_seen, worst


def test_agent_mix_small_every_step():
    w = W.AgentMix().scaled(B=4, turns=4, first=9000, per_turn=300, out_tokens=24, K=512,
                            hot_rows=1024, resident_tail=4096, H=16, tail=64)
    tot, states, _ = _run(w, attn_every=5)
    assert states == {0, 1, 2}
    assert tot[0] > 0 and tot[1] > 0 and tot[2] > 0


def test_agent_mix_full_size():
    """All 13 turns x 55 steps of the full-size mix: resolve and counts every step,
    gathered bytes and LRU state every 20th step, sampled attention rows."""
    w = W.AgentMix()
    tot, states, _ = _run(w, attn_every=143, attn_rows=192, state_every=20, gathered_every=20)
    assert states == {0, 1, 2}
    assert tot[1] > 0 and tot[2] > 0
