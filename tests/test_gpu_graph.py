"""CUDA-graph capture of the step (resolve + decode).

The pages require the fused resolve kernel to be capturable in a CUDA graph.
Captured steps replayed from a restored state must give the same outputs and
state as eager execution, and the device clock must advance per replay.
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


def test_graph_replay_matches_eager():
    from harness import GpuWorkload
    from _mirror import gpu_state
    w = W.WORKLOADS["hybrid"].scaled(B=3, ctx=32768, resident_tail=4096, H=32, steps=4)
    gw = GpuWorkload(w)
    qs = [W.make_q(w, s, device="cuda") for s in range(w.steps)]
    snap = gw.pool.snapshot()

    eager = []
    for s in range(w.steps):
        gw.resolve(s)
        gw.decode(s, qs[s])
        torch.cuda.synchronize()
        eager.append((gw.resolved.clone(), gw.gathered.clone(), gw.counts.clone(),
                      gw.out.clone(), gw.lse.clone()))
    state_eager = gpu_state(gw)

    gw.pool.restore(snap)
    # warm up on a side stream, as graph capture requires
    stream = torch.cuda.Stream()
    graphs = []
    for s in range(w.steps):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            gw.resolve(s, stream=torch.cuda.current_stream())
            gw.decode(s, qs[s], stream=torch.cuda.current_stream())
        graphs.append(g)
    torch.cuda.synchronize()
    # capture does not execute: state is still the snapshot's
    gw.pool.restore(snap)
    clock0 = gw.pool.tables()["clock"].clone()
    for s in range(w.steps):
        graphs[s].replay()
        torch.cuda.synchronize()
        e = eager[s]
        assert torch.equal(gw.resolved, e[0]) and torch.equal(gw.gathered, e[1])
        assert torch.equal(gw.counts, e[2])
        assert torch.equal(gw.out, e[3]) and torch.equal(gw.lse, e[4])
    state_graph = gpu_state(gw)
    for k in state_eager:
        assert np.array_equal(state_eager[k], state_graph[k])
    assert torch.equal(gw.pool.tables()["clock"], clock0 + w.steps)
    assert gw.pool.get_error() == 0
    gw.pool.close()


def test_bench_e2e_pipeline_results():
    """The bench's end-to-end loop (one graph launch per step: the step's calls,
    the next step's upload and the previous step's download as parallel
    branches) hands back, in pinned host memory, exactly what eager calls on
    the same inputs give."""
    import bench
    from harness import GpuWorkload
    w = W.WORKLOADS["resident"].scaled(B=4, ctx=16384, steps=6)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        gw = GpuWorkload(w, stream=stream, in_place=True)
        qs = [W.make_q(w, s, device="cuda") for s in range(4)]
    torch.cuda.synchronize()
    r = bench.run_e2e(None, gw, qs, stream, w, check=True)
    assert r["check"] == {"out_equal": True, "lse_equal": True}, r["check"]
    assert r["h2d_bytes_per_step"] == w.B * w.K * 4 + w.B * w.T * w.H * 576 * 2
    assert r["d2h_bytes_per_step"] == w.B * w.T * w.H * (512 * 2 + 4)
    gw.pool.close()
