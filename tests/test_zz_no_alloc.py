"""The allocation-free decode entry point (hs_sparse_mla_decode_static_ws).

For callers that cannot allocate device memory (an engine that has reserved
the device's memory for its own KV pool, a C plugin without an allocator), the
library offers decode with its split-KV scratch in a fixed array inside the
library. Called through the C ABI, twice in a row, it must give what the
allocating entry point gives. Both run the same kernels with the same split
of the keys on the same inputs, so the outputs must agree bit for bit (a
wrong offset into the fixed array would show up here).
This file sorts last so that a run stopping at the first failure has run every
other test first; it also passes when run alone.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["resident", "hybrid"])
def test_static_workspace_decode_matches_allocating_entry_point(name):
    import __graft_entry__ as g
    g.build()
    import tiered_sparse_mla_gb300 as hs
    from harness import GpuWorkload

    w = {"resident": W.WORKLOADS["resident"].scaled(B=2, ctx=16384, steps=1),
         "hybrid": W.WORKLOADS["hybrid"].scaled(B=2, ctx=32768, resident_tail=4096, H=32,
                                                steps=1)}[name]
    need = hs.hs_decode_workspace_bytes(w.B, w.T, w.H, w.K)
    assert 0 < need <= hs.HS_STATIC_DECODE_WS_BYTES  # the shape does use scratch memory
    gw = GpuWorkload(w)
    q = W.make_q(w, 0, device="cuda")
    gw.resolve(0)
    gw.decode(0, q)  # allocating entry point, caller-provided workspace
    torch.cuda.synchronize()
    ref_out, ref_lse = gw.out.clone(), gw.lse.clone()

    lib = hs.load()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        out = torch.full_like(gw.out, float("nan"))
        lse = torch.full_like(gw.lse, float("nan"))
        st = lib.hs_sparse_mla_decode_static_ws(
            gw.pool.handle, w.B, w.T, w.H, w.K, q.data_ptr(), gw.gathered.data_ptr(),
            None if gw.gscale is None else gw.gscale.data_ptr(), gw.resolved.data_ptr(),
            gw.topk[0].data_ptr(), gw.req_ids.data_ptr(), ctypes.c_float(w.sm_scale),
            out.data_ptr(), lse.data_ptr(), stream)
        assert st == hs.HS_OK, hs.status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), f"call {call}: out"
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32)), f"call {call}: lse"
    assert gw.pool.get_error() == 0
    gw.pool.close()
