"""Sets a synthetic workload up in a GPU pool (harness for tests and bench.py).

Plumbing only: page mapping, hot-buffer leases and row contents come from
``workloads``; every operation goes through the C ABI binding.
"""
from __future__ import annotations

import numpy as np
import torch

import tiered_sparse_mla_gb300 as hs
import workloads as W


class GpuWorkload:
    """A workload's pool, its request tables and the step buffers on cuda:0."""

    def __init__(self, w: W.Workload, stream=None, build_topk: bool = True,
                 in_place: bool = False, per_token: bool = False):
        """in_place: no gathered buffer; attention reads the rows from the pool.
        per_token: one top-K list per query token (topk [steps][B][T][K]); the
        resolve takes each request's T lists as one union, the decode gives
        each token its own list."""
        self.w = w
        self.in_place = in_place
        self.per_token = per_token
        KL = w.T * w.K if per_token else w.K  # entries resolved per request
        lay = self.lay = W.layout(w)
        has_host = bool((lay.page_host >= 0).any())
        dtype = hs.HS_BF16 if w.dtype == "bf16" else hs.HS_FP8_E4M3_ROWSCALE
        self.pool = hs.Pool(dtype=dtype, n_gpu_blocks=lay.n_gpu_blocks,
                            n_host_blocks=lay.n_host_blocks if has_host else 0,
                            max_requests=w.B, max_ctx=w.ctx, max_topk=KL,
                            hot_rows=w.hot_rows, stream=stream)
        for r in range(w.B):
            self.pool.request_init(r, w.ctx)
            self.pool.page_map_range(r, 0, lay.page_gpu[r], lay.page_host[r])
            self.pool.hot_lease(r, lay.hot_blocks[r])
        W.fill_rows(w.dtype, self.pool.gpu_rows(), self.pool.gpu_scales(), W.row_seed(w, "gpu"))
        if has_host:
            hr = torch.from_numpy(self.pool.host_rows())
            hsc = self.pool.host_scales()
            W.fill_rows(w.dtype, hr, None if hsc is None else torch.from_numpy(hsc),
                        W.row_seed(w, "host"), gen_device="cuda")
        torch.cuda.synchronize()
        dev = "cuda"
        B, rb = w.B, w.row_bytes
        self.req_ids = torch.arange(B, dtype=torch.int32, device=dev)
        self.resolved = torch.empty((B, KL), dtype=torch.int32, device=dev)
        if in_place:
            self.gathered = self.gscale = None
        else:
            self.gathered = torch.empty((B, KL, rb), dtype=torch.uint8, device=dev)
            self.gscale = (torch.empty((B, KL), dtype=torch.float32, device=dev)
                           if w.dtype == "fp8" else None)
        self.counts = torch.empty((B, 3), dtype=torch.int32, device=dev)
        self.out = torch.empty((B, w.T, w.H, 512), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((B, w.T, w.H), dtype=torch.float32, device=dev)
        ws = (hs.hs_decode_workspace_bytes(B * w.T, 1, w.H, w.K) if per_token
              else hs.hs_decode_workspace_bytes(B, w.T, w.H, w.K))
        self.workspace = torch.empty(max(ws, 1), dtype=torch.uint8, device=dev)
        self.topk_host = None
        if build_topk:
            lists = list(W.topk_lists(w))
            if per_token:
                lists = [W.token_lists(w, b, s) for s, b in enumerate(lists)]
            self.topk_host = np.stack(lists)
        self.topk = torch.from_numpy(self.topk_host).to(dev) if build_topk else None

    def resolve(self, step: int, topk=None, stream=None):
        t = self.topk[step] if topk is None else topk
        if self.per_token:
            self.pool.resolve_topk_union(self.req_ids, t, self.resolved, self.gathered,
                                         self.gscale, self.counts, stream)
        else:
            self.pool.resolve_topk(self.req_ids, t, self.resolved, self.gathered, self.gscale,
                                   self.counts, stream)

    def decode(self, step: int, q, topk=None, stream=None, sm_scale=None):
        t = self.topk[step] if topk is None else topk
        sc = self.w.sm_scale if sm_scale is None else sm_scale
        if self.per_token:
            self.pool.sparse_mla_decode_per_token(q, self.gathered, self.gscale, self.resolved,
                                                  t, self.req_ids, sc, self.out, self.lse,
                                                  self.workspace, stream)
        else:
            self.pool.sparse_mla_decode(q, self.gathered, self.gscale, self.resolved, t,
                                        self.req_ids, sc, self.out, self.lse, self.workspace,
                                        stream)


class GpuAgent:
    """The agent mix in a GPU pool: all pages have a GPU block and a host copy;
    each step maps only the pages its residency state keeps resident."""

    def __init__(self, w: "W.AgentMix", stream=None, in_place: bool = False):
        self.w = w
        self.in_place = in_place
        lay = self.lay = W.agent_layout(w)
        self.pool = hs.Pool(dtype=hs.HS_FP8_E4M3_ROWSCALE if w.dtype == "fp8" else hs.HS_BF16,
                            n_gpu_blocks=lay.n_gpu_blocks, n_host_blocks=lay.n_host_blocks,
                            max_requests=w.B, max_ctx=w.ctx, max_topk=w.K, hot_rows=w.hot_rows,
                            stream=stream)
        for r in range(w.B):
            self.pool.request_init(r, w.first)
            self.pool.hot_lease(r, lay.hot_blocks[r])
        rows, scales = self.pool.gpu_rows(), self.pool.gpu_scales()
        W.fill_rows(w.dtype, rows, scales, W.row_seed(w, "gpu"))  # hot blocks: arbitrary start
        hr = torch.from_numpy(self.pool.host_rows())
        hsc = self.pool.host_scales()
        hst = None if hsc is None else torch.from_numpy(hsc)
        W.fill_rows(w.dtype, hr, hst, W.row_seed(w, "host"), gen_device="cuda")
        n = lay.n_host_blocks * 64  # GPU page blocks hold the same rows as their host copies
        rows[:n].copy_(hr[:n])
        if scales is not None:
            scales[:n].copy_(hst[:n])
        torch.cuda.synchronize()
        self.page_gpu = np.full((w.B, w.pages), -1, np.int32)
        dev = "cuda"
        B, K, rb = w.B, w.K, w.row_bytes
        self.req_ids = torch.arange(B, dtype=torch.int32, device=dev)
        self.ctx = torch.empty(B, dtype=torch.int32, device=dev)
        self.resolved = torch.empty((B, K), dtype=torch.int32, device=dev)
        if in_place:
            self.gathered = self.gscale = None
        else:
            self.gathered = torch.empty((B, K, rb), dtype=torch.uint8, device=dev)
            self.gscale = (torch.empty((B, K), dtype=torch.float32, device=dev)
                           if w.dtype == "fp8" else None)
        self.counts = torch.empty((B, 3), dtype=torch.int32, device=dev)
        self.out = torch.empty((B, w.T, w.H, 512), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((B, w.T, w.H), dtype=torch.float32, device=dev)
        ws = hs.hs_decode_workspace_bytes(B, w.T, w.H, K)
        self.workspace = torch.empty(max(ws, 1), dtype=torch.uint8, device=dev)

    def apply(self, st: "W.AgentStep"):
        """Context lengths and the pages whose residency changed (host bookkeeping)."""
        self.ctx.copy_(torch.from_numpy(st.ctx))
        self.pool.set_ctx_lens(self.ctx)
        for r in range(self.w.B):
            diff = np.nonzero(st.page_gpu[r] != self.page_gpu[r])[0]
            if diff.size:
                a, b = int(diff[0]), int(diff[-1]) + 1
                self.pool.page_map_range(r, a, st.page_gpu[r, a:b], self.lay.page_host[r, a:b])
        self.page_gpu = st.page_gpu.copy()

    def resolve(self, topk, stream=None):
        self.pool.resolve_topk(self.req_ids, topk, self.resolved, self.gathered, self.gscale,
                               self.counts, stream)

    def decode(self, q, topk, stream=None):
        self.pool.sparse_mla_decode(q, self.gathered, self.gscale, self.resolved, topk,
                                    self.req_ids, self.w.sm_scale, self.out, self.lse,
                                    self.workspace, stream)
