"""Seeded synthetic inputs for the tiered sparse-MLA decode path.

This module is the only code shared by the CUDA path's harness (tests,
``bench.py``) and by the CPU oracle's harness. It produces *inputs* only:
page layouts, top-K index lists, latent rows and queries. It contains none of
the method's arithmetic (no resolve, no LRU, no attention).

Workloads follow the shapes of the "vLLM Hybrid HiSparse" pages:

* 64-token pages in one shared block pool ("vLLM GLM 5.3 优化：混合 HiSparse 卸载",
  section 混合 HiSparse 的技术实现; "vLLM Hybrid HiSparse：稀疏MLA破解长上下文显存瓶颈",
  section 分级内存的运作机制);
* latent rows of 576 elements (512 "nope" + 64 "rope"), BF16, or FP8 e4m3 with
  one fp32 scale per row (the FP8 KV cache of the 性能基准测试 section);
* a hot buffer of 2x top-K rows per request (关键架构细节, 热缓冲区);
* the agent mix shaped like the multi-turn benchmark of 性能基准测试 (13 turns,
  74,160-token first turn, +753 tokens per later turn, 220 output tokens,
  MTP3). The traces themselves are not available; only their shape is used.

Recipe (all seeded, seed = 20261202 + workload index):

* rows: N(0,1) float32, stored as BF16 (round to nearest even) or as FP8 e4m3
  with scale = amax(|row|)/448 per row (torch's RNE conversion);
* q: N(0,1), BF16;
* "Zipf(s) over positions": rank order is a per-request seeded permutation of
  the candidate positions, fixed across steps; P(rank i) ∝ i^-s. Sampling
  without replacement is successive sampling, done as i.i.d. draws with
  repeats discarded (the same distribution as Efraimidis–Spirakis top-k of
  u^(1/w));
* reuse fraction f: round(f·n) entries drawn uniformly without replacement
  from the previous step's list, the rest fresh and distinct;
* each list is shuffled, since an indexer emits its top-K in score order, not
  position order.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field
from typing import Iterator, Optional

import numpy as np

SEED_BASE = 20261202
PAGE = 64
NOPE = 512
ROPE = 64
DIM = NOPE + ROPE          # 576-wide latent row
FP8_MAX = 448.0            # largest finite e4m3fn value


@dataclass(frozen=True)
class Workload:
    """One decode workload: a batch of requests, their tiers and their top-K lists."""

    name: str
    index: int                 # seed = SEED_BASE + index
    B: int                     # requests in the batch
    ctx: int                   # context length per request (tokens)
    H: int                     # heads
    T: int                     # query tokens per step (1 + MTP draft tokens)
    K: int                     # top-K
    hot_rows: int              # hot-buffer capacity per request (rows)
    dtype: str                 # "bf16" or "fp8"
    steps: int                 # decode steps
    residency: str             # "all", "none", "tail", "from_page"
    resident_tail: int = 0     # tokens resident at the end ("tail")
    resident_from_page: int = 0  # first resident page ("from_page")
    topk_kind: str = "zipf_tail"  # "zipf_tail", "reuse_zipf", "reuse_uniform"
    tail: int = 0              # last `tail` tokens always selected (zipf kinds)
    zipf_s: float = 1.0
    reuse: float = 0.0

    # ---------------------------------------------------------------- derived
    @property
    def seed(self) -> int:
        return SEED_BASE + self.index

    @property
    def pages(self) -> int:
        return (self.ctx + PAGE - 1) // PAGE

    @property
    def row_bytes(self) -> int:
        return DIM * (2 if self.dtype == "bf16" else 1)

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(DIM)

    def scaled(self, **kw) -> "Workload":
        """A copy with some fields replaced (smaller test sizes)."""
        return dataclasses.replace(self, **kw)

    def resident_pages(self) -> np.ndarray:
        """Boolean [pages]: which pages of every request are GPU-resident."""
        res = np.zeros(self.pages, dtype=bool)
        if self.residency == "all":
            res[:] = True
        elif self.residency == "tail":
            res[self.pages - self.resident_tail // PAGE:] = True
        elif self.residency == "from_page":
            res[self.resident_from_page:] = True
        elif self.residency != "none":
            raise ValueError(self.residency)
        return res


WORKLOADS = {
    "tiny": Workload(
        name="tiny", index=0, B=1, ctx=4096, H=16, T=1, K=256, hot_rows=512,
        dtype="bf16", steps=8, residency="from_page", resident_from_page=32,
        topk_kind="zipf_tail", tail=64, zipf_s=1.1),
    "resident": Workload(
        name="resident", index=1, B=32, ctx=131072, H=128, T=1, K=2048,
        hot_rows=4096, dtype="bf16", steps=64, residency="all",
        topk_kind="zipf_tail", tail=128, zipf_s=1.0),
    "hybrid": Workload(
        name="hybrid", index=2, B=16, ctx=1048576, H=128, T=4, K=2048,
        hot_rows=4096, dtype="fp8", steps=128, residency="tail",
        resident_tail=32768, topk_kind="reuse_zipf", tail=128, zipf_s=1.0,
        reuse=0.7),
    "noresident": Workload(
        name="noresident", index=3, B=32, ctx=524288, H=128, T=1, K=2048,
        hot_rows=4096, dtype="fp8", steps=32, residency="none",
        topk_kind="reuse_uniform", reuse=0.5),
}


# ------------------------------------------------------------------ layout
@dataclass
class Layout:
    """Block numbering of one workload in the GPU pool and the host arena."""

    page_gpu: np.ndarray       # int32 [B][pages], -1 = not resident
    page_host: np.ndarray      # int32 [B][pages], -1 = no host copy
    hot_blocks: np.ndarray     # int32 [B][hot_rows/64], blocks leased from the pool
    n_gpu_blocks: int
    n_host_blocks: int


def layout(w: Workload) -> Layout:
    """Request r's resident pages get consecutive GPU blocks, requests in order;
    the hot-buffer blocks are leased from the same pool after all page blocks.
    Non-resident pages get consecutive host-arena blocks."""
    res = w.resident_pages()
    n_res, n_host = int(res.sum()), int((~res).sum())
    page_gpu = np.full((w.B, w.pages), -1, np.int32)
    page_host = np.full((w.B, w.pages), -1, np.int32)
    for r in range(w.B):
        page_gpu[r, res] = r * n_res + np.arange(n_res, dtype=np.int32)
        page_host[r, ~res] = r * n_host + np.arange(n_host, dtype=np.int32)
    hb = w.hot_rows // PAGE
    base = w.B * n_res
    hot_blocks = (base + np.arange(w.B * hb, dtype=np.int32)).reshape(w.B, hb)
    return Layout(page_gpu, page_host, hot_blocks,
                  n_gpu_blocks=base + w.B * hb, n_host_blocks=max(1, w.B * n_host))


# ------------------------------------------------------------------ top-K
class _Zipf:
    """Seeded Zipf(s) sampler over a per-request permutation of candidates."""

    def __init__(self, n: int, s: float):
        w = np.arange(1, n + 1, dtype=np.float64) ** (-s)
        c = np.cumsum(w)
        self.cdf = c / c[-1]
        self.n = n

    def draw(self, rng, perm, k, taken: np.ndarray) -> np.ndarray:
        """k distinct positions not marked in `taken` (a bool mask over positions);
        marks them in `taken`."""
        out = []
        need = k
        while need > 0:
            u = rng.random(max(2 * need, 64))
            ranks = np.minimum(np.searchsorted(self.cdf, u, side="right"), self.n - 1)
            pos = perm[ranks]
            _, first = np.unique(pos, return_index=True)
            pos = pos[np.sort(first)]
            pos = pos[~taken[pos]][:need]
            taken[pos] = True
            out.append(pos)
            need -= len(pos)
        return np.concatenate(out).astype(np.int32)


def _uniform_distinct(rng, lo, hi, k, taken):
    out = []
    need = k
    while need > 0:
        pos = rng.integers(lo, hi, size=max(2 * need, 64))
        _, first = np.unique(pos, return_index=True)
        pos = pos[np.sort(first)]
        pos = pos[~taken[pos]][:need]
        taken[pos] = True
        out.append(pos)
        need -= len(pos)
    return np.concatenate(out).astype(np.int32)


def topk_lists(w: Workload) -> Iterator[np.ndarray]:
    """Yields one int32 [B][K] top-K list per decode step (positions, unsorted)."""
    rng = np.random.Generator(np.random.PCG64(w.seed))
    L = w.ctx
    if w.topk_kind == "zipf_tail":
        cand = L - w.tail
        zipf = _Zipf(cand, w.zipf_s)
        perms = [rng.permutation(cand).astype(np.int32) for _ in range(w.B)]
        taken = np.zeros(L, dtype=bool)
        for _ in range(w.steps):
            out = np.empty((w.B, w.K), np.int32)
            for r in range(w.B):
                tail = np.arange(L - w.tail, L, dtype=np.int32)
                z = zipf.draw(rng, perms[r], w.K - w.tail, taken)
                taken[z] = False
                lst = np.concatenate([tail, z])
                out[r] = lst[rng.permutation(w.K)]
            yield out
    elif w.topk_kind == "reuse_zipf":
        cold = L - w.resident_tail
        zipf = _Zipf(cold, w.zipf_s)
        perms = [rng.permutation(cold).astype(np.int32) for _ in range(w.B)]
        taken = np.zeros(L, dtype=bool)
        prev = None
        n_reuse = int(round(w.reuse * w.K))
        for _ in range(w.steps):
            out = np.empty((w.B, w.K), np.int32)
            for r in range(w.B):
                if prev is None:
                    tail = np.arange(L - w.tail, L, dtype=np.int32)
                    taken[tail] = True
                    z = zipf.draw(rng, perms[r], w.K - w.tail, taken)
                    lst = np.concatenate([tail, z])
                else:
                    keep = rng.choice(prev[r], size=n_reuse, replace=False).astype(np.int32)
                    taken[keep] = True
                    z = zipf.draw(rng, perms[r], w.K - n_reuse, taken)
                    lst = np.concatenate([keep, z])
                taken[lst] = False
                out[r] = lst[rng.permutation(w.K)]
            prev = out
            yield out
    elif w.topk_kind == "reuse_uniform":
        taken = np.zeros(L, dtype=bool)
        prev = None
        n_reuse = int(round(w.reuse * w.K))
        for _ in range(w.steps):
            out = np.empty((w.B, w.K), np.int32)
            for r in range(w.B):
                if prev is None:
                    lst = _uniform_distinct(rng, 0, L, w.K, taken)
                else:
                    keep = rng.choice(prev[r], size=n_reuse, replace=False).astype(np.int32)
                    taken[keep] = True
                    z = _uniform_distinct(rng, 0, L, w.K - n_reuse, taken)
                    lst = np.concatenate([keep, z])
                taken[lst] = False
                out[r] = lst[rng.permutation(w.K)]
            prev = out
            yield out
    else:
        raise ValueError(w.topk_kind)


def token_lists(w: Workload, base: np.ndarray, step: int, fresh: float = 0.1) -> np.ndarray:
    """One top-K list per query token for one decode step: int32 [B][T][K].

    Token 0 keeps the step's list `base` ([B][K]); token t >= 1 (query position
    L - T + t) keeps it too except for round(fresh*K) entries, at seeded random
    indices, replaced by distinct positions drawn uniformly from [0, L - T + t]
    that are not already in that token's list. Lists of different tokens
    therefore overlap in about (1 - fresh) of their entries."""
    rng = np.random.Generator(np.random.PCG64([w.seed, 7, step]))
    B, K = base.shape
    L = w.ctx
    n_new = int(round(fresh * K))
    out = np.empty((B, w.T, K), np.int32)
    taken = np.zeros(L, dtype=bool)
    for r in range(B):
        out[r, 0] = base[r]
        for t in range(1, w.T):
            lst = base[r].copy()
            idx = rng.choice(K, size=n_new, replace=False)
            taken[lst] = True
            new = _uniform_distinct(rng, 0, L - w.T + t + 1, n_new, taken)
            taken[lst] = False
            taken[new] = False
            lst[idx] = new
            out[r, t] = lst
    return out


# ------------------------------------------------------------------ rows, q
def fill_rows(dtype: str, rows, scales, seed: int, chunk_rows: int = 1 << 20, gen_device=None):
    """Fill `rows` (torch uint8 [n, row_bytes], any device) with N(0,1) latent rows.

    BF16: the float32 draws rounded to bfloat16. FP8: scale = amax/448 per row,
    codes = e4m3fn(x / scale) with round-to-nearest-even; the scale goes to
    `scales` (torch float32 [n]) in a parallel array. The draws are made on
    `gen_device` (default: the device of `rows`) and copied; the values are
    deterministic for a given seed and generating device."""
    import torch
    n = rows.shape[0]
    dev = torch.device(gen_device) if gen_device is not None else rows.device
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    for a in range(0, n, chunk_rows):
        b = min(n, a + chunk_rows)
        x = torch.randn((b - a, DIM), generator=g, device=dev, dtype=torch.float32)
        if dtype == "bf16":
            rows[a:b].copy_(x.to(torch.bfloat16).view(torch.uint8))
        else:
            s = x.abs().amax(dim=1) / FP8_MAX
            rows[a:b].copy_((x / s[:, None]).to(torch.float8_e4m3fn).view(torch.uint8))
            scales[a:b].copy_(s)


def make_q(w: Workload, step: int, device="cpu"):
    """Queries for one decode step: bf16 [B][T][H][576], N(0,1)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(w.seed * 1000003 + 7919 * (step + 1))
    x = torch.randn((w.B, w.T, w.H, DIM), generator=g, device=device, dtype=torch.float32)
    return x.to(torch.bfloat16)


def row_seed(w: Workload, tier: str) -> int:
    return w.seed * 1000003 + (1 if tier == "gpu" else 2)


# ------------------------------------------------------------------ agent mix
@dataclass(frozen=True)
class AgentMix:
    """Multi-turn agent-shaped mix, shaped like the benchmark of [A] 性能基准测试
    (13 turns, 74,160-token first turn, +753 prefill tokens per later turn, 220
    output tokens per turn, MTP3, FP8 KV). The traces themselves are not
    available; only this shape is used.

    Residency follows a seeded pressure schedule: u_r ~ U(0,1) once per request,
    pi_t = (t-1)/(turns-1); in turn t a request is full-resident if u_r >= pi_t,
    hybrid (resident tail of `resident_tail` tokens) if u_r >= pi_t/2, else none
    (only the pages being written are resident). States only move full ->
    hybrid -> none. Every page has a host copy (finished pages are copied to
    host while still served from the GPU, [A] 关键架构细节, 主动复制), so a page
    that stops being resident is still readable from host memory.

    Decode step s of a turn that starts with `start` tokens sees context
    L = start + T*(s+1): the T query tokens (1 + 3 MTP drafts, all accepted)
    sit at positions L-T .. L-1."""

    name: str = "agent"
    index: int = 4
    B: int = 32
    turns: int = 13
    first: int = 74160
    per_turn: int = 753
    out_tokens: int = 220
    H: int = 128
    T: int = 4
    K: int = 2048
    hot_rows: int = 4096
    dtype: str = "fp8"
    resident_tail: int = 32768
    tail: int = 128          # last tokens always selected
    reuse: float = 0.7
    zipf_s: float = 1.0

    @property
    def seed(self) -> int:
        return SEED_BASE + self.index

    @property
    def steps_per_turn(self) -> int:
        return self.out_tokens // self.T

    @property
    def steps(self) -> int:
        return self.turns * self.steps_per_turn

    @property
    def ctx(self) -> int:  # largest context any step sees
        return self.turn_start(self.turns) + self.T * self.steps_per_turn

    @property
    def pages(self) -> int:
        return (self.ctx + PAGE - 1) // PAGE

    @property
    def row_bytes(self) -> int:
        return DIM * (2 if self.dtype == "bf16" else 1)

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(DIM)

    def turn_start(self, t: int) -> int:
        return self.first + (t - 1) * (self.per_turn + self.out_tokens)

    def scaled(self, **kw) -> "AgentMix":
        return dataclasses.replace(self, **kw)


@dataclass
class AgentStep:
    turn: int
    step: int
    ctx: np.ndarray        # int32 [B], context length at this step
    state: np.ndarray      # int8 [B]: 0 full, 1 hybrid, 2 none
    page_gpu: np.ndarray   # int32 [B][pages], -1 = not resident
    topk: np.ndarray       # int32 [B][K]


def agent_layout(w: AgentMix) -> Layout:
    """Every page of request r has GPU block r*pages + page and host block
    r*pages + page (the host copy); hot-buffer blocks follow all page blocks."""
    P = w.pages
    ids = (np.arange(w.B, dtype=np.int32)[:, None] * P + np.arange(P, dtype=np.int32)[None, :])
    hb = w.hot_rows // PAGE
    base = w.B * P
    hot = (base + np.arange(w.B * hb, dtype=np.int32)).reshape(w.B, hb)
    return Layout(ids.copy(), ids.copy(), hot, n_gpu_blocks=base + w.B * hb, n_host_blocks=w.B * P)


def agent_steps(w: AgentMix) -> Iterator[AgentStep]:
    """The agent mix, one decode step at a time (residency, context, top-K)."""
    rng = np.random.Generator(np.random.PCG64(w.seed))
    u = rng.random(w.B)
    lay = agent_layout(w)
    P = w.pages
    full_cand = w.ctx - w.tail
    zipf = _Zipf(full_cand, w.zipf_s)
    perms = [rng.permutation(full_cand).astype(np.int32) for _ in range(w.B)]
    taken = np.zeros(w.ctx, dtype=bool)
    state = np.zeros(w.B, np.int8)
    prev = [None] * w.B
    n_body = w.K - w.tail
    n_reuse = int(round(w.reuse * n_body))
    page_idx = np.arange(P)
    for t in range(1, w.turns + 1):
        pi = (t - 1) / max(1, w.turns - 1)
        new_state = np.where(u >= pi, 0, np.where(u >= pi / 2, 1, 2)).astype(np.int8)
        state = np.maximum(state, new_state)  # full -> hybrid -> none only
        start = w.turn_start(t)
        for s in range(w.steps_per_turn):
            L = start + w.T * (s + 1)
            ctx = np.full(w.B, L, np.int32)
            first_res = np.where(state == 0, 0,
                                 np.where(state == 1, max(0, L - w.resident_tail) // PAGE,
                                          (L - w.T) // PAGE))
            page_gpu = np.where(page_idx[None, :] >= first_res[:, None], lay.page_gpu, -1)
            page_gpu = page_gpu.astype(np.int32)
            topk = np.empty((w.B, w.K), np.int32)
            limit = L - w.tail  # body positions lie in [0, L - tail)
            for r in range(w.B):
                tail = np.arange(limit, L, dtype=np.int32)
                keep = np.empty(0, np.int32)
                if prev[r] is not None:
                    cand = prev[r][prev[r] < limit]
                    k = min(n_reuse, len(cand))
                    keep = rng.choice(cand, size=k, replace=False).astype(np.int32)
                taken[keep] = True
                fresh = _zipf_below(zipf, rng, perms[r], n_body - len(keep), taken, limit)
                body = np.concatenate([keep, fresh])
                taken[body] = False
                prev[r] = body
                lst = np.concatenate([tail, body])
                topk[r] = lst[rng.permutation(w.K)]
            yield AgentStep(t, s, ctx, state.copy(), page_gpu, topk)


def _zipf_below(zipf: _Zipf, rng, perm, k, taken, limit) -> np.ndarray:
    """k distinct Zipf draws among positions < limit not marked in `taken`."""
    out = []
    need = k
    while need > 0:
        u = rng.random(max(4 * need, 64))
        ranks = np.minimum(np.searchsorted(zipf.cdf, u, side="right"), zipf.n - 1)
        pos = perm[ranks]
        pos = pos[pos < limit]
        _, first = np.unique(pos, return_index=True)
        pos = pos[np.sort(first)]
        pos = pos[~taken[pos]][:need]
        taken[pos] = True
        out.append(pos)
        need -= len(pos)
    res = np.concatenate(out).astype(np.int32) if out else np.empty(0, np.int32)
    taken[res] = False
    return res
