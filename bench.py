"""Benchmark of the tiered sparse-MLA decode hot path on GB300.

One step = one decode step of the whole path over one batch: hs_resolve_topk
(fused resolve of 32 top-K lists against the tiered cache) followed by
hs_sparse_mla_decode (attention over the 2048 selected latent rows per request).

Workload: the fully resident configuration -- 32 requests x 131,072 tokens,
64-token pages all GPU-resident, BF16 576-wide latent rows N(0,1), 128 heads,
1 query token, top-K = 2048 (last 128 tokens + Zipf(1.0) over the rest),
64 pregenerated decode steps cycled. L2 is flushed before every timed step
(a 256 MiB write, then a 256 MiB read of other data so that no write-back of
the flush lands in the timed kernels); per-step CUDA events exclude the flush.

Prints one JSON line. --impl reference times the CPU oracle instead (bounded
sample of the same workload, on the host cores).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import select
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "resolved top-K rows/s & sparse-MLA decode steps/s; % of HBM/host-link roofline"
WORKLOAD = "resident"
WORKLOAD_DESC = ("fully resident: 32 requests x 131072-token context, 64-token pages all "
                 "GPU-resident, BF16 576-wide latent rows, 128 heads, 1 query token, "
                 "top-K 2048 (last 128 + Zipf(1.0)), hot buffer 4096 rows/request")


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float) -> float:
    """The largest value over all ranks (CUDA tensor under NCCL, CPU under gloo)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, ms_per_step_max: float) -> float:
    """Units all ranks processed per second, timed by the slowest rank."""
    return units_per_rank * world / (ms_per_step_max * 1e-3)


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d.get("hbm_gbs"), d.get("bf16_tflops"), "measured"
    return 6800.0, 1900.0, "fallback"


def _traffic(kernel: str, src: str, in_place: bool):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's
    source is unchanged since the capture and the rows reached attention the
    same way (in place or gathered) as in the capture (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel)
    if not d:
        return None
    sha = hashlib.sha256(open(os.path.join(ROOT, src), "rb").read()).hexdigest()[:16]
    if d.get("source_sha") != sha or d.get("in_place") != in_place:
        return None
    return d["dram_bytes_per_launch"]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.p = None

    def __enter__(self):
        self.first = ""
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.p = None
        if self.p is not None:
            # the sampler's start-up (its own GPU queries) before the timed
            # steps, not inside them: wait for its first sample (2 s at most)
            ready, _, _ = select.select([self.p.stdout], [], [], 2.0)
            if ready:
                self.first = self.p.stdout.readline()
        return self

    def __exit__(self, *a):
        self.out = self.first
        if self.p is not None:
            self.p.terminate()
            try:
                rest, _ = self.p.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()
                rest, _ = self.p.communicate()
            self.out += rest or ""

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (getattr(self, "out", "") or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def run_config(desc, w, ws, layers=1, in_place=False):
    """The line's config: the workload and how it is run (the same dict for
    the GPU arm and the CPU-oracle arm on the headline workload)."""
    return {"workload": desc, "global_batch": w.B * ws, "top_k": w.K, "layers": layers,
            "heads": w.H, "query_tokens": w.T, "ctx": w.ctx,
            "parallelism": f"replicas x{ws} (requests sharded by rank, no collective)",
            "rows": ("read in place from the pool by attention (no gathered buffer)"
                     if in_place else "gathered by the resolve, then read by attention"),
            "l2": ("GPU arm: flushed before every timed step, 256 MiB written then 256 MiB of "
                   "other data read (clean, cold L2), the flush outside the events; CPU-oracle "
                   "arm: not applicable"),
            "host_arena": ("GPU arm: read once through the GPU's mapping before the warm-up steps "
                           "(the first GPU reads of a pinned host page are slow; a serving "
                           "process reads its arena for its whole life)")}


def algorithmic(w, counts_sum, in_place=False, per_token=None):
    """Algorithmic bytes / flops of one step (per-unit figures x units).

    Gathered rows: the resolve reads every hit row and writes every row to the
    gathered buffer (plus the miss rows into their slots); in place it writes
    only the miss rows into their slots. Either way attention reads each
    selected row once.

    per_token = (distinct rows, distinct misses) per step when every query
    token has its own list: entries = B*T*K; a row that several tokens select
    is read from HBM (and a missing one from the host) once."""
    B, K, rb = w.B, w.K, w.row_bytes
    res, hot, miss = counts_sum
    if per_token is None:
        rows = entries = B * K
    else:
        entries = B * w.T * K
        rows, miss = per_token
    if in_place:
        resolve_hbm = miss * rb + entries * 12
    else:
        resolve_hbm = (res + hot) * rb + entries * rb + miss * rb + entries * 12
    resolve_link = miss * rb
    q = B * w.T * w.H * 576 * 2
    out = B * w.T * w.H * 512 * 2 + B * w.T * w.H * 4
    decode_bytes = rows * rb + q + out + entries * 8
    flops = 2.0 * B * w.T * w.H * K * (576 + 512)
    return resolve_hbm, resolve_link, decode_bytes, flops


# ------------------------------------------------------------------ GPU arm
DESCS = {
    "resident": WORKLOAD_DESC,
    "tiny": ("tiny: 1 request x 4096-token context, pages 0-31 host-only and 32-63 resident, "
             "BF16, 16 heads, 1 query token, top-K 256, hot buffer 512 rows"),
    "hybrid": ("hybrid residency: 16 requests x 1,048,576-token context, last 32K tokens resident, "
               "older pages in pinned host memory, FP8 e4m3 rows + fp32 scale, hot buffer 4096 "
               "rows/request, 128 heads, MTP3 (4 query tokens), top-K 2048, 70% reuse per step"),
    "noresident": ("no-resident prefix reuse: 32 requests x 524,288-token context all host-only, "
                   "empty hot buffer at start, FP8 rows, 128 heads, top-K 2048 uniform, 50% reuse"),
    "agent": ("multi-turn agent-shaped mix: 32 requests x 13 turns (74,160-token first turn, +753 "
              "per turn, 220 output tokens), MTP3, FP8 rows, 128 heads, top-K 2048, residency "
              "full/hybrid/none from a seeded pressure schedule"),
}
DEFAULT_STEPS = {"resident": 2000, "tiny": 2000, "hybrid": 512, "noresident": 256, "agent": 715}
# How each workload's rows reach attention by default: read in place from the
# pool (no gathered buffer) where that gives the shorter step on a GB300,
# gathered by the resolve elsewhere (measured, steps/s in place against
# gathered: resident 17.7K / 13.6K, tiny 27.4K / 25.7K, hybrid 8.0K / 8.4K,
# no-resident and agent mix within 1%)
DEFAULT_IN_PLACE = {"resident": True, "tiny": True, "hybrid": False, "noresident": False,
                    "agent": False}


def _link_peak_gbs(to_host: bool = False):
    """Measured pinned host <-> device copy bandwidth (best of 3, 256 MiB)."""
    import torch
    h = torch.empty(256 << 20, dtype=torch.uint8).pin_memory()
    d = torch.empty_like(h, device="cuda")
    best = 0.0
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        if to_host:
            h.copy_(d, non_blocking=True)
        else:
            d.copy_(h, non_blocking=True)
        e1.record()
        torch.cuda.synchronize()
        best = max(best, h.numel() / (e0.elapsed_time(e1) * 1e-3) / 1e9)
    return best


def _touch_host_arenas(pools):
    """Reads every pool's pinned host arena once through the GPU's mapping
    (untimed). The GPU's first reads of a pinned host page run at a small
    fraction of the link's rate, later ones at full rate; a serving process
    reads the same arena for its whole life, so the timed steps start warm."""
    import torch
    for pool in pools:
        rows = pool.host_rows_device()
        if rows is not None:
            rows.max()
        scales = pool.host_scales_device()
        if scales is not None:
            scales.sum()
    torch.cuda.synchronize()


def measure(args, name, steps, with_e2e=False):
    """Times `steps` decode steps of workload `name` (resolve + decode per
    step, CUDA events on the launching stream, cold L2) and returns the
    bench line's fields for it. with_e2e adds the end-to-end figure through
    the C ABI with host buffers."""
    import numpy as np
    import torch
    import tiered_sparse_mla_gb300 as hs
    import workloads as W
    from harness import GpuAgent, GpuWorkload

    ws, rank, local = _dist()
    agent = name == "agent"
    w = W.AgentMix() if agent else W.WORKLOADS[name]
    if args.batch and args.batch != w.B:
        w = w.scaled(B=args.batch)
    if args.ctx and not agent and args.ctx != w.ctx:
        # a shorter context keeps the decode work (K rows per request) and
        # shrinks the pool, for profiler captures; not a bench line
        w = w.scaled(ctx=args.ctx)
    per_token = bool(args.per_token)
    if per_token and (agent or w.T < 2):
        raise SystemExit("--per-token needs a workload with several query tokens (hybrid)")
    L = max(1, args.layers)
    if L > 1 and (agent or per_token):
        raise SystemExit("--layers applies to the single-list workloads")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        if agent:
            gw = GpuAgent(w, stream=stream, in_place=args.in_place)
            plan = list(W.agent_steps(w))
            lists = [torch.from_numpy(st.topk).to("cuda") for st in plan]
        else:
            gw = GpuWorkload(w, stream=stream, in_place=args.in_place, per_token=per_token)
            plan = None
            lists = [gw.topk[s] for s in range(w.steps)]
            if per_token:
                # distinct selected positions of each step (the rows attention
                # must read at least once)
                uniq = [sum(len(np.unique(gw.topk_host[s][b][gw.topk_host[s][b] >= 0]))
                            for b in range(w.B)) for s in range(w.steps)]
        gws, group = [gw], None
        if L > 1:
            # layers 1..L-1: pools of the same shape with their own seeds; one
            # resolve launch covers all layers, each layer then decodes on its own
            gws += [GpuWorkload(w.scaled(index=w.index + 100 * l), stream=stream,
                                in_place=args.in_place) for l in range(1, L)]
            res_all = torch.empty((L, w.B, w.K), dtype=torch.int32, device="cuda")
            gat_all = (None if args.in_place else
                       torch.empty((L, w.B, w.K, w.row_bytes), dtype=torch.uint8, device="cuda"))
            gsc_all = (torch.empty((L, w.B, w.K), dtype=torch.float32, device="cuda")
                       if (w.dtype == "fp8" and not args.in_place) else None)
            cnt_all = torch.empty((L, w.B, 3), dtype=torch.int32, device="cuda")
            for l, x in enumerate(gws):
                x.resolved, x.counts = res_all[l], cnt_all[l]
                x.gathered = None if gat_all is None else gat_all[l]
                x.gscale = None if gsc_all is None else gsc_all[l]
            lists = [torch.stack([x.topk[s] for x in gws]).contiguous() for s in range(w.steps)]
            group = hs.hs_layer_group_create([x.pool for x in gws])
        nq = min(len(lists), 16)
        qs = [W.make_q(w, s, device="cuda") for s in range(nq)]
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        flush_rd = torch.ones(64 << 20, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    _touch_host_arenas([x.pool for x in gws])
    if agent:
        gw.apply(plan[0])
    snaps = [x.pool.snapshot() for x in gws]
    n_lists = len(lists)

    def l2_flush():
        # write 256 MiB (evicts everything), then read 256 MiB of other data so
        # that the write-backs happen here and not inside the timed kernels
        flush.zero_()
        flush_rd.sum()

    def prepare(s):
        """Untimed bookkeeping before step s: residency/context updates of the
        agent mix, and the hot-buffer state restored when the step list wraps."""
        i = s % n_lists
        if i == 0 and s > 0:
            torch.cuda.synchronize()
            for x, sn in zip(gws, snaps):
                x.pool.restore(sn)
        if agent:
            gw.apply(plan[i])

    def step(s, ev=None):
        t = lists[s % n_lists]
        q = qs[s % nq]
        if ev is not None:
            ev[0].record(stream)
        if L > 1:
            hs.hs_resolve_topk_layers(group, gw.req_ids, t, res_all, gat_all, gsc_all, cnt_all,
                                      stream)
        elif per_token:
            gw.pool.resolve_topk_union(gw.req_ids, t, gw.resolved, gw.gathered, gw.gscale,
                                       gw.counts, stream)
        else:
            gw.pool.resolve_topk(gw.req_ids, t, gw.resolved, gw.gathered, gw.gscale, gw.counts,
                                 stream)
        if ev is not None and ev[1] is not None:
            ev[1].record(stream)
        if L > 1:
            for l, x in enumerate(gws):  # the layers' queries: the step's q, reused
                x.pool.sparse_mla_decode(q, x.gathered, x.gscale, x.resolved, t[l], x.req_ids,
                                         w.sm_scale, x.out, x.lse, x.workspace, stream)
        elif per_token:
            gw.pool.sparse_mla_decode_per_token(q, gw.gathered, gw.gscale, gw.resolved, t,
                                                gw.req_ids, w.sm_scale, gw.out, gw.lse,
                                                gw.workspace, stream)
        else:
            gw.pool.sparse_mla_decode(q, gw.gathered, gw.gscale, gw.resolved, t, gw.req_ids,
                                      w.sm_scale, gw.out, gw.lse, gw.workspace, stream)
        if ev is not None:
            ev[2].record(stream)

    with torch.cuda.stream(stream):
        for s in range(args.warmup):
            prepare(s)
            l2_flush()
            step(s)
    torch.cuda.synchronize()
    assert all(x.pool.get_error() == 0 for x in gws)
    # Timed steps start from the beginning of the step list and its initial
    # state (restored by each pass).
    # Pass 1 (the timed region of the line): each step timed from before the
    # resolve to after the decode, nothing recorded between the two kernels,
    # so the decode may launch while the resolve runs as it does in use.
    # Pass 2: the same steps from the same state with an event between the
    # kernels, for the per-kernel times (that event keeps the decode from
    # launching early, so pass 2's steps are a few microseconds longer).
    def run_pass(split):
        evs = [[torch.cuda.Event(enable_timing=True),
                torch.cuda.Event(enable_timing=True) if split else None,
                torch.cuda.Event(enable_timing=True)] for _ in range(steps)]
        counts_acc = torch.zeros(3, dtype=torch.int64, device="cuda")
        retagged = torch.zeros((), dtype=torch.int64, device="cuda")
        for x, sn in zip(gws, snaps):
            x.pool.restore(sn)
        if agent:
            gw.apply(plan[0])
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with ClockSampler(local) as clk, torch.cuda.stream(stream):
            # about 1 ms of untimed GPU delay before the first step's events, so
            # that the host is already launching ahead when the timed steps run
            # (otherwise the first steps' events also time the host's launches)
            torch.cuda._sleep(2_000_000)
            torch.cuda.nvtx.range_push("timed_region" if not split else "kernel_split")
            for s in range(steps):
                if s > 0:
                    prepare(s)
                if per_token:
                    tag_prev.copy_(slot_tag)
                l2_flush()
                step(s, evs[s])
                counts_acc += cnt_all.sum((0, 1)) if L > 1 else gw.counts.sum(0)
                if per_token:
                    retagged += (slot_tag != tag_prev).sum()
            torch.cuda.nvtx.range_pop()
            torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        if ws > 1:
            dist.barrier()
        assert gw.pool.get_error() == 0
        return evs, counts_acc, retagged, clk, wall

    # distinct placed misses: each takes one slot and retags it (outside the events)
    slot_tag = gw.pool.tables()["slot_tag"]
    tag_prev = torch.empty_like(slot_tag)
    evs, counts_acc, retagged, clk, wall = run_pass(False)
    cnt_sum = counts_acc.cpu().numpy()
    t_step = [evs[s][0].elapsed_time(evs[s][2]) for s in range(steps)]
    ms_step = max_over_ranks(sum(t_step) / steps)
    steps_per_s = whole_job_rate(1.0, ws, ms_step)
    evs2, _, _, _, _ = run_pass(True)
    t_res = [evs2[s][0].elapsed_time(evs2[s][1]) for s in range(steps)]
    t_dec = [evs2[s][1].elapsed_time(evs2[s][2]) for s in range(steps)]
    res_ms = sum(t_res) / steps
    dec_ms = sum(t_dec) / steps
    rows_per_s = ws * L * w.B * w.K / (res_ms * 1e-3)

    per_step_counts = cnt_sum / steps
    pt = None
    if per_token:
        pt = (sum(uniq[s % n_lists] for s in range(steps)) / steps,
              float(retagged.item()) / steps)
        rows_per_s = ws * w.B * w.T * w.K / (res_ms * 1e-3)
    r_hbm, r_link, d_bytes, flops = algorithmic(w, per_step_counts / L, args.in_place, pt)
    r_hbm, r_link, d_bytes, flops = r_hbm * L, r_link * L, d_bytes * L, flops * L
    hbm_peak, tf_peak, peak_kind = _peaks()
    kernels = {
        "resolve": {"ms": res_ms, "achieved": r_hbm / (res_ms * 1e-3) / 1e9, "unit": "GB/s",
                    "peak": hbm_peak, "bound": "hbm", "bytes_per_launch": r_hbm,
                    "traffic": _traffic("resolve", "tiered_sparse_mla_gb300/csrc/hs_resolve.cu",
                                        args.in_place)},
        "decode": {"ms": dec_ms, "achieved": d_bytes / (dec_ms * 1e-3) / 1e9, "unit": "GB/s",
                   "peak": hbm_peak, "bound": "hbm", "bytes_per_launch": d_bytes,
                   "tflops": flops / (dec_ms * 1e-3) / 1e12,
                   "traffic": _traffic("decode", "tiered_sparse_mla_gb300/csrc/hs_decode.cu",
                                       args.in_place)},
    }
    if name != WORKLOAD or w.B != W.WORKLOADS[WORKLOAD].B or L > 1 or per_token \
            or args.in_place != DEFAULT_IN_PLACE[WORKLOAD]:
        kernels["resolve"]["traffic"] = kernels["decode"]["traffic"] = None  # captured on another workload
    # the decode's roofline time is max(bytes / BW, flops / tensor peak)
    t_bytes = d_bytes / (hbm_peak * 1e9)
    t_flops = flops / (tf_peak * 1e12)
    if t_flops > t_bytes:
        kernels["decode"].update(bound="tensor", achieved=flops / (dec_ms * 1e-3) / 1e12,
                                 unit="TFLOP/s", peak=tf_peak)
    # the resolve's roofline time is max(HBM bytes / BW, miss bytes / host-link BW)
    link_peak = _link_peak_gbs() if r_link > 0 else None
    if r_link > 0 and r_link / (link_peak * 1e9) > r_hbm / (hbm_peak * 1e9):
        kernels["resolve"].update(bound="host-link", achieved=r_link / (res_ms * 1e-3) / 1e9,
                                  peak=round(link_peak, 1), bytes_per_launch=r_link,
                                  hbm_bytes_per_launch=r_hbm)
    top = max(kernels, key=lambda k: kernels[k]["ms"])
    kt = kernels[top]
    src = (f"{peak_kind} (MEASURED_PEAKS.json)" if peak_kind == "measured" else "fallback")
    if kt["bound"] == "host-link":
        src = "measured live: pinned 256 MiB host-to-device copy"
    roofline = {"kernel": top, "bound": kt["bound"], "achieved": round(kt["achieved"], 1),
                "peak": kt["peak"], "unit": kt["unit"],
                "frac": round(kt["achieved"] / kt["peak"], 4), "traffic": kt["traffic"],
                "peak_source": src}

    launches = 1 + L * (1 + (1 if (hs.hs_decode_workspace_bytes(w.B * w.T, 1, w.H, w.K) if per_token
                                   else hs.hs_decode_workspace_bytes(w.B, w.T, w.H, w.K)) > 0 else 0))
    desc = DESCS[name] if (agent or w.B == W.WORKLOADS[name].B) else f"{DESCS[name]} [batch {w.B}]"
    if not agent and w.ctx != W.WORKLOADS[name].ctx:
        desc += f" [context {w.ctx}]"
    if per_token:
        desc += (f" [one top-{w.K} list per query token (10% fresh per later token), the "
                 f"{w.T} lists of a request resolved as one union]")
    if L > 1:
        desc += (f" [{L} layers, each its own pool and lists: one resolve launch for all layers, "
                 f"then one decode per layer]")
    line = {
        "metric": METRIC, "value": round(steps_per_s, 2), "unit": "decode steps/s",
        "n_gpus": ws, "steps": steps, "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "fp8 rows, bf16 MMA",
        "data": "synthetic",
        "config": run_config(desc, w, ws, L, args.in_place),
        "resolved_rows_per_s": round(rows_per_s, 1),
        "resolve_ms": round(res_ms, 5), "decode_ms": round(dec_ms, 5),
        "kernel_times": ("ms_per_step: each timed step from before the resolve to after the "
                         "decode, nothing between the kernels; resolve_ms and decode_ms: a second "
                         "pass over the same steps with an event between the kernels, which keeps "
                         "the decode from launching while the resolve runs (so they add up to "
                         "more than ms_per_step)"),
        "counts_per_step": {"resident": float(per_step_counts[0]), "hot": float(per_step_counts[1]),
                            "miss": float(per_step_counts[2])},
        **({"per_token": {"entries_per_step": w.B * w.T * w.K, "distinct_rows_per_step": pt[0],
                          "distinct_misses_per_step": pt[1]}} if per_token else {}),
        "roofline": roofline,
        "kernels": {k: {kk: (round(vv, 4) if isinstance(vv, float) else vv) for kk, vv in v.items()}
                    for k, v in kernels.items()},
        "gpu_launches": launches * steps,
        "clocks": clk.summary(), "wall_s": round(wall, 3),
    }
    if r_link > 0:
        ach = r_link / (res_ms * 1e-3) / 1e9
        line["host_link"] = {"miss_bytes_per_step": r_link, "achieved": round(ach, 1),
                             "peak": round(link_peak, 1), "unit": "GB/s",
                             "frac": round(ach / link_peak, 4),
                             "peak_source": "measured live: pinned 256 MiB host-to-device copy"}
    if agent:
        per_turn = []
        for t in range(w.turns):
            a, b = t * w.steps_per_turn, min(steps, (t + 1) * w.steps_per_turn)
            if a < b:
                per_turn.append(round(sum(t_step[a:b]), 3))
        line["per_turn_ms"] = per_turn
    if with_e2e and not agent and L == 1:
        line["e2e"] = run_e2e(args, gw, qs, stream, w)
    if group is not None:
        hs.hs_layer_group_destroy(group)
    for x in gws:
        x.pool.close()
    torch.cuda.synchronize()
    return line, w


# Configurations measured after the headline in the default run (one object
# per configuration in the same JSON line); the agent mix runs all its steps.
PER_CONFIG = ["tiny", "hybrid", "noresident", "agent"]
# the headline workload again with its rows gathered by the resolve
PER_CONFIG_VARIANTS = {"resident_gathered": ("resident", {"in_place": False})}
PER_CONFIG_KEYS = ("value", "unit", "steps", "ms_per_step", "resolved_rows_per_s", "resolve_ms",
                   "decode_ms", "counts_per_step", "roofline", "kernels", "host_link", "clocks",
                   "per_turn_ms", "dtype")


def run_gpu(args):
    import torch

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    import __graft_entry__ as g
    g.build()
    plain = args.layers <= 1 and args.in_place == DEFAULT_IN_PLACE[args.workload] \
        and not args.per_token and not args.batch and not args.ctx
    headline = args.workload == WORKLOAD and plain
    line, w = measure(args, args.workload, args.steps, with_e2e=headline or args.workload == WORKLOAD)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and args.workload == WORKLOAD \
            and args.layers <= 1:
        line["cpu_baseline"] = cpu_baseline(w, args)
    if headline and not args.no_per_config:
        per = {}
        for name in PER_CONFIG:
            n_steps = DEFAULT_STEPS[name] if name == "agent" else max(args.steps, 32)
            torch.cuda.empty_cache()
            sub_args = argparse.Namespace(**{**vars(args), "in_place": DEFAULT_IN_PLACE[name]})
            sub, wn = measure(sub_args, name, n_steps)
            entry = {k: sub[k] for k in PER_CONFIG_KEYS if k in sub}
            entry["workload"] = sub["config"]["workload"]
            entry["rows"] = sub["config"]["rows"]
            if rank == 0 and ws == 1 and not args.no_cpu_baseline:
                entry["cpu_baseline"] = cpu_baseline_config(name, wn, args)
            per[name] = entry
        for key, (name, over) in PER_CONFIG_VARIANTS.items():
            torch.cuda.empty_cache()
            sub_args = argparse.Namespace(**{**vars(args), **over})
            sub, wn = measure(sub_args, name, max(args.steps, 32))
            entry = {k: sub[k] for k in PER_CONFIG_KEYS if k in sub}
            entry["workload"] = sub["config"]["workload"]
            entry["rows"] = sub["config"]["rows"]
            per[key] = entry
        line["per_config"] = per
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_transitions(args):
    """Residency transitions on the resident workload's shape: every request
    fully resident with a host block reserved per page; one active-copy launch
    copies every finished page to host memory (timed), then one demotion
    launch releases every request's pages before its last 32K tokens (timed).
    Prints one JSON line."""
    import numpy as np
    import torch
    import __graft_entry__ as g
    g.build()
    import tiered_sparse_mla_gb300 as hs
    import workloads as W
    w = W.WORKLOADS[args.workload if args.workload != "agent" else WORKLOAD]
    if args.batch:
        w = w.scaled(B=args.batch)
    P, hb = w.pages, w.hot_rows // 64
    pool = hs.Pool(dtype=hs.HS_FP8_E4M3_ROWSCALE if w.dtype == "fp8" else hs.HS_BF16,
                   n_gpu_blocks=w.B * (P + hb), n_host_blocks=w.B * P, max_requests=w.B,
                   max_ctx=w.ctx, max_topk=w.K, hot_rows=w.hot_rows)
    page_gpu = np.arange(w.B * P, dtype=np.int32).reshape(w.B, P)
    for r in range(w.B):
        pool.request_init(r, w.ctx)
        pool.page_map_range(r, 0, page_gpu[r], np.full(P, -1, np.int32))
        pool.hot_lease(r, w.B * P + r * hb + np.arange(hb))
    W.fill_rows(w.dtype, pool.gpu_rows(), pool.gpu_scales(), W.row_seed(w, "gpu"))
    reqs = np.repeat(np.arange(w.B), P - 1).astype(np.int32)
    pages = np.tile(np.arange(P - 1), w.B).astype(np.int32)
    t_req = torch.from_numpy(reqs).cuda()
    t_pg = torch.from_numpy(pages).cuda()
    t_hb = torch.from_numpy(reqs * P + pages).cuda()
    keep = torch.full((w.B,), 32768, dtype=torch.int32, device="cuda")
    rq = torch.arange(w.B, dtype=torch.int32, device="cuda")
    freed = torch.empty((w.B, P), dtype=torch.int32, device="cuda")
    nfreed = torch.empty(w.B, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    with torch.cuda.stream(stream):
        hs.hs_active_copy(pool.handle, t_req[:w.B], t_pg[:w.B], t_hb[:w.B], stream)  # warm-up
        stream.synchronize()
        ev[0].record(stream)
        hs.hs_active_copy(pool.handle, t_req, t_pg, t_hb, stream)
        ev[1].record(stream)
        hs.hs_demote_cold_pages(pool.handle, rq, keep, freed, nfreed, stream)
        ev[2].record(stream)
    torch.cuda.synchronize()
    assert pool.get_error() == 0
    copy_ms, demote_ms = ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2])
    n_pages = len(reqs)
    bytes_ = n_pages * 64 * (w.row_bytes + (4 if w.dtype == "fp8" else 0))
    gbs = bytes_ / (copy_ms * 1e-3) / 1e9
    peak = _link_peak_gbs(to_host=True)
    line = {"metric": "residency transitions: active copy GB/s, demotion time", "impl": "gb300",
            "value": round(gbs, 1), "unit": "GB/s device-to-host (active copy)",
            "higher_is_better": True, "n_gpus": 1, "data": "synthetic",
            "config": {"workload": f"{DESCS.get(w.name, w.name)} [batch {w.B}]",
                       "pages_copied": n_pages, "bytes_copied": bytes_,
                       "demotion": "every request keeps its last 32768 tokens"},
            "active_copy_ms": round(copy_ms, 3), "demote_ms": round(demote_ms, 4),
            "pages_freed": int(nfreed.sum().item()),
            "roofline": {"bound": "host-link", "achieved": round(gbs, 1), "peak": round(peak, 1),
                         "unit": "GB/s", "frac": round(gbs / peak, 4),
                         "peak_source": "measured live: pinned 256 MiB device-to-host copy"},
            "gpu_launches": 2}
    print(json.dumps(line), flush=True)
    pool.close()


def run_e2e(args, gw, qs, stream, w, check=False):
    """Same step through the C ABI, inputs copied from pinned host memory and the
    result (out, lse) read back to host memory inside the timed region.

    Each step is one CUDA-graph launch with three branches: the step's two
    library calls (resolve, decode) on its input buffer; the upload of the
    next step's top-K lists and q from pinned host memory into the other
    buffer; and the download of the previous step's out and lse from that
    buffer into pinned host memory. The copies overlap the compute in both
    directions, every step still moves its own inputs and result, and the host
    issues one launch per step: issued from Python one by one, the four copies,
    the two calls and the events that order them cost about as much host time
    as the GPU spends on the step, and the loop ran at the host's pace. The
    graphs are captured once per position in the cycle of inputs (each names
    its buffers and pinned host arrays) and replayed; the calls are capturable
    (the launch shapes depend only on the sizes, and the LRU clock advances in
    device memory). The timed region starts before the first step's upload and
    ends when the last step's result is in host memory. check: afterwards, the
    last step's downloaded out and lse are compared bit for bit with eager
    calls on that step's inputs (a resident workload, whose LRU state does not
    change between steps), and the result is added as "check"."""
    import math
    import torch
    # a fixed count, whatever the timed region's: with a few steps the first
    # ones (launch pipeline filling, copy engines starting) dominate
    n = 200
    nt, nq = w.steps, len(qs)
    topk_h = [gw.topk[s].cpu().pin_memory() for s in range(nt)]
    q_h = [q.cpu().pin_memory() for q in qs]
    out_h = [torch.empty(gw.out.shape, dtype=gw.out.dtype).pin_memory() for _ in range(2)]
    lse_h = [torch.empty(gw.lse.shape, dtype=gw.lse.dtype).pin_memory() for _ in range(2)]
    t_d = [torch.empty_like(gw.topk[0]) for _ in range(2)]
    q_d = [torch.empty_like(qs[0]) for _ in range(2)]
    out_d = [torch.empty_like(gw.out) for _ in range(2)]
    lse_d = [torch.empty_like(gw.lse) for _ in range(2)]
    h2d = topk_h[0].numel() * 4 + q_h[0].numel() * 2
    d2h = out_h[0].numel() * 2 + lse_h[0].numel() * 4
    cycle = math.lcm(nt, nq, 2)
    up_s, dn_s, cap = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    graphs = []
    for s in range(cycle):
        i, j = s % 2, (s + 1) % 2  # this step's buffer; the next step's and the previous one's
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            main = torch.cuda.current_stream()
            up_s.wait_stream(main)
            dn_s.wait_stream(main)
            with torch.cuda.stream(up_s):
                t_d[j].copy_(topk_h[(s + 1) % nt], non_blocking=True)
                q_d[j].copy_(q_h[(s + 1) % nq], non_blocking=True)
            with torch.cuda.stream(dn_s):
                out_h[j].copy_(out_d[j], non_blocking=True)
                lse_h[j].copy_(lse_d[j], non_blocking=True)
            gw.pool.resolve_topk(gw.req_ids, t_d[i], gw.resolved, gw.gathered, gw.gscale,
                                 gw.counts, main)
            gw.pool.sparse_mla_decode(q_d[i], gw.gathered, gw.gscale, gw.resolved, t_d[i],
                                      gw.req_ids, w.sm_scale, out_d[i], lse_d[i], gw.workspace,
                                      main)
            main.wait_stream(up_s)
            main.wait_stream(dn_s)
        graphs.append(g)
    torch.cuda.synchronize()

    def run(nsteps):
        # the first step's inputs, one launch per step, the last step's result
        t_d[0].copy_(topk_h[0], non_blocking=True)
        q_d[0].copy_(q_h[0], non_blocking=True)
        for s in range(nsteps):
            graphs[s % cycle].replay()
        k = (nsteps - 1) % 2
        out_h[k].copy_(out_d[k], non_blocking=True)
        lse_h[k].copy_(lse_d[k], non_blocking=True)

    with torch.cuda.stream(stream):
        run(10)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        run(n)
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    ws, _, _ = _dist()
    extra = {}
    if check:
        last, k = n - 1, (n - 1) % 2
        with torch.cuda.stream(stream):
            t_e, q_e = topk_h[last % nt].cuda(), q_h[last % nq].cuda()
            gw.pool.resolve_topk(gw.req_ids, t_e, gw.resolved, gw.gathered, gw.gscale, gw.counts,
                                 stream)
            gw.pool.sparse_mla_decode(q_e, gw.gathered, gw.gscale, gw.resolved, t_e, gw.req_ids,
                                      w.sm_scale, gw.out, gw.lse, gw.workspace, stream)
        torch.cuda.synchronize()
        extra["check"] = {
            "out_equal": bool(torch.equal(out_h[k].view(torch.int16), gw.out.cpu().view(torch.int16))),
            "lse_equal": bool(torch.equal(lse_h[k].view(torch.int32), gw.lse.cpu().view(torch.int32)))}
    return {**extra, "value": round(ws / (ms * 1e-3), 2), "unit": "decode steps/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "note": ("pinned host inputs (top-K lists, q) and outputs (out, lse); each step one "
                     "CUDA-graph launch holding the step's resolve and decode calls, the upload "
                     "of the next step's inputs and the download of the previous step's result "
                     "as parallel branches (double buffers); L2 not flushed")}


# ------------------------------------------------------------------ CPU oracle
class OracleSampler:
    """The oracle, as it stands, on a bounded sample of the workload: a
    sub-batch of `n_req` requests of the same shape (same context, top-K,
    heads, own seeded lists and rows, generated on the host). Each step
    resolves the whole sub-batch and attends `n_rows` query rows; the time is
    extrapolated to the full batch (requests are independent and identical
    in shape)."""

    def __init__(self, w_full, n_req, threads):
        import numpy as np
        import torch
        import oracle
        import workloads as W
        oracle.build()
        self.np, self.torch, self.oracle, self.W = np, torch, oracle, W
        self.full = w_full
        self.w = w = w_full.scaled(B=n_req)
        self.threads = threads
        lay = W.layout(w)
        pool = torch.empty((lay.n_gpu_blocks * 64, w.row_bytes), dtype=torch.uint8)
        W.fill_rows(w.dtype, pool, None, W.row_seed(w, "gpu"))
        self.ot = oracle.OracleTiers(
            page_gpu=lay.page_gpu, page_host=lay.page_host, hot_blocks=lay.hot_blocks,
            ctx_len=np.full(w.B, w.ctx, np.int32), pool_rows=pool.numpy(), pool_scales=None,
            host_rows=np.zeros((64, w.row_bytes), np.uint8), host_scales=None,
            hot_rows=w.hot_rows, max_ctx=w.ctx)
        self.lists = list(W.topk_lists(w))

    def step(self, s, n_rows):
        np, torch, w = self.np, self.torch, self.w
        topk = self.lists[s % len(self.lists)]
        q_bits = self.W.make_q(w, s).view(torch.int16).numpy().view(np.uint16)
        t0 = time.perf_counter()
        res, gat, _, _, err = self.ot.resolve(np.arange(w.B), topk, nthreads=self.threads)
        t1 = time.perf_counter()
        n = w.B * w.T * w.H
        idx = np.arange(min(n_rows, n))
        sel = np.stack([idx // (w.T * w.H), (idx // w.H) % w.T, idx % w.H], 1).astype(np.int32)
        self.oracle.sparse_mla_decode(q_bits, gat, None, res, topk, np.full(w.B, w.ctx, np.int32),
                                      w.sm_scale, sel=sel, nthreads=self.threads)
        t2 = time.perf_counter()
        full = self.full
        extrap = (t1 - t0) * full.B / w.B + (t2 - t1) * (full.B * full.T * full.H) / len(idx)
        return extrap, t2 - t0, t1 - t0, (t2 - t1) / len(idx)


def cpu_baseline(w, args):
    import oracle
    oracle.build()
    threads = oracle.max_threads()
    n_req = 4
    smp = OracleSampler(w, n_req, threads)
    per, spent, s = [], 0.0, 0
    while s < len(smp.lists) and (spent < args.cpu_seconds or s < 1):
        e, m, _, _ = smp.step(s, n_req * w.T * w.H)
        per.append(e)
        spent += m
        s += 1
    v = len(per) / sum(per)
    # the same oracle on one core: one step of a one-request sub-batch, its
    # resolve and the attention of 32 query rows, extrapolated the same way
    one = OracleSampler(w, 1, 1)
    e1, m1, _, _ = one.step(0, 32)
    return {"value": round(v, 5), "unit": "decode steps/s", "cores": threads, "kind": "oracle",
            "sample": (f"{s} decode steps of a {n_req}-request sub-batch of the same workload "
                       f"(resolve and attention of all {n_req * w.T * w.H} query rows), "
                       f"extrapolated to {w.B} requests; {spent:.1f} s of CPU work"),
            "value_1core": round(1.0 / e1, 6),
            "sample_1core": (f"1 core: one step of a 1-request sub-batch (resolve, attention of 32 "
                             f"query rows) extrapolated to {w.B} requests; {m1:.1f} s of CPU work")}


def cpu_baseline_config(name, w, args, budget_s=4.0):
    """The oracle as it stands on a bounded sample of configuration `name`:
    one request of the configuration's shape with its own seeded lists
    (pool rows N(0,1); host rows zero: the resolve copies them all the same),
    whose resolve is timed over the first steps and whose attention is timed
    on a sample of query rows, both extrapolated to the full batch. For the
    agent mix the request is a hybrid-shaped one at the mix's first-turn
    context (every step's attention has the same shape: FP8, 4 query
    tokens, 128 heads, top-2048)."""
    import numpy as np
    import torch
    import oracle
    import workloads as W
    oracle.build()
    threads = oracle.max_threads()
    B = w.B
    if name == "agent":
        w1 = W.WORKLOADS["hybrid"].scaled(B=1, ctx=w.first, index=w.index if hasattr(w, "index")
                                          else 4)
        label = (f"a hybrid-shaped request (FP8, 4 tokens, 128 heads, top-2048) at the mix's "
                 f"first-turn context {w.first}")
    else:
        w1 = w.scaled(B=1)
        label = f"one request of the same shape ({w.ctx}-token context)"
    lay = W.layout(w1)
    rows = torch.empty((lay.n_gpu_blocks * 64, w1.row_bytes), dtype=torch.uint8)
    scales = torch.empty(lay.n_gpu_blocks * 64, dtype=torch.float32) if w1.dtype == "fp8" else None
    W.fill_rows(w1.dtype, rows, scales, W.row_seed(w1, "gpu"))
    nh = max(lay.n_host_blocks, 1) * 64
    host = np.zeros((nh, w1.row_bytes), np.uint8)
    hsc = np.zeros(nh, np.float32) if w1.dtype == "fp8" else None
    ot = oracle.OracleTiers(
        page_gpu=lay.page_gpu, page_host=lay.page_host, hot_blocks=lay.hot_blocks,
        ctx_len=np.full(1, w1.ctx, np.int32), pool_rows=rows.numpy(),
        pool_scales=None if scales is None else scales.numpy(), host_rows=host, host_scales=hsc,
        hot_rows=w1.hot_rows, max_ctx=w1.ctx)
    t_res, n_res, spent = 0.0, 0, 0.0
    res = gat = gsc = topk = None
    for s_, topk in enumerate(W.topk_lists(w1)):
        t0 = time.perf_counter()
        res, gat, gsc, _, _ = ot.resolve(np.arange(1), topk, nthreads=threads)
        dt = time.perf_counter() - t0
        t_res, n_res, spent = t_res + dt, n_res + 1, spent + dt
        if spent > budget_s / 4 or s_ >= 7:
            break
    q = W.make_q(w1, 0).view(torch.int16).numpy().view(np.uint16)
    n_all = w1.T * w1.H
    n_rows = 16
    t0 = time.perf_counter()
    while True:
        idx = np.arange(min(n_rows, n_all))
        sel = np.stack([np.zeros_like(idx), idx // w1.H, idx % w1.H], 1).astype(np.int32)
        t0 = time.perf_counter()
        oracle.sparse_mla_decode(q, gat, gsc, res, topk, np.full(1, w1.ctx, np.int32), w1.sm_scale,
                                 sel=sel, nthreads=threads)
        t_att = time.perf_counter() - t0
        if t_att > budget_s / 2 or n_rows >= n_all:
            break
        n_rows = min(n_all, n_rows * 4)
    per_req = t_res / n_res
    per_row = t_att / len(idx)
    step_s = B * per_req + B * w.T * w.H * per_row
    return {"value": round(1.0 / step_s, 6), "unit": "decode steps/s", "cores": threads,
            "kind": "oracle",
            "sample": (f"{label}: resolve of {n_res} steps and attention of {len(idx)} of its "
                       f"{n_all} query rows, extrapolated to {B} requests x {w.T * w.H} query "
                       f"rows per step; {spent + t_att:.1f} s of CPU work")}


def run_reference(args):
    """--impl reference: the CPU oracle as it stands, same workload and metric;
    each step a bounded sample (one request resolved, some query rows attended)
    sized so that the whole run ends within a few minutes."""
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import oracle
    import workloads as W
    oracle.build()
    w = W.WORKLOADS[WORKLOAD]
    threads = oracle.max_threads()
    smp = OracleSampler(w, 1, threads)
    budget = 150.0 / (args.steps + args.warmup)
    _, _, t_res, t_row = smp.step(0, 8)
    n_rows = int(max(1, min(w.T * w.H, (budget - t_res) / max(t_row, 1e-9))))
    times, walls = [], []
    for s in range(args.warmup + args.steps):
        e, m, _, _ = smp.step(s, n_rows)
        if s >= args.warmup:
            times.append(e)
            walls.append(m)
    ms = 1e3 * sum(times) / len(times)
    wall_ms = 1e3 * sum(walls) / len(walls)
    v = 1e3 / ms
    sample = (f"each step: resolve of 1 of {w.B} requests and attention of {n_rows} of its "
              f"{w.T * w.H} query rows, extrapolated to the full {w.B}-request step")
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 5), "unit": "decode steps/s",
            "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(wall_ms, 3),
            "ms_per_step_extrapolated": round(ms, 3),
            "timing": ("ms_per_step is the wall time of the sampled work actually run per step; "
                       "value is the full step's rate extrapolated from it (ms_per_step_extrapolated)"),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": run_config(WORKLOAD_DESC, w, ws, 1, DEFAULT_IN_PLACE[WORKLOAD]),
            "cpu_baseline": {"value": round(v, 5), "unit": "decode steps/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 5), "unit": "decode steps/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0,
                    help="timed steps (default: 2000 for the resident workload)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="CPU work spent on the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the other configurations measured after the headline")
    ap.add_argument("--batch", type=int, default=0,
                    help="requests per step (default: the workload's; smaller only for profiling)")
    ap.add_argument("--transitions", action="store_true",
                    help="time the active copy and the demotion kernels (one JSON line)")
    ap.add_argument("--layers", type=int, default=1,
                    help="L layers (own pools and lists): one multi-layer resolve launch per step")
    ap.add_argument("--per-token", action="store_true",
                    help="one top-K list per query token: union resolve + per-token decode")
    ap.add_argument("--in-place", action="store_true",
                    help="attention reads rows from the pool by id; no gathered buffer "
                         "(the resident workload's default)")
    ap.add_argument("--gathered", action="store_true",
                    help="the resolve gathers the rows into a buffer that attention reads "
                         "(the other workloads' default)")
    ap.add_argument("--ctx", type=int, default=0,
                    help="override the context length (profiling captures only)")
    ap.add_argument("--workload", default=WORKLOAD, choices=sorted(DESCS),
                    help="resident (default, the headline) or another configuration")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    args.steps = args.steps or DEFAULT_STEPS[args.workload]
    if args.in_place and args.gathered:
        ap.error("--in-place and --gathered exclude each other")
    # per-token lists (a union resolve): in place measured shorter (hybrid,
    # 5.9K against 5.3K steps/s), whatever the workload's default
    args.in_place = args.in_place or (not args.gathered and
                                      (DEFAULT_IN_PLACE[args.workload] or args.per_token))
    if args.impl == "reference":
        run_reference(args)
    elif args.transitions:
        run_transitions(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
