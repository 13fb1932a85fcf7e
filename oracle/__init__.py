"""CPU oracle for the tiered sparse-MLA decode path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package. The product
path (the CUDA library and its binding) never does.

The arithmetic lives in ``hs_oracle.c`` (plain C, float64 attention); this
module builds it with gcc and wraps it with ctypes. It shares no code with the
CUDA path: both sides only read the seeded inputs from ``workloads``.

Pins (tests marked ``not gpu``): hand-computed LRU scenarios under
``tests/golden/``, two independent formulations of the LRU rule checked
against each other, the state invariants, brute-force dense MLA attention in
float64 via ``torch`` on small inputs, closed-form special cases, and all 256
e4m3 codes against ``torch.float8_e4m3fn``. The union of per-token lists is
pinned to the single-list rule with repeats blanked; per-token attention to
the shared-list MTP decode; the residency transitions (plain numpy here) to
the workloads' tail layout, to invariants, and to the resolve serving demoted
rows with their original bytes.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hs_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

ERR_INDEX_RANGE = 1
ERR_DUPLICATE = 2
ERR_NO_HOST = 4
ERR_BAD_REQUEST = 8
ERR_CAPACITY = 16
ERR_BAD_PAGE = 64

PAGE = 64


def build(force: bool = False) -> str:
    """Compile hs_oracle.c into liboracle.so (OpenMP when gcc has it)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    os.replace(tmp, _LIB)
    return _LIB


class _State(C.Structure):
    _fields_ = [
        ("max_req", C.c_int32), ("max_pages", C.c_int32), ("max_ctx", C.c_int32),
        ("hot_rows", C.c_int32), ("row_bytes", C.c_int32), ("fp8", C.c_int32),
        ("page_gpu", C.c_void_p), ("page_host", C.c_void_p), ("hot_blocks", C.c_void_p),
        ("tag", C.c_void_p), ("stamp", C.c_void_p), ("pos_to_slot", C.c_void_p),
        ("clock", C.c_void_p), ("ctx_len", C.c_void_p),
        ("pool_rows", C.c_void_p), ("pool_scales", C.c_void_p),
        ("host_rows", C.c_void_p), ("host_scales", C.c_void_p),
    ]


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build())
        _lib.or_resolve.restype = C.c_uint32
        _lib.or_resolve.argtypes = [C.POINTER(_State), C.c_int32, C.c_void_p, C.c_void_p,
                                    C.c_int32, C.c_int32, C.c_void_p, C.c_void_p,
                                    C.c_void_p, C.c_void_p, C.c_int32]
        _lib.or_sparse_mla_decode.restype = None
        _lib.or_sparse_mla_decode.argtypes = [C.c_int32] * 5 + [C.c_void_p] * 6 + [
            C.c_double, C.c_int32, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int32]
        _lib.or_e4m3_to_double.restype = C.c_double
        _lib.or_e4m3_to_double.argtypes = [C.c_uint8]
        _lib.or_bf16_to_double.restype = C.c_double
        _lib.or_bf16_to_double.argtypes = [C.c_uint16]
        _lib.or_max_threads.restype = C.c_int32
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def _c(a, dt):
    a = np.ascontiguousarray(a, dtype=dt)
    return a


def e4m3_to_double(code: int) -> float:
    return lib().or_e4m3_to_double(code)


def bf16_to_double(bits: int) -> float:
    return lib().or_bf16_to_double(bits)


def max_threads() -> int:
    return lib().or_max_threads()


@dataclass
class OracleTiers:
    """The oracle's own copy of one pool: tables, hot-buffer LRU state and rows.

    All arrays are numpy; the oracle mutates tag/stamp/pos_to_slot/clock and the
    pool rows (miss copies) in place. host_rows/host_scales may alias the
    caller's (read-only) host arena."""

    page_gpu: np.ndarray      # int32 [max_req][max_pages]
    page_host: np.ndarray     # int32 [max_req][max_pages]
    hot_blocks: np.ndarray    # int32 [max_req][hot_rows/64]
    ctx_len: np.ndarray       # int32 [max_req]
    pool_rows: np.ndarray     # uint8 [n_gpu_rows][row_bytes]
    pool_scales: np.ndarray | None
    host_rows: np.ndarray     # uint8 [n_host_rows][row_bytes]
    host_scales: np.ndarray | None
    hot_rows: int
    max_ctx: int

    def __post_init__(self):
        self.page_gpu = _c(self.page_gpu, np.int32)
        self.page_host = _c(self.page_host, np.int32)
        self.hot_blocks = _c(self.hot_blocks, np.int32)
        self.ctx_len = _c(self.ctx_len, np.int32)
        R = self.page_gpu.shape[0]
        self.tag = np.full((R, self.hot_rows), -1, np.int32)
        self.stamp = np.full((R, self.hot_rows), -1, np.int32)
        self.pos_to_slot = np.full((R, self.max_ctx), -1, np.int32)
        self.clock = np.zeros(R, np.int32)
        self.fp8 = self.pool_scales is not None
        self.row_bytes = self.pool_rows.shape[1]

    def _state(self) -> _State:
        R, P = self.page_gpu.shape
        return _State(R, P, self.max_ctx, self.hot_rows, self.row_bytes, int(self.fp8),
                      _p(self.page_gpu), _p(self.page_host), _p(self.hot_blocks),
                      _p(self.tag), _p(self.stamp), _p(self.pos_to_slot), _p(self.clock),
                      _p(self.ctx_len), _p(self.pool_rows), _p(self.pool_scales),
                      _p(self.host_rows), _p(self.host_scales))

    # ------------------------------------------------------------ residency transitions
    def active_copy(self, reqs, pages, host_blocks) -> int:
        """Active copy ("vLLM GLM 5.3 优化：混合 HiSparse 卸载", 混合 HiSparse 的技术实现
        item 1 and 关键架构细节, 主动复制): a finished page of a resident request is
        copied to host memory while the GPU keeps serving it. For each triple
        (r, p, hb), in order: the 64 rows (and scales) of the page's GPU block
        are copied into host block hb, and the page table records hb as the
        page's host copy. A triple with r, p or hb out of range, or whose page
        has no GPU block, changes nothing and sets ERR_BAD_PAGE. Needs a
        writable host arena of the oracle's own. Returns the error bits."""
        R, P = self.page_gpu.shape
        n_hb = self.host_rows.shape[0] // PAGE
        err = 0
        for r, p, hb in zip(np.asarray(reqs).tolist(), np.asarray(pages).tolist(),
                            np.asarray(host_blocks).tolist()):
            if not (0 <= r < R and 0 <= p < P and 0 <= hb < n_hb) or self.page_gpu[r, p] < 0:
                err |= ERR_BAD_PAGE
                continue
            gb = int(self.page_gpu[r, p])
            self.host_rows[hb * PAGE:(hb + 1) * PAGE] = self.pool_rows[gb * PAGE:(gb + 1) * PAGE]
            if self.fp8:
                self.host_scales[hb * PAGE:(hb + 1) * PAGE] = self.pool_scales[gb * PAGE:(gb + 1) * PAGE]
            self.page_host[r, p] = hb
        return err

    def demote(self, reqs, keep_tail):
        """Demotion under pressure (same page, 混合 HiSparse 的技术实现 item 2; "vLLM
        Hybrid HiSparse：稀疏MLA破解长上下文显存瓶颈", 分级内存的运作机制): a request
        keeps its tail on the GPU and releases its coldest pages, read as its
        oldest: every page p with (p+1)*64 <= ctx_len - keep_tail that is
        resident and has a host copy loses its GPU block. Returns (per request
        the freed GPU blocks in ascending page order, error bits); a bad request
        id (ERR_BAD_REQUEST) or a negative tail (ERR_BAD_PAGE) frees nothing."""
        R, P = self.page_gpu.shape
        freed, err = [], 0
        for r, kt in zip(np.asarray(reqs).tolist(), np.asarray(keep_tail).tolist()):
            out = []
            if not 0 <= r < R:
                err |= ERR_BAD_REQUEST
            elif kt < 0:
                err |= ERR_BAD_PAGE
            else:
                ncold = min(max(0, (int(self.ctx_len[r]) - kt) // PAGE), P)
                for p in range(ncold):
                    if self.page_gpu[r, p] >= 0 and self.page_host[r, p] >= 0:
                        out.append(int(self.page_gpu[r, p]))
                        self.page_gpu[r, p] = -1
            freed.append(np.array(out, np.int32))
        return freed, err

    def reset_request(self, r: int):
        self.tag[r] = -1
        self.stamp[r] = -1
        self.pos_to_slot[r] = -1
        self.clock[r] = 0

    def resolve(self, req_ids, topk, formulation: int = 0, nthreads: int = 1,
                union: bool = False):
        """One decode step. Returns (resolved [B][K] int32, gathered [B][K][rb] uint8,
        gathered_scale [B][K] f32 or None, counts [B][3] int32, error bits).

        union: each list is the union of several lists sharing the request's hot
        state (per-token MTP lists, concatenated); a missing position repeated
        in it is served once and all its occurrences resolve to that row."""
        req_ids = _c(req_ids, np.int32)
        topk = _c(topk, np.int32)
        B, K = topk.shape
        resolved = np.empty((B, K), np.int32)
        gathered = np.empty((B, K, self.row_bytes), np.uint8)
        gscale = np.empty((B, K), np.float32) if self.fp8 else None
        counts = np.empty((B, 3), np.int32)
        st = self._state()
        err = lib().or_resolve(C.byref(st), B, _p(req_ids), _p(topk), K,
                               formulation | (2 if union else 0),
                               _p(resolved), _p(gathered), _p(gscale), _p(counts), nthreads)
        return resolved, gathered, gscale, counts, int(err)


def sparse_mla_decode(q_bf16_bits, gathered, gscale, resolved, topk, L_b, sm_scale,
                      sel=None, nthreads: int = 1):
    """Sparse MLA decode in float64.

    q_bf16_bits: uint16 [B][T][H][576] (bf16 bit patterns); gathered: uint8
    [B][K][rb]; gscale: f32 [B][K] for FP8, else None; resolved/topk: int32 [B][K];
    L_b: int32 [B] context length of each batch entry. sel: optional int32 [n][3]
    of (b, t, h) rows to compute. Returns (out f64 [n][512], lse f64 [n])."""
    q = _c(q_bf16_bits, np.uint16)
    B, T, H, D = q.shape
    gathered = _c(gathered, np.uint8)
    K = gathered.shape[1]
    fp8 = gscale is not None
    if fp8:
        gscale = _c(gscale, np.float32)
    resolved = _c(resolved, np.int32)
    topk = _c(topk, np.int32)
    L_b = _c(L_b, np.int32)
    if sel is not None:
        sel = _c(sel, np.int32).reshape(-1, 3)
        n = sel.shape[0]
    else:
        n = B * T * H
    out = np.empty((n, 512), np.float64)
    lse = np.empty(n, np.float64)
    lib().or_sparse_mla_decode(B, T, H, K, int(fp8), _p(q), _p(gathered), _p(gscale),
                               _p(resolved), _p(topk), _p(L_b), float(sm_scale),
                               n if sel is not None else 0, _p(sel), _p(out), _p(lse), nthreads)
    return out, lse
