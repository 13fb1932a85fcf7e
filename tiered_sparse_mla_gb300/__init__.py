"""GB300 (sm_103a) tiered sparse-MLA decode path: Python binding of ``include/hs.h``.

Thin ctypes marshalling over ``libhs.so``: every step of the path runs in the
library's CUDA kernels. PyTorch supplies device memory (tensor data pointers)
and streams only. Function names follow the C ABI (``hs_pool_create``,
``hs_resolve_topk``, ``hs_sparse_mla_decode`` ...); :class:`Pool` is a small
convenience wrapper around a pool handle.

There is no CPU fallback: importing the ops without a built library, or using
them on a device other than sm_103, raises.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libhs.so")

HS_OK, HS_ERR_INVALID_ARG, HS_ERR_CAPACITY, HS_ERR_OUT_OF_MEMORY = 0, 1, 2, 3
HS_ERR_CUDA, HS_ERR_DEVICE_DATA, HS_ERR_TIMEOUT, HS_ERR_UNSUPPORTED = 4, 5, 6, 7
HS_DEVERR_INDEX_RANGE, HS_DEVERR_DUPLICATE, HS_DEVERR_NO_HOST = 1, 2, 4
HS_DEVERR_BAD_REQUEST, HS_DEVERR_CAPACITY, HS_DEVERR_TIMEOUT = 8, 16, 32
HS_DEVERR_BAD_PAGE = 64
HS_BF16, HS_FP8_E4M3_ROWSCALE = 0, 1

EXPORTED = [
    "hs_pool_create", "hs_pool_destroy", "hs_pool_get_config", "hs_pool_get_tables",
    "hs_request_init", "hs_request_set_ctx_len", "hs_set_ctx_len", "hs_page_map",
    "hs_page_map_range", "hs_hot_lease", "hs_hot_release", "hs_gpu_rows", "hs_host_rows",
    "hs_gpu_scales", "hs_host_scales", "hs_host_rows_device", "hs_host_scales_device",
    "hs_pool_snapshot", "hs_pool_restore",
    "hs_pool_get_error", "hs_resolve_topk", "hs_sparse_mla_decode",
    "hs_decode_workspace_bytes", "hs_status_string", "hs_sparse_mla_decode_static_ws",
    "hs_pool_check_bounded_wait", "hs_resolve_topk_union", "hs_sparse_mla_decode_per_token",
    "hs_layer_group_create", "hs_layer_group_destroy", "hs_resolve_topk_layers",
    "hs_active_copy", "hs_demote_cold_pages",
]
HS_STATIC_DECODE_WS_BYTES = 24 << 20


class HsError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} (status {status})")


class hs_pool_config(C.Structure):
    _fields_ = [("nope_dim", C.c_int32), ("rope_dim", C.c_int32), ("page_size", C.c_int32),
                ("dtype", C.c_int32), ("n_gpu_blocks", C.c_int64), ("n_host_blocks", C.c_int64),
                ("max_requests", C.c_int32), ("max_ctx", C.c_int32), ("hot_rows", C.c_int32),
                ("max_topk", C.c_int32)]


class hs_pool_tables(C.Structure):
    _fields_ = [("page_table", C.c_void_p), ("hot_blocks", C.c_void_p), ("slot_tag", C.c_void_p),
                ("slot_stamp", C.c_void_p), ("lru_order", C.c_void_p),
                ("pos_to_slot", C.c_void_p), ("clock", C.c_void_p), ("ctx_len", C.c_void_p),
                ("max_pages", C.c_int32), ("row_bytes", C.c_int32)]


_lib = None


def load() -> C.CDLL:
    """Loads libhs.so. Raises if it was not built (no fallback exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            "tiered_sparse_mla_gb300: libhs.so is not built; run "
            "`python -c 'import __graft_entry__ as g; g.build()'` first")
    lib = C.CDLL(LIB_PATH)
    vp, i32, i64, sz = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t
    sig = {
        "hs_pool_create": ([C.POINTER(hs_pool_config), vp, C.POINTER(vp)], i32),
        "hs_pool_destroy": ([vp], i32),
        "hs_pool_get_config": ([vp, C.POINTER(hs_pool_config)], i32),
        "hs_pool_get_tables": ([vp, C.POINTER(hs_pool_tables)], i32),
        "hs_request_init": ([vp, i32, i32], i32),
        "hs_request_set_ctx_len": ([vp, i32, i32], i32),
        "hs_set_ctx_len": ([vp, vp, i32, vp], i32),
        "hs_page_map": ([vp, i32, i32, i64, i64], i32),
        "hs_page_map_range": ([vp, i32, i32, i32, vp, vp], i32),
        "hs_hot_lease": ([vp, i32, vp, i32], i32),
        "hs_hot_release": ([vp, i32], i32),
        "hs_gpu_rows": ([vp], vp), "hs_host_rows": ([vp], vp),
        "hs_gpu_scales": ([vp], vp), "hs_host_scales": ([vp], vp),
        "hs_host_rows_device": ([vp], vp), "hs_host_scales_device": ([vp], vp),
        "hs_pool_snapshot": ([vp, vp, sz, C.POINTER(sz)], i32),
        "hs_pool_restore": ([vp, vp, sz], i32),
        "hs_pool_get_error": ([vp, C.POINTER(C.c_uint32)], i32),
        "hs_resolve_topk": ([vp, i32, vp, vp, i32, vp, vp, vp, vp, vp], i32),
        "hs_sparse_mla_decode": ([vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, C.c_float,
                                  vp, vp, vp, sz, vp], i32),
        "hs_decode_workspace_bytes": ([i32, i32, i32, i32], sz),
        "hs_sparse_mla_decode_static_ws": ([vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp,
                                            C.c_float, vp, vp, vp], i32),
        "hs_status_string": ([i32], C.c_char_p),
        "hs_resolve_topk_union": ([vp, i32, vp, vp, i32, vp, vp, vp, vp, vp], i32),
        "hs_layer_group_create": ([C.POINTER(vp), i32, C.POINTER(vp)], i32),
        "hs_layer_group_destroy": ([vp], i32),
        "hs_resolve_topk_layers": ([vp, i32, vp, vp, i32, vp, vp, vp, vp, vp], i32),
        "hs_active_copy": ([vp, i32, vp, vp, vp, vp], i32),
        "hs_demote_cold_pages": ([vp, i32, vp, vp, vp, vp, vp], i32),
        "hs_sparse_mla_decode_per_token": ([vp, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp,
                                            C.c_float, vp, vp, vp, sz, vp], i32),
        "hs_pool_check_bounded_wait": ([vp, C.c_uint32, vp], i32),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().hs_status_string(status).decode()


def _check(fn: str, st: int):
    if st != HS_OK:
        raise HsError(fn, st)


def _ptr(t) -> int | None:
    """Device pointer of a CUDA tensor (None passes NULL)."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream) -> int | None:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


class _CudaArray:
    def __init__(self, ptr: int, shape, typestr: str):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr,
                                         "data": (ptr, False), "version": 3, "strides": None}


def _device_view(ptr: int, shape, typestr: str):
    import torch
    return torch.as_tensor(_CudaArray(ptr, shape, typestr), device="cuda")


# ------------------------------------------------------------- C ABI functions
def hs_pool_create(cfg: hs_pool_config, stream=None) -> int:
    h = C.c_void_p()
    _check("hs_pool_create", load().hs_pool_create(C.byref(cfg), _stream(stream), C.byref(h)))
    return h.value


def hs_pool_destroy(pool: int):
    _check("hs_pool_destroy", load().hs_pool_destroy(pool))


def hs_resolve_topk(pool: int, req_ids, topk_idx, resolved, gathered, gathered_scale, counts,
                    stream=None):
    """One decode step's resolve (see hs.h). Tensors: req_ids int32 [B], topk_idx
    int32 [B][K], resolved int32 [B][K], gathered uint8 [B][K][row_bytes],
    gathered_scale float32 [B][K] or None, counts int32 [B][3]."""
    B, K = topk_idx.shape
    _check("hs_resolve_topk", load().hs_resolve_topk(
        pool, B, _ptr(req_ids), _ptr(topk_idx), K, _ptr(resolved), _ptr(gathered),
        _ptr(gathered_scale), _ptr(counts), _stream(stream)))


def hs_resolve_topk_union(pool: int, req_ids, topk_idx, resolved, gathered, gathered_scale,
                          counts, stream=None):
    """Resolve of several lists per request as their union (see hs.h). topk_idx
    int32 [B][T*K] (or [B][T][K]): each request's tokens' lists, concatenated;
    other tensors as hs_resolve_topk with K replaced by T*K."""
    B = topk_idx.shape[0]
    K = topk_idx.numel() // max(B, 1)
    _check("hs_resolve_topk_union", load().hs_resolve_topk_union(
        pool, B, _ptr(req_ids), _ptr(topk_idx), K, _ptr(resolved), _ptr(gathered),
        _ptr(gathered_scale), _ptr(counts), _stream(stream)))


def hs_layer_group_create(pools) -> int:
    """Group of pools (one per layer) for hs_resolve_topk_layers; returns a handle."""
    arr = (C.c_void_p * len(pools))(*[p.handle if hasattr(p, "handle") else p for p in pools])
    h = C.c_void_p()
    _check("hs_layer_group_create", load().hs_layer_group_create(arr, len(pools), C.byref(h)))
    return h.value


def hs_layer_group_destroy(group: int):
    _check("hs_layer_group_destroy", load().hs_layer_group_destroy(group))


def hs_resolve_topk_layers(group: int, req_ids, topk_idx, resolved, gathered, gathered_scale,
                           counts, stream=None):
    """All layers' resolve in one launch (see hs.h). topk_idx / resolved int32
    [L][B][K]; gathered [L][B][K][row_bytes] or None; gathered_scale [L][B][K]
    or None; counts int32 [L][B][3]."""
    _, B, K = topk_idx.shape
    _check("hs_resolve_topk_layers", load().hs_resolve_topk_layers(
        group, B, _ptr(req_ids), _ptr(topk_idx), K, _ptr(resolved), _ptr(gathered),
        _ptr(gathered_scale), _ptr(counts), _stream(stream)))


def hs_active_copy(pool: int, req, page, host_block, stream=None):
    """Active copy of pages to host blocks (see hs.h); int32 device tensors [n]."""
    _check("hs_active_copy", load().hs_active_copy(
        pool, req.numel(), _ptr(req), _ptr(page), _ptr(host_block), _stream(stream)))


def hs_demote_cold_pages(pool: int, req, keep_tail, freed, n_freed, stream=None):
    """Demotion of each request's pages before its tail (see hs.h). req, keep_tail,
    n_freed int32 [n]; freed int32 [n][max_pages]."""
    _check("hs_demote_cold_pages", load().hs_demote_cold_pages(
        pool, req.numel(), _ptr(req), _ptr(keep_tail), _ptr(freed), _ptr(n_freed),
        _stream(stream)))


def hs_decode_workspace_bytes(B: int, T: int, H: int, K: int) -> int:
    return load().hs_decode_workspace_bytes(B, T, H, K)


def hs_sparse_mla_decode(pool: int, q, gathered, gathered_scale, resolved, topk_idx, req_ids,
                         sm_scale: float, out, lse, workspace=None, stream=None):
    """Sparse MLA decode (see hs.h). q bf16 [B][T][H][576], out bf16 [B][T][H][512],
    lse float32 [B][T][H]; workspace uint8 tensor of hs_decode_workspace_bytes."""
    B, T, H, _ = q.shape
    K = topk_idx.shape[1]
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("hs_sparse_mla_decode", load().hs_sparse_mla_decode(
        pool, B, T, H, K, _ptr(q), _ptr(gathered), _ptr(gathered_scale), _ptr(resolved),
        _ptr(topk_idx), _ptr(req_ids), float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace),
        ws, _stream(stream)))


def hs_sparse_mla_decode_per_token(pool: int, q, gathered, gathered_scale, resolved, topk_idx,
                                   req_ids, sm_scale: float, out, lse, workspace=None,
                                   stream=None):
    """Decode with one list per query token (see hs.h). q bf16 [B][T][H][576];
    topk_idx / resolved int32 [B][T][K]; gathered [B][T][K][row_bytes] or None;
    workspace of hs_decode_workspace_bytes(B*T, 1, H, K) bytes."""
    B, T, H, _ = q.shape
    K = topk_idx.shape[-1]
    ws = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("hs_sparse_mla_decode_per_token", load().hs_sparse_mla_decode_per_token(
        pool, B, T, H, K, _ptr(q), _ptr(gathered), _ptr(gathered_scale), _ptr(resolved),
        _ptr(topk_idx), _ptr(req_ids), float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace),
        ws, _stream(stream)))


def hs_sparse_mla_decode_static_ws(pool: int, q, gathered, gathered_scale, resolved, topk_idx,
                                   req_ids, sm_scale: float, out, lse, stream=None):
    """hs_sparse_mla_decode without a workspace argument, for callers that cannot
    allocate device memory: the split-KV partials use a fixed array inside the
    library (HS_STATIC_DECODE_WS_BYTES; see hs.h for the sharing rules)."""
    B, T, H, _ = q.shape
    K = topk_idx.shape[1]
    _check("hs_sparse_mla_decode_static_ws", load().hs_sparse_mla_decode_static_ws(
        pool, B, T, H, K, _ptr(q), _ptr(gathered), _ptr(gathered_scale), _ptr(resolved),
        _ptr(topk_idx), _ptr(req_ids), float(sm_scale), _ptr(out), _ptr(lse), _stream(stream)))


# ------------------------------------------------------------- convenience
class Pool:
    """Owns one hs_pool handle; methods map one-to-one onto the C ABI."""

    def __init__(self, *, dtype: int, n_gpu_blocks: int, n_host_blocks: int, max_requests: int,
                 max_ctx: int, max_topk: int, hot_rows: int = 0, stream=None):
        self.cfg = hs_pool_config(512, 64, 64, dtype, n_gpu_blocks, n_host_blocks, max_requests,
                                  max_ctx, hot_rows, max_topk)
        self.handle = hs_pool_create(self.cfg, stream)
        got = hs_pool_config()
        _check("hs_pool_get_config", load().hs_pool_get_config(self.handle, C.byref(got)))
        self.cfg = got
        t = hs_pool_tables()
        _check("hs_pool_get_tables", load().hs_pool_get_tables(self.handle, C.byref(t)))
        self._tables = t
        self.row_bytes = t.row_bytes
        self.max_pages = t.max_pages
        self.fp8 = dtype == HS_FP8_E4M3_ROWSCALE

    def close(self):
        if self.handle:
            hs_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # bookkeeping
    def request_init(self, req: int, ctx_len: int):
        _check("hs_request_init", load().hs_request_init(self.handle, req, ctx_len))

    def set_ctx_len(self, req: int, ctx_len: int):
        _check("hs_request_set_ctx_len", load().hs_request_set_ctx_len(self.handle, req, ctx_len))

    def set_ctx_lens(self, d_ctx_len, stream=None):
        """Context lengths of requests 0..n-1 from an int32 CUDA tensor."""
        _check("hs_set_ctx_len", load().hs_set_ctx_len(self.handle, _ptr(d_ctx_len),
                                                       d_ctx_len.numel(), _stream(stream)))

    def page_map(self, req: int, page: int, gpu_block: int, host_block: int):
        _check("hs_page_map", load().hs_page_map(self.handle, req, page, gpu_block, host_block))

    def page_map_range(self, req: int, first: int, gpu_blocks, host_blocks):
        g = np.ascontiguousarray(gpu_blocks, dtype=np.int32)
        h = np.ascontiguousarray(host_blocks, dtype=np.int32)
        _check("hs_page_map_range", load().hs_page_map_range(
            self.handle, req, first, len(g), g.ctypes.data, h.ctypes.data))

    def hot_lease(self, req: int, blocks):
        b = np.ascontiguousarray(blocks, dtype=np.int64)
        _check("hs_hot_lease", load().hs_hot_lease(self.handle, req, b.ctypes.data, len(b)))

    def hot_release(self, req: int):
        _check("hs_hot_release", load().hs_hot_release(self.handle, req))

    def check_bounded_wait(self, limit_us: int, stream=None):
        """Runs a device wait that nothing completes; it must time out (see hs.h)."""
        _check("hs_pool_check_bounded_wait",
               load().hs_pool_check_bounded_wait(self.handle, limit_us, _stream(stream)))

    def get_error(self) -> int:
        v = C.c_uint32()
        _check("hs_pool_get_error", load().hs_pool_get_error(self.handle, C.byref(v)))
        return v.value

    def snapshot(self) -> bytearray:
        n = C.c_size_t()
        _check("hs_pool_snapshot", load().hs_pool_snapshot(self.handle, None, 0, C.byref(n)))
        buf = bytearray(n.value)
        cbuf = (C.c_char * n.value).from_buffer(buf)
        _check("hs_pool_snapshot", load().hs_pool_snapshot(self.handle, C.addressof(cbuf),
                                                           n.value, C.byref(n)))
        return buf

    def restore(self, buf: bytearray):
        cbuf = (C.c_char * len(buf)).from_buffer(buf)
        _check("hs_pool_restore", load().hs_pool_restore(self.handle, C.addressof(cbuf), len(buf)))

    # storage views (zero-copy)
    def gpu_rows(self):
        n = self.cfg.n_gpu_blocks * 64
        return _device_view(load().hs_gpu_rows(self.handle), (n, self.row_bytes), "|u1")

    def gpu_scales(self):
        if not self.fp8:
            return None
        return _device_view(load().hs_gpu_scales(self.handle), (self.cfg.n_gpu_blocks * 64,), "<f4")

    def host_rows(self) -> np.ndarray | None:
        p = load().hs_host_rows(self.handle)
        if not p:
            return None
        n = self.cfg.n_host_blocks * 64 * self.row_bytes
        return np.ctypeslib.as_array((C.c_uint8 * n).from_address(p)).reshape(-1, self.row_bytes)

    def host_scales(self) -> np.ndarray | None:
        p = load().hs_host_scales(self.handle)
        if not p:
            return None
        n = self.cfg.n_host_blocks * 64
        return np.ctypeslib.as_array((C.c_float * n).from_address(p))

    def host_rows_device(self):
        """The host arena as seen by the GPU (reads go over the host link), or None."""
        p = load().hs_host_rows_device(self.handle)
        if not p:
            return None
        return _device_view(p, (self.cfg.n_host_blocks * 64, self.row_bytes), "|u1")

    def host_scales_device(self):
        p = load().hs_host_scales_device(self.handle)
        if not p:
            return None
        return _device_view(p, (self.cfg.n_host_blocks * 64,), "<f4")

    def tables(self) -> dict:
        t, R, C_ = self._tables, self.cfg.max_requests, self.cfg.hot_rows
        return {
            "page_table": _device_view(t.page_table, (R, self.max_pages, 2), "<i4"),
            "hot_blocks": _device_view(t.hot_blocks, (R, C_ // 64), "<i4"),
            "slot_tag": _device_view(t.slot_tag, (R, C_), "<i4"),
            "slot_stamp": _device_view(t.slot_stamp, (R, C_), "<i4"),
            "lru_order": _device_view(t.lru_order, (R, C_), "<i4"),
            "pos_to_slot": _device_view(t.pos_to_slot, (R, self.cfg.max_ctx), "<i4"),
            "clock": _device_view(t.clock, (R,), "<i4"),
            "ctx_len": _device_view(t.ctx_len, (R,), "<i4"),
        }

    # hot path
    def resolve_topk(self, req_ids, topk_idx, resolved, gathered, gathered_scale, counts,
                     stream=None):
        hs_resolve_topk(self.handle, req_ids, topk_idx, resolved, gathered, gathered_scale,
                        counts, stream)

    def sparse_mla_decode(self, q, gathered, gathered_scale, resolved, topk_idx, req_ids,
                          sm_scale, out, lse, workspace=None, stream=None):
        hs_sparse_mla_decode(self.handle, q, gathered, gathered_scale, resolved, topk_idx,
                             req_ids, sm_scale, out, lse, workspace, stream)

    def resolve_topk_union(self, req_ids, topk_idx, resolved, gathered, gathered_scale, counts,
                           stream=None):
        hs_resolve_topk_union(self.handle, req_ids, topk_idx, resolved, gathered,
                              gathered_scale, counts, stream)

    def sparse_mla_decode_per_token(self, q, gathered, gathered_scale, resolved, topk_idx,
                                    req_ids, sm_scale, out, lse, workspace=None, stream=None):
        hs_sparse_mla_decode_per_token(self.handle, q, gathered, gathered_scale, resolved,
                                       topk_idx, req_ids, sm_scale, out, lse, workspace, stream)
