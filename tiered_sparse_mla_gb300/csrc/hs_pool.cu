// hs_pool.cu -- the tiered KV pool: HBM block pool, pinned device-mapped host
// arena, page/residency table and per-request hot-buffer LRU state.
//
// One shared block pool holds every GPU row, pages and hot buffers alike; the
// hot buffer is a set of ordinary blocks leased from it ("vLLM GLM 5.3 优化：
// 混合 HiSparse 卸载", sections 混合 HiSparse 的技术实现 and 关键架构细节; "vLLM
// Hybrid HiSparse：稀疏MLA破解长上下文显存瓶颈", section 复用现有内存池).
// Residency is tracked per page.
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "hs_internal.cuh"

namespace {

__global__ void fill_i32_kernel(int32_t *p, int64_t n, int32_t v) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        p[i] = v;
}

// lru_order rows = 0..C-1 (every stamp is -1, so (stamp, slot) order is slot order)
__global__ void iota_rows_kernel(int32_t *p, int64_t rows, int32_t C) {
    const int64_t n = rows * C;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        p[i] = static_cast<int32_t>(i % C);
}

hs_status fill(int32_t *p, int64_t n, int32_t v, cudaStream_t s) {
    if (n <= 0) return HS_OK;
    int blocks = static_cast<int>((n + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    fill_i32_kernel<<<blocks, 256, 0, s>>>(p, n, v);
    HS_CUDA_TRY(cudaGetLastError());
    return HS_OK;
}

hs_status iota_rows(int32_t *p, int64_t rows, int32_t C, cudaStream_t s) {
    int64_t n = rows * C;
    if (n <= 0) return HS_OK;
    int blocks = static_cast<int>((n + 255) / 256);
    if (blocks > 4096) blocks = 4096;
    iota_rows_kernel<<<blocks, 256, 0, s>>>(p, rows, C);
    HS_CUDA_TRY(cudaGetLastError());
    return HS_OK;
}

// Clears the hot-buffer state of one request.
hs_status clear_hot_state(hs_pool *p, int32_t req) {
    const int C = p->cfg.hot_rows;
    hs_status st;
    if ((st = fill(p->d_tag + (int64_t)req * C, C, -1, p->stream)) != HS_OK) return st;
    if ((st = fill(p->d_stamp + (int64_t)req * C, C, -1, p->stream)) != HS_OK) return st;
    if ((st = iota_rows(p->d_lru + (int64_t)req * C, 1, C, p->stream)) != HS_OK) return st;
    if ((st = fill(p->d_p2s + (int64_t)req * p->cfg.max_ctx, p->cfg.max_ctx, -1, p->stream)) !=
        HS_OK)
        return st;
    HS_CUDA_TRY(cudaMemsetAsync(p->d_clock + req, 0, sizeof(int32_t), p->stream));
    return HS_OK;
}

void free_all(hs_pool *p) {
    cudaFree(p->d_rows);
    cudaFree(p->d_scales);
    if (p->h_rows) cudaFreeHost(p->h_rows);
    if (p->h_scales) cudaFreeHost(p->h_scales);
    cudaFree(p->d_page);
    cudaFree(p->d_hot_blocks);
    cudaFree(p->d_tag);
    cudaFree(p->d_stamp);
    cudaFree(p->d_lru);
    cudaFree(p->d_p2s);
    cudaFree(p->d_clock);
    cudaFree(p->d_ctx);
    cudaFree(p->d_err);
    free(p->h_hot_blocks);
}

bool req_ok(hs_pool *p, int32_t req) { return p && req >= 0 && req < p->cfg.max_requests; }

struct SnapHeader {
    uint32_t magic;
    int32_t max_req, hot_rows, max_ctx;
};
constexpr uint32_t kSnapMagic = 0x31535348u;  // "HSS1"

}  // namespace

extern "C" {

const char *hs_status_string(hs_status s) {
    switch (s) {
        case HS_OK: return "ok";
        case HS_ERR_INVALID_ARG: return "invalid argument";
        case HS_ERR_CAPACITY: return "capacity exceeded";
        case HS_ERR_OUT_OF_MEMORY: return "out of memory";
        case HS_ERR_CUDA: return "CUDA error";
        case HS_ERR_DEVICE_DATA: return "device data error";
        case HS_ERR_TIMEOUT: return "device wait timed out";
        case HS_ERR_UNSUPPORTED: return "unsupported";
    }
    return "unknown status";
}

hs_status hs_pool_create(const hs_pool_config *cfg_in, void *stream, hs_pool_t *out) {
    if (!cfg_in || !out) return HS_ERR_INVALID_ARG;
    *out = nullptr;
    hs_pool_config cfg = *cfg_in;
    if (cfg.nope_dim != hs::kNope || cfg.rope_dim != hs::kRope || cfg.page_size != hs::kPage)
        return HS_ERR_UNSUPPORTED;
    if (cfg.dtype != HS_BF16 && cfg.dtype != HS_FP8_E4M3_ROWSCALE) return HS_ERR_INVALID_ARG;
    if (cfg.max_topk < 1 || cfg.max_topk > 8192) return HS_ERR_INVALID_ARG;
    if (cfg.hot_rows == 0) cfg.hot_rows = 2 * cfg.max_topk;
    if (cfg.hot_rows < 0 || cfg.hot_rows % hs::kPage != 0 || cfg.hot_rows > 16384)
        return HS_ERR_INVALID_ARG;
    if (cfg.max_requests < 1 || cfg.max_ctx < 1 || cfg.n_gpu_blocks < 1 || cfg.n_host_blocks < 0)
        return HS_ERR_INVALID_ARG;
    // row ids are int32 on the device
    if ((cfg.n_gpu_blocks + 1) * hs::kPage >= (int64_t(1) << 31) ||
        cfg.n_host_blocks * hs::kPage >= (int64_t(1) << 31))
        return HS_ERR_INVALID_ARG;

    int dev = 0;
    HS_CUDA_TRY(cudaGetDevice(&dev));
    cudaDeviceProp prop;
    HS_CUDA_TRY(cudaGetDeviceProperties(&prop, dev));
    if (!(prop.major == 10 && prop.minor == 3)) return HS_ERR_UNSUPPORTED;

    hs_pool *p = new (std::nothrow) hs_pool();
    if (!p) return HS_ERR_OUT_OF_MEMORY;
    p->cfg = cfg;
    p->device = dev;
    p->sm_count = prop.multiProcessorCount;
    p->stream = static_cast<cudaStream_t>(stream);
    p->row_bytes = cfg.dtype == HS_BF16 ? 2 * hs::kDim : hs::kDim;
    p->max_pages = (cfg.max_ctx + hs::kPage - 1) / hs::kPage;
    p->hb = cfg.hot_rows / hs::kPage;
    const int64_t R = cfg.max_requests, C = cfg.hot_rows;
    const bool fp8 = cfg.dtype == HS_FP8_E4M3_ROWSCALE;
    // one block more than the caller's: a block of zero rows (scale 0) that
    // attention reads in place of absent entries
    const size_t gpu_rows = (size_t)(cfg.n_gpu_blocks + 1) * hs::kPage;
    const size_t host_rows = (size_t)cfg.n_host_blocks * hs::kPage;

    bool ok = true;
    ok = ok && cudaMalloc(&p->d_rows, gpu_rows * p->row_bytes) == cudaSuccess;
    if (fp8) ok = ok && cudaMalloc(&p->d_scales, gpu_rows * sizeof(float)) == cudaSuccess;
    if (ok && host_rows > 0) {
        ok = cudaHostAlloc(reinterpret_cast<void **>(&p->h_rows), host_rows * p->row_bytes,
                           cudaHostAllocMapped | cudaHostAllocPortable) == cudaSuccess;
        ok = ok && cudaHostGetDevicePointer(reinterpret_cast<void **>(&p->hd_rows), p->h_rows, 0) ==
                       cudaSuccess;
        if (ok && fp8) {
            ok = cudaHostAlloc(reinterpret_cast<void **>(&p->h_scales), host_rows * sizeof(float),
                               cudaHostAllocMapped | cudaHostAllocPortable) == cudaSuccess;
            ok = ok && cudaHostGetDevicePointer(reinterpret_cast<void **>(&p->hd_scales),
                                                p->h_scales, 0) == cudaSuccess;
        }
    }
    ok = ok && cudaMalloc(&p->d_page, R * p->max_pages * 2 * sizeof(int32_t)) == cudaSuccess;
    ok = ok && cudaMalloc(&p->d_hot_blocks, R * p->hb * sizeof(int32_t)) == cudaSuccess;
    ok = ok && cudaMalloc(&p->d_tag, R * C * sizeof(int32_t)) == cudaSuccess;
    ok = ok && cudaMalloc(&p->d_stamp, R * C * sizeof(int32_t)) == cudaSuccess;
    ok = ok && cudaMalloc(&p->d_lru, R * C * sizeof(int32_t)) == cudaSuccess;
    ok = ok && cudaMalloc(&p->d_p2s, R * (int64_t)cfg.max_ctx * sizeof(int32_t)) == cudaSuccess;
    ok = ok && cudaMalloc(&p->d_clock, R * sizeof(int32_t)) == cudaSuccess;
    ok = ok && cudaMalloc(&p->d_ctx, R * sizeof(int32_t)) == cudaSuccess;
    ok = ok && cudaMalloc(&p->d_err, sizeof(uint32_t)) == cudaSuccess;
    p->h_hot_blocks = static_cast<int32_t *>(malloc(R * p->hb * sizeof(int32_t)));
    ok = ok && p->h_hot_blocks != nullptr;
    if (!ok) {
        cudaGetLastError();  // clear the sticky-free allocation error
        free_all(p);
        delete p;
        return HS_ERR_OUT_OF_MEMORY;
    }
    for (int64_t i = 0; i < R * p->hb; ++i) p->h_hot_blocks[i] = -1;

    hs_status st = HS_OK;
    cudaStream_t s = p->stream;
    if (st == HS_OK) st = fill(p->d_page, R * p->max_pages * 2, -1, s);
    if (st == HS_OK) st = fill(p->d_hot_blocks, R * p->hb, -1, s);
    if (st == HS_OK) st = fill(p->d_tag, R * C, -1, s);
    if (st == HS_OK) st = fill(p->d_stamp, R * C, -1, s);
    if (st == HS_OK) st = iota_rows(p->d_lru, R, (int32_t)C, s);
    if (st == HS_OK) st = fill(p->d_p2s, R * (int64_t)cfg.max_ctx, -1, s);
    if (st == HS_OK) st = fill(p->d_clock, R, 0, s);
    if (st == HS_OK) st = fill(p->d_ctx, R, 0, s);
    if (st == HS_OK && cudaMemsetAsync(p->d_err, 0, sizeof(uint32_t), s) != cudaSuccess)
        st = HS_ERR_CUDA;
    const size_t zero0 = (size_t)cfg.n_gpu_blocks * hs::kPage;
    if (st == HS_OK && cudaMemsetAsync(p->d_rows + zero0 * p->row_bytes, 0,
                                       (size_t)hs::kPage * p->row_bytes, s) != cudaSuccess)
        st = HS_ERR_CUDA;
    if (st == HS_OK && fp8 &&
        cudaMemsetAsync(p->d_scales + zero0, 0, hs::kPage * sizeof(float), s) != cudaSuccess)
        st = HS_ERR_CUDA;
    if (st == HS_OK) st = hs_resolve_prepare(p);
    if (st == HS_OK && cudaStreamSynchronize(s) != cudaSuccess) st = HS_ERR_CUDA;
    if (st != HS_OK) {
        free_all(p);
        delete p;
        return st;
    }
    *out = p;
    return HS_OK;
}

hs_status hs_pool_destroy(hs_pool_t p) {
    if (!p) return HS_ERR_INVALID_ARG;
    cudaStreamSynchronize(p->stream);
    free_all(p);
    delete p;
    return HS_OK;
}

hs_status hs_pool_get_config(hs_pool_t p, hs_pool_config *out) {
    if (!p || !out) return HS_ERR_INVALID_ARG;
    *out = p->cfg;
    return HS_OK;
}

hs_status hs_pool_get_tables(hs_pool_t p, hs_pool_tables *out) {
    if (!p || !out) return HS_ERR_INVALID_ARG;
    out->page_table = p->d_page;
    out->hot_blocks = p->d_hot_blocks;
    out->slot_tag = p->d_tag;
    out->slot_stamp = p->d_stamp;
    out->lru_order = p->d_lru;
    out->pos_to_slot = p->d_p2s;
    out->clock = p->d_clock;
    out->ctx_len = p->d_ctx;
    out->max_pages = p->max_pages;
    out->row_bytes = p->row_bytes;
    return HS_OK;
}

hs_status hs_request_init(hs_pool_t p, int32_t req, int32_t ctx_len) {
    if (!req_ok(p, req) || ctx_len < 0 || ctx_len > p->cfg.max_ctx) return HS_ERR_INVALID_ARG;
    hs_status st = fill(p->d_page + (int64_t)req * p->max_pages * 2, p->max_pages * 2, -1, p->stream);
    if (st != HS_OK) return st;
    if ((st = clear_hot_state(p, req)) != HS_OK) return st;
    return hs_request_set_ctx_len(p, req, ctx_len);
}

hs_status hs_request_set_ctx_len(hs_pool_t p, int32_t req, int32_t ctx_len) {
    if (!req_ok(p, req) || ctx_len < 0 || ctx_len > p->cfg.max_ctx) return HS_ERR_INVALID_ARG;
    return fill(p->d_ctx + req, 1, ctx_len, p->stream);
}

hs_status hs_set_ctx_len(hs_pool_t p, const int32_t *d_ctx_len, int32_t n, void *stream) {
    if (!p || !d_ctx_len || n < 0 || n > p->cfg.max_requests) return HS_ERR_INVALID_ARG;
    if (n == 0) return HS_OK;
    HS_CUDA_TRY(cudaMemcpyAsync(p->d_ctx, d_ctx_len, n * sizeof(int32_t), cudaMemcpyDeviceToDevice,
                                static_cast<cudaStream_t>(stream)));
    return HS_OK;
}

hs_status hs_page_map(hs_pool_t p, int32_t req, int32_t page, int64_t gpu_block,
                      int64_t host_block) {
    int32_t g = static_cast<int32_t>(gpu_block), h = static_cast<int32_t>(host_block);
    if (gpu_block < -1 || host_block < -1) return HS_ERR_INVALID_ARG;
    return hs_page_map_range(p, req, page, 1, &g, &h);
}

hs_status hs_page_map_range(hs_pool_t p, int32_t req, int32_t first, int32_t n,
                            const int32_t *gpu_blocks, const int32_t *host_blocks) {
    if (!req_ok(p, req) || !gpu_blocks || !host_blocks || n < 0 || first < 0 ||
        (int64_t)first + n > p->max_pages)
        return HS_ERR_INVALID_ARG;
    std::vector<int32_t> buf(2 * (size_t)n);
    for (int32_t i = 0; i < n; ++i) {
        if (gpu_blocks[i] < -1 || gpu_blocks[i] >= p->cfg.n_gpu_blocks) return HS_ERR_INVALID_ARG;
        if (host_blocks[i] < -1 || host_blocks[i] >= p->cfg.n_host_blocks) return HS_ERR_INVALID_ARG;
        buf[2 * i] = gpu_blocks[i];
        buf[2 * i + 1] = host_blocks[i];
    }
    if (n == 0) return HS_OK;
    // pageable source: the bytes are staged before cudaMemcpyAsync returns
    HS_CUDA_TRY(cudaMemcpyAsync(p->d_page + ((int64_t)req * p->max_pages + first) * 2, buf.data(),
                                buf.size() * sizeof(int32_t), cudaMemcpyHostToDevice, p->stream));
    return HS_OK;
}

hs_status hs_hot_lease(hs_pool_t p, int32_t req, const int64_t *blocks, int32_t n) {
    if (!req_ok(p, req) || !blocks || n != p->hb) return HS_ERR_INVALID_ARG;
    std::vector<int32_t> b(n);
    for (int32_t i = 0; i < n; ++i) {
        if (blocks[i] < 0 || blocks[i] >= p->cfg.n_gpu_blocks) return HS_ERR_INVALID_ARG;
        b[i] = static_cast<int32_t>(blocks[i]);
    }
    memcpy(p->h_hot_blocks + (int64_t)req * p->hb, b.data(), n * sizeof(int32_t));
    HS_CUDA_TRY(cudaMemcpyAsync(p->d_hot_blocks + (int64_t)req * p->hb, b.data(),
                                n * sizeof(int32_t), cudaMemcpyHostToDevice, p->stream));
    return clear_hot_state(p, req);
}

hs_status hs_hot_release(hs_pool_t p, int32_t req) {
    if (!req_ok(p, req)) return HS_ERR_INVALID_ARG;
    for (int i = 0; i < p->hb; ++i) p->h_hot_blocks[(int64_t)req * p->hb + i] = -1;
    hs_status st = fill(p->d_hot_blocks + (int64_t)req * p->hb, p->hb, -1, p->stream);
    if (st != HS_OK) return st;
    return clear_hot_state(p, req);
}

void *hs_gpu_rows(hs_pool_t p) { return p ? p->d_rows : nullptr; }
void *hs_host_rows(hs_pool_t p) { return p ? p->h_rows : nullptr; }
float *hs_gpu_scales(hs_pool_t p) { return p ? p->d_scales : nullptr; }
float *hs_host_scales(hs_pool_t p) { return p ? p->h_scales : nullptr; }
void *hs_host_rows_device(hs_pool_t p) { return p ? p->hd_rows : nullptr; }
float *hs_host_scales_device(hs_pool_t p) { return p ? p->hd_scales : nullptr; }

hs_status hs_pool_snapshot(hs_pool_t p, void *dst, size_t cap, size_t *used) {
    if (!p) return HS_ERR_INVALID_ARG;
    const size_t R = p->cfg.max_requests, C = p->cfg.hot_rows, X = p->cfg.max_ctx;
    const size_t need = sizeof(SnapHeader) + sizeof(int32_t) * (R + 3 * R * C + R * X);
    if (used) *used = need;
    if (!dst) return HS_OK;
    if (cap < need) return HS_ERR_CAPACITY;
    SnapHeader h{kSnapMagic, (int32_t)R, (int32_t)C, (int32_t)X};
    memcpy(dst, &h, sizeof h);
    char *o = static_cast<char *>(dst) + sizeof h;
    HS_CUDA_TRY(cudaStreamSynchronize(p->stream));
    HS_CUDA_TRY(cudaDeviceSynchronize());
    HS_CUDA_TRY(cudaMemcpy(o, p->d_clock, R * 4, cudaMemcpyDeviceToHost));
    o += R * 4;
    HS_CUDA_TRY(cudaMemcpy(o, p->d_tag, R * C * 4, cudaMemcpyDeviceToHost));
    o += R * C * 4;
    HS_CUDA_TRY(cudaMemcpy(o, p->d_stamp, R * C * 4, cudaMemcpyDeviceToHost));
    o += R * C * 4;
    HS_CUDA_TRY(cudaMemcpy(o, p->d_lru, R * C * 4, cudaMemcpyDeviceToHost));
    o += R * C * 4;
    HS_CUDA_TRY(cudaMemcpy(o, p->d_p2s, R * X * 4, cudaMemcpyDeviceToHost));
    return HS_OK;
}

hs_status hs_pool_restore(hs_pool_t p, const void *src, size_t n) {
    if (!p || !src) return HS_ERR_INVALID_ARG;
    const size_t R = p->cfg.max_requests, C = p->cfg.hot_rows, X = p->cfg.max_ctx;
    const size_t need = sizeof(SnapHeader) + sizeof(int32_t) * (R + 3 * R * C + R * X);
    if (n < need) return HS_ERR_INVALID_ARG;
    SnapHeader h;
    memcpy(&h, src, sizeof h);
    if (h.magic != kSnapMagic || h.max_req != (int32_t)R || h.hot_rows != (int32_t)C ||
        h.max_ctx != (int32_t)X)
        return HS_ERR_INVALID_ARG;
    const char *o = static_cast<const char *>(src) + sizeof h;
    HS_CUDA_TRY(cudaDeviceSynchronize());
    HS_CUDA_TRY(cudaMemcpy(p->d_clock, o, R * 4, cudaMemcpyHostToDevice));
    o += R * 4;
    HS_CUDA_TRY(cudaMemcpy(p->d_tag, o, R * C * 4, cudaMemcpyHostToDevice));
    o += R * C * 4;
    HS_CUDA_TRY(cudaMemcpy(p->d_stamp, o, R * C * 4, cudaMemcpyHostToDevice));
    o += R * C * 4;
    HS_CUDA_TRY(cudaMemcpy(p->d_lru, o, R * C * 4, cudaMemcpyHostToDevice));
    o += R * C * 4;
    HS_CUDA_TRY(cudaMemcpy(p->d_p2s, o, R * X * 4, cudaMemcpyHostToDevice));
    return HS_OK;
}

hs_status hs_pool_get_error(hs_pool_t p, uint32_t *bits) {
    if (!p || !bits) return HS_ERR_INVALID_ARG;
    HS_CUDA_TRY(cudaDeviceSynchronize());
    HS_CUDA_TRY(cudaMemcpy(bits, p->d_err, sizeof(uint32_t), cudaMemcpyDeviceToHost));
    HS_CUDA_TRY(cudaMemset(p->d_err, 0, sizeof(uint32_t)));
    return HS_OK;
}

}  // extern "C"
