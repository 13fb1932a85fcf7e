// hs_transition.cu -- residency transitions of pages, on the device.
//
// Active copy ("vLLM GLM 5.3 优化：混合 HiSparse 卸载", 混合 HiSparse 的技术实现 item 1
// and 关键架构细节, 主动复制): the finished prefix pages of a fully resident request
// are copied to pinned host memory while the GPU keeps serving them, so that a
// later demotion frees their GPU blocks without another copy.
//
// Demotion under pressure (same page, 混合 HiSparse 的技术实现 item 2; "vLLM Hybrid
// HiSparse：稀疏MLA破解长上下文显存瓶颈", 分级内存的运作机制): a request releases
// its coldest pages to host memory and keeps its tail on the GPU. The coldest
// pages are read as the oldest ones: every page that ends before the tail.
//
// Both are single launches over many pages or requests, asynchronous on the
// caller's stream (a side stream keeps the active copy off the decode path).
#include <cstdint>

#include "hs_internal.cuh"

namespace {

constexpr int CT = 256;  // threads per CTA

// One CTA per (request, page, host block) triple: the page's 64 rows (and FP8
// scales) go from its GPU block into the host block through the device-mapped
// arena, then the page table records the host copy. The page stays resident.
template <int RB>
__global__ void __launch_bounds__(CT)
active_copy_kernel(const uint8_t *__restrict__ rows, const float *__restrict__ scales,
                   uint8_t *__restrict__ host_rows, float *__restrict__ host_scales,
                   int32_t *__restrict__ page, int max_req, int max_pages, int n_host_blocks,
                   const int32_t *__restrict__ req, const int32_t *__restrict__ pg,
                   const int32_t *__restrict__ hblk, uint32_t *__restrict__ err) {
    constexpr int V = RB / 16;
    const int i = blockIdx.x;
    const int r = req[i], p = pg[i], hb = hblk[i];
    const bool in_range = r >= 0 && r < max_req && p >= 0 && p < max_pages && hb >= 0 &&
                          hb < n_host_blocks;
    int32_t *e = page + ((size_t)(in_range ? r : 0) * max_pages + (in_range ? p : 0)) * 2;
    const int gb = in_range ? e[0] : -1;
    if (gb < 0) {  // bad triple, or the page has no GPU block to copy from
        if (threadIdx.x == 0) atomicOr(err, HS_DEVERR_BAD_PAGE);
        return;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(rows + (size_t)gb * hs::kPage * RB);
    uint4 *dst = reinterpret_cast<uint4 *>(host_rows + (size_t)hb * hs::kPage * RB);
    constexpr int N = hs::kPage * V;  // 16-byte vectors per page
    for (int b = threadIdx.x; b < N; b += CT * 4) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (b + u * CT < N) v[u] = src[b + u * CT];
#pragma unroll
        for (int u = 0; u < 4; ++u)
            if (b + u * CT < N) dst[b + u * CT] = v[u];
    }
    if (scales && threadIdx.x < hs::kPage)
        host_scales[(size_t)hb * hs::kPage + threadIdx.x] = scales[(size_t)gb * hs::kPage + threadIdx.x];
    __threadfence_system();  // the host copy is complete before the table names it
    __syncthreads();
    if (threadIdx.x == 0) e[1] = hb;
}

// One CTA per request: pages [0, (L - keep_tail) / 64) that are resident and
// have a host copy lose their GPU block; the freed blocks are listed in
// ascending page order.
__global__ void __launch_bounds__(CT)
demote_kernel(int32_t *__restrict__ page, const int32_t *__restrict__ ctx, int max_req,
              int max_pages, const int32_t *__restrict__ req, const int32_t *__restrict__ keep_tail,
              int32_t *__restrict__ freed, int32_t *__restrict__ n_freed, uint32_t *__restrict__ err) {
    __shared__ int s_warp[CT / 32];
    const int i = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int r = req[i], kt = keep_tail[i];
    int32_t *out = freed + (size_t)i * max_pages;
    if (r < 0 || r >= max_req || kt < 0) {
        if (tid == 0) {
            n_freed[i] = 0;
            atomicOr(err, r < 0 || r >= max_req ? HS_DEVERR_BAD_REQUEST : HS_DEVERR_BAD_PAGE);
        }
        return;
    }
    const long long cold_tokens = (long long)ctx[r] - kt;
    const long long cold_pages = cold_tokens <= 0 ? 0 : cold_tokens / hs::kPage;
    const int ncold = cold_pages < max_pages ? (int)cold_pages : max_pages;
    int32_t *pr = page + (size_t)r * max_pages * 2;
    int done = 0;
    for (int base = 0; base < ncold; base += CT) {  // uniform trip count
        const int p = base + tid;
        int gb = -1;
        if (p < ncold && pr[2 * p] >= 0 && pr[2 * p + 1] >= 0) gb = pr[2 * p];
        const unsigned bal = __ballot_sync(0xffffffffu, gb >= 0);
        if (lane == 0) s_warp[w] = __popc(bal);
        __syncthreads();
        int before = 0, tot = 0;
        for (int q = 0; q < CT / 32; ++q) {
            before += q < w ? s_warp[q] : 0;
            tot += s_warp[q];
        }
        if (gb >= 0) {
            out[done + before + __popc(bal & ((1u << lane) - 1u))] = gb;
            pr[2 * p] = -1;
        }
        done += tot;
        __syncthreads();  // s_warp is rewritten next round
    }
    if (tid == 0) n_freed[i] = done;
}

}  // namespace

extern "C" hs_status hs_active_copy(hs_pool_t pool, int32_t n, const int32_t *d_req,
                                    const int32_t *d_page, const int32_t *d_host_block,
                                    void *stream) {
    if (!pool || n < 0 || (n > 0 && (!d_req || !d_page || !d_host_block)))
        return HS_ERR_INVALID_ARG;
    if (pool->cfg.n_host_blocks < 1) return HS_ERR_INVALID_ARG;
    if (n == 0) return HS_OK;
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int hb = static_cast<int>(pool->cfg.n_host_blocks);
    float *hsc = pool->hd_scales;
    if (pool->row_bytes == 1152)
        active_copy_kernel<1152><<<n, CT, 0, s>>>(pool->d_rows, pool->d_scales, pool->hd_rows, hsc,
                                                  pool->d_page, pool->cfg.max_requests,
                                                  pool->max_pages, hb, d_req, d_page, d_host_block,
                                                  pool->d_err);
    else
        active_copy_kernel<576><<<n, CT, 0, s>>>(pool->d_rows, pool->d_scales, pool->hd_rows, hsc,
                                                 pool->d_page, pool->cfg.max_requests,
                                                 pool->max_pages, hb, d_req, d_page, d_host_block,
                                                 pool->d_err);
    return cudaGetLastError() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

extern "C" hs_status hs_demote_cold_pages(hs_pool_t pool, int32_t n, const int32_t *d_req,
                                          const int32_t *d_keep_tail, int32_t *d_freed,
                                          int32_t *d_n_freed, void *stream) {
    if (!pool || n < 0 || (n > 0 && (!d_req || !d_keep_tail || !d_freed || !d_n_freed)))
        return HS_ERR_INVALID_ARG;
    if (n == 0) return HS_OK;
    demote_kernel<<<n, CT, 0, static_cast<cudaStream_t>(stream)>>>(
        pool->d_page, pool->d_ctx, pool->cfg.max_requests, pool->max_pages, d_req, d_keep_tail,
        d_freed, d_n_freed, pool->d_err);
    return cudaGetLastError() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}
