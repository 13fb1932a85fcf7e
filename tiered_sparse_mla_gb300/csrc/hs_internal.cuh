// hs_internal.cuh -- internal definitions of the CUDA path (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "hs.h"

namespace hs {

constexpr int kPage = 64;
constexpr int kNope = 512;
constexpr int kRope = 64;
constexpr int kDim = kNope + kRope;  // 576-wide latent row

// Device view of a pool, passed by value to kernels.
struct DevPool {
    uint8_t *rows;             // [n_gpu_rows][row_bytes] HBM pool
    float *scales;             // [n_gpu_rows] (FP8) or nullptr
    const uint8_t *host_rows;  // device address of the pinned host arena
    const float *host_scales;  // device address of the host scales (FP8) or nullptr
    const int2 *page;          // [max_req][max_pages] {gpu_block, host_block}
    const int32_t *hot_blocks; // [max_req][HB]
    int32_t *tag;              // [max_req][C]
    int32_t *stamp;            // [max_req][C]
    int32_t *lru;              // [max_req][C] slots sorted by (stamp, slot)
    int32_t *p2s;              // [max_req][max_ctx]
    int32_t *clock;            // [max_req]
    const int32_t *ctx;        // [max_req]
    uint32_t *err;             // device error word
    int max_req, max_pages, max_ctx, C, HB, row_bytes;
    int zero_row;              // a row of zeros (and scale 0) after the pool's blocks
};

}  // namespace hs

struct hs_pool {
    hs_pool_config cfg;
    int device = 0, sm_count = 0;
    cudaStream_t stream = nullptr;
    int row_bytes = 0, max_pages = 0, hb = 0;
    uint8_t *d_rows = nullptr;
    float *d_scales = nullptr;
    uint8_t *h_rows = nullptr, *hd_rows = nullptr;
    float *h_scales = nullptr, *hd_scales = nullptr;
    int32_t *d_page = nullptr, *d_hot_blocks = nullptr, *d_tag = nullptr, *d_stamp = nullptr;
    int32_t *d_lru = nullptr, *d_p2s = nullptr, *d_clock = nullptr, *d_ctx = nullptr;
    uint32_t *d_err = nullptr;
    int32_t *h_hot_blocks = nullptr;  // host shadow of hot_blocks (lease state)

    hs::DevPool dev() const {
        hs::DevPool p;
        p.rows = d_rows;
        p.scales = d_scales;
        p.host_rows = hd_rows;
        p.host_scales = hd_scales;
        p.page = reinterpret_cast<const int2 *>(d_page);
        p.hot_blocks = d_hot_blocks;
        p.tag = d_tag;
        p.stamp = d_stamp;
        p.lru = d_lru;
        p.p2s = d_p2s;
        p.clock = d_clock;
        p.ctx = d_ctx;
        p.err = d_err;
        p.max_req = cfg.max_requests;
        p.max_pages = max_pages;
        p.max_ctx = cfg.max_ctx;
        p.C = cfg.hot_rows;
        p.HB = hb;
        p.row_bytes = row_bytes;
        p.zero_row = (int)(cfg.n_gpu_blocks * hs::kPage);
        return p;
    }
};

#define HS_CUDA_TRY(expr)                                   \
    do {                                                    \
        cudaError_t e_ = (expr);                            \
        if (e_ != cudaSuccess) return HS_ERR_CUDA;          \
    } while (0)

// ---------------------------------------------------------------- PTX helpers
namespace hs {

__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// Address of the same shared-memory variable in cluster CTA `rank`.
__device__ __forceinline__ uint32_t dsmem_map(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ int32_t dsmem_ld(uint32_t a) {
    int32_t v;
    asm volatile("ld.shared::cluster.s32 %0, [%1];\n" : "=r"(v) : "r"(a) : "memory");
    return v;
}
__device__ __forceinline__ void dsmem_st(uint32_t a, int32_t v) {
    asm volatile("st.shared::cluster.s32 [%0], %1;\n" ::"r"(a), "r"(v) : "memory");
}

__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ld_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}
__device__ __forceinline__ void st_v4(void *p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};\n" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// Block-wide exclusive scan of a 0/1 flag. `s_warp` holds >= NT/32 ints.
// Contains __syncthreads(); every thread of the block must call it.
template <int NT>
__device__ __forceinline__ int block_scan_flag(int flag, int *s_warp, int &total) {
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const unsigned bal = __ballot_sync(0xffffffffu, flag);
    const int pre = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0) s_warp[w] = __popc(bal);
    __syncthreads();
    if (w == 0) {
        int v = lane < NW ? s_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int t = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += t;
        }
        if (lane < NW) s_warp[lane] = v;  // inclusive
    }
    __syncthreads();
    const int base = w ? s_warp[w - 1] : 0;
    total = s_warp[NW - 1];
    __syncthreads();
    return base + pre;
}

}  // namespace hs

// Launchers implemented in the .cu files.
hs_status hs_launch_resolve(hs_pool *pool, int32_t B, const int32_t *req_ids, const int32_t *topk,
                            int32_t K, int32_t *resolved, void *gathered, float *gscale,
                            int32_t *counts, cudaStream_t stream, int uni,
                            const hs::DevPool *layers, int nlayers);
size_t hs_resolve_smem_bytes(int K, int G, int C, int RB, bool stage);
hs_status hs_resolve_prepare(hs_pool *pool);
