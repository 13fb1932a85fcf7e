// hs_decode.cu -- sparse MLA decode over the gathered top-K latent rows.
//
// Attention restricted to the K rows the indexer selected ("vLLM GLM 5.3 优化：
// 混合 HiSparse 卸载", section 解决 KV 缓存内存压力; "vLLM Hybrid HiSparse：稀疏MLA
// 破解长上下文显存瓶颈", section 稀疏MLA的核心思想). MLA keeps one 576-wide latent
// row per token; the key is the whole row and the value its first 512 elements.
// Query token t of a request sits at position L - T + t and sees entries whose
// position is <= that (MTP draft tokens share one top-K list).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <cstdint>

#include "hs_internal.cuh"

namespace {

constexpr int SIMPLE_WARPS = 8;

// One warp per query row (b, t, h); lanes own latent elements d = 32*i + lane.
template <bool FP8>
__global__ void __launch_bounds__(SIMPLE_WARPS * 32)
decode_rowwise_kernel(const __nv_bfloat16 *__restrict__ q, const uint8_t *__restrict__ gathered,
                      const float *__restrict__ gscale, const int32_t *__restrict__ resolved,
                      const int32_t *__restrict__ topk, const int32_t *__restrict__ req_ids,
                      const int32_t *__restrict__ ctx, int max_req, int T, int H, int K,
                      float sm_scale, __nv_bfloat16 *__restrict__ out, float *__restrict__ lse) {
    constexpr int NI = hs::kDim / 32;   // 18 elements per lane
    constexpr int NV = hs::kNope / 32;  // 16 value elements per lane
    const int lane = threadIdx.x & 31;
    const int h = blockIdx.x * SIMPLE_WARPS + (threadIdx.x >> 5);
    const int t = blockIdx.y, b = blockIdx.z;
    if (h >= H) return;
    const int r = req_ids[b];
    const int Lr = (r >= 0 && r < max_req) ? ctx[r] : 0;
    const int pos = Lr - T + t;
    const size_t qrow = ((size_t)b * T + t) * H + h;
    float qv[NI], acc[NV];
#pragma unroll
    for (int i = 0; i < NI; ++i) qv[i] = __bfloat162float(q[qrow * hs::kDim + 32 * i + lane]);
#pragma unroll
    for (int i = 0; i < NV; ++i) acc[i] = 0.f;
    float m = -INFINITY, l = 0.f;
    for (int j = 0; j < K; ++j) {
        const size_t bj = (size_t)b * K + j;
        if (resolved[bj] < 0 || topk[bj] > pos) continue;
        float kv[NI];
        if (FP8) {
            const uint8_t *row = gathered + bj * hs::kDim;
            const float sc = gscale[bj];
#pragma unroll
            for (int i = 0; i < NI; ++i) {
                __nv_fp8_e4m3 x;
                x.__x = row[32 * i + lane];
                kv[i] = static_cast<float>(x) * sc;
            }
        } else {
            const __nv_bfloat16 *row = reinterpret_cast<const __nv_bfloat16 *>(gathered) + bj * hs::kDim;
#pragma unroll
            for (int i = 0; i < NI; ++i) kv[i] = __bfloat162float(row[32 * i + lane]);
        }
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < NI; ++i) s = fmaf(qv[i], kv[i], s);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        s *= sm_scale;
        const float mn = fmaxf(m, s);
        const float alpha = expf(m - mn), p = expf(s - mn);
        l = l * alpha + p;
#pragma unroll
        for (int i = 0; i < NV; ++i) acc[i] = fmaf(acc[i], alpha, p * kv[i]);
        m = mn;
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int i = 0; i < NV; ++i) out[qrow * hs::kNope + 32 * i + lane] = __float2bfloat16_rn(acc[i] * inv);
    if (lane == 0) lse[qrow] = l > 0.f ? m + logf(l) : -INFINITY;
}

}  // namespace

extern "C" size_t hs_decode_workspace_bytes(int32_t B, int32_t T, int32_t H, int32_t K) {
    (void)B;
    (void)T;
    (void)H;
    (void)K;
    return 0;
}

extern "C" hs_status hs_sparse_mla_decode(hs_pool_t pool, int32_t B, int32_t T, int32_t H, int32_t K,
                                          const void *d_q, const void *d_gathered,
                                          const float *d_gathered_scale, const int32_t *d_resolved,
                                          const int32_t *d_topk_idx, const int32_t *d_req_ids,
                                          float sm_scale, void *d_out, float *d_lse,
                                          void *d_workspace, size_t ws_bytes, void *stream) {
    (void)d_workspace;
    (void)ws_bytes;
    if (!pool || !d_q || !d_gathered || !d_resolved || !d_topk_idx || !d_req_ids || !d_out || !d_lse)
        return HS_ERR_INVALID_ARG;
    if (B < 0 || T < 1 || H < 1 || K < 1 || B > 65535 || T > 65535 || H * T > 128 * 64)
        return HS_ERR_INVALID_ARG;
    const bool fp8 = pool->cfg.dtype == HS_FP8_E4M3_ROWSCALE;
    if (fp8 != (d_gathered_scale != nullptr)) return HS_ERR_INVALID_ARG;
    if (B == 0) return HS_OK;
    const dim3 grid((H + SIMPLE_WARPS - 1) / SIMPLE_WARPS, T, B);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const auto *q = static_cast<const __nv_bfloat16 *>(d_q);
    const auto *g = static_cast<const uint8_t *>(d_gathered);
    auto *o = static_cast<__nv_bfloat16 *>(d_out);
    if (fp8)
        decode_rowwise_kernel<true><<<grid, SIMPLE_WARPS * 32, 0, s>>>(
            q, g, d_gathered_scale, d_resolved, d_topk_idx, d_req_ids, pool->d_ctx,
            pool->cfg.max_requests, T, H, K, sm_scale, o, d_lse);
    else
        decode_rowwise_kernel<false><<<grid, SIMPLE_WARPS * 32, 0, s>>>(
            q, g, nullptr, d_resolved, d_topk_idx, d_req_ids, pool->d_ctx, pool->cfg.max_requests,
            T, H, K, sm_scale, o, d_lse);
    return cudaGetLastError() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}
