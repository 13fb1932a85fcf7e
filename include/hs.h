/*
 * hs.h -- C ABI of the GB300 (sm_103a) tiered sparse-MLA decode path.
 *
 * The operation ("vLLM GLM 5.3 优化：混合 HiSparse 卸载", sections 解决 KV 缓存内存压力,
 * 混合 HiSparse 的技术实现 and 关键架构细节; "vLLM Hybrid HiSparse：稀疏MLA破解长上下文
 * 显存瓶颈", sections 稀疏MLA的核心思想, 分级内存的运作机制 and 融合内核与CUDA图兼容):
 * each decode step a sparse-MLA indexer selects K token positions per request.
 * The request's latent KV rows live in a tiered cache: pages resident in one
 * shared GPU block pool, a per-request hot buffer of (by default) 2*K rows made
 * of ordinary blocks leased from that same pool, and pinned host memory.
 * hs_resolve_topk makes every selected row GPU-addressable in one fused,
 * CUDA-graph-capturable launch; hs_sparse_mla_decode then runs MLA attention
 * over only those K rows. Variants: one list per speculative query token
 * (hs_resolve_topk_union, hs_sparse_mla_decode_per_token), several layers'
 * pools resolved in one launch (hs_resolve_topk_layers), and the residency
 * transitions around the path (hs_active_copy, hs_demote_cold_pages).
 *
 * Conventions
 *  - Streams are cudaStream_t values passed as void* (NULL = legacy stream).
 *  - Pointers named d_* are device pointers owned by the caller. The pool owns
 *    its HBM pool, its pinned host arena and every table.
 *  - Host-side argument errors return a status at once and launch nothing.
 *  - Data errors found on the device set bits in the pool's device error word
 *    (HS_DEVERR_*), never trap; the affected entries resolve to -1.
 *  - A pool is not thread-safe; use it from one host thread.
 *  - Row layout: 576 latent elements per token (512 "nope" + 64 "rope").
 *    HS_BF16 rows are 1152 bytes. HS_FP8_E4M3_ROWSCALE rows are 576 e4m3fn
 *    bytes; each row's fp32 scale lives in a parallel array (value = code*scale).
 */
#ifndef HS_H
#define HS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct hs_pool *hs_pool_t;
typedef struct hs_layer_group *hs_layer_group_t;

typedef enum {
    HS_OK = 0,
    HS_ERR_INVALID_ARG = 1,   /* bad pointer, size, id or alignment            */
    HS_ERR_CAPACITY = 2,      /* K above the hot buffer or max_topk, etc.      */
    HS_ERR_OUT_OF_MEMORY = 3, /* device or pinned host allocation failed       */
    HS_ERR_CUDA = 4,          /* a CUDA runtime call failed                    */
    HS_ERR_DEVICE_DATA = 5,   /* the device error word is non-zero             */
    HS_ERR_TIMEOUT = 6,       /* a bounded device wait gave up                 */
    HS_ERR_UNSUPPORTED = 7    /* shape or device outside what is implemented   */
} hs_status;

/* Bits of the device error word (hs_pool_get_error). */
#define HS_DEVERR_INDEX_RANGE 1u  /* position outside [0, ctx_len) (and not -1)   */
#define HS_DEVERR_DUPLICATE   2u  /* a missing position repeated in one list      */
#define HS_DEVERR_NO_HOST     4u  /* non-resident, non-hot row without host copy  */
#define HS_DEVERR_BAD_REQUEST 8u  /* request id outside [0, max_requests)         */
#define HS_DEVERR_CAPACITY    16u /* more misses than unprotected hot slots       */
#define HS_DEVERR_TIMEOUT     32u /* a bounded device wait gave up                */
#define HS_DEVERR_BAD_PAGE    64u /* a page transition named a page, block or tail
                                     it cannot apply to (that entry is skipped)     */

typedef enum { HS_BF16 = 0, HS_FP8_E4M3_ROWSCALE = 1 } hs_kv_dtype;

typedef struct {
    int32_t nope_dim;      /* 512 (only value implemented)                          */
    int32_t rope_dim;      /* 64  (only value implemented)                          */
    int32_t page_size;     /* 64 tokens per block (only value implemented)          */
    int32_t dtype;         /* hs_kv_dtype                                           */
    int64_t n_gpu_blocks;  /* blocks in the HBM pool (pages and hot buffers)        */
    int64_t n_host_blocks; /* blocks in the pinned, device-mapped host arena (>= 0) */
    int32_t max_requests;  /* request ids are 0 .. max_requests-1                   */
    int32_t max_ctx;       /* largest context length of any request (tokens)       */
    int32_t hot_rows;      /* hot-buffer rows per request; multiple of page_size;
                              0 selects 2*max_topk                                  */
    int32_t max_topk;      /* largest K (1 .. 8192) of any resolve: one list of at
                              most hot_rows entries, or a union of several lists  */
} hs_pool_config;

/* Device pointers to the pool's tables, for inspection after synchronising the
 * pool's stream. Layouts (row-major):
 *   page_table  int32 [max_requests][max_pages][2] = {gpu_block, host_block}, -1 = none
 *   hot_blocks  int32 [max_requests][hot_rows/64]  (-1 = not leased)
 *   slot_tag    int32 [max_requests][hot_rows]  token position held, -1 = empty
 *   slot_stamp  int32 [max_requests][hot_rows]  clock of last use, -1 = never
 *   lru_order   int32 [max_requests][hot_rows]  slots sorted by (stamp, slot)
 *   pos_to_slot int32 [max_requests][max_ctx]   hot slot of a position, -1 = none
 *   clock       int32 [max_requests]            decode steps resolved so far
 *   ctx_len     int32 [max_requests]
 * Pool row i (block i/64, offset i%64) is at gpu_rows + i*row_bytes. */
typedef struct {
    int32_t *page_table, *hot_blocks, *slot_tag, *slot_stamp, *lru_order, *pos_to_slot;
    int32_t *clock, *ctx_len;
    int32_t max_pages, row_bytes;
} hs_pool_tables;

/* ---- pool lifetime (allocates; not for the graph path) ------------------- */

/* Creates a pool on the current device: HBM pool, pinned mapped host arena,
 * tables (all entries -1, clocks 0). `stream` orders the pool's own copies.
 * Returns HS_ERR_UNSUPPORTED on a device without sm_103 features. */
hs_status hs_pool_create(const hs_pool_config *cfg, void *stream, hs_pool_t *out);
hs_status hs_pool_destroy(hs_pool_t pool);
hs_status hs_pool_get_config(hs_pool_t pool, hs_pool_config *out);
hs_status hs_pool_get_tables(hs_pool_t pool, hs_pool_tables *out);

/* ---- scheduler bookkeeping (host calls, ordered on the pool's stream) ----- */

/* Starts request `req` afresh: unmaps every page, clears its hot-buffer state
 * (tags, stamps, pos_to_slot, LRU order), sets clock 0 and ctx_len. Leased hot
 * blocks stay leased. */
hs_status hs_request_init(hs_pool_t pool, int32_t req, int32_t ctx_len);
/* Sets ctx_len of one request (positions >= ctx_len are out of range). */
hs_status hs_request_set_ctx_len(hs_pool_t pool, int32_t req, int32_t ctx_len);
/* Copies n context lengths from device memory into requests 0..n-1. */
hs_status hs_set_ctx_len(hs_pool_t pool, const int32_t *d_ctx_len, int32_t n, void *stream);
/* Maps one page: gpu_block (-1 = not resident) and host_block (-1 = no copy). */
hs_status hs_page_map(hs_pool_t pool, int32_t req, int32_t page, int64_t gpu_block,
                      int64_t host_block);
/* Maps pages first..first+n-1 from two host arrays (entries may be -1). */
hs_status hs_page_map_range(hs_pool_t pool, int32_t req, int32_t first, int32_t n,
                            const int32_t *gpu_blocks, const int32_t *host_blocks);
/* Leases n = hot_rows/64 pool blocks as the request's hot buffer and clears
 * its hot state. The hot buffer is made of ordinary pool blocks, not a
 * separate allocation (关键架构细节, 热缓冲区). */
hs_status hs_hot_lease(hs_pool_t pool, int32_t req, const int64_t *blocks, int32_t n);
/* Returns the hot blocks (entries -1) and clears the request's hot state. */
hs_status hs_hot_release(hs_pool_t pool, int32_t req);

/* Row storage. Rows may be written by the caller (stream-ordered before the
 * step that reads them). Host pointers are the CPU addresses of the arena. */
void *hs_gpu_rows(hs_pool_t pool);
void *hs_host_rows(hs_pool_t pool);
float *hs_gpu_scales(hs_pool_t pool);  /* NULL for HS_BF16 */
float *hs_host_scales(hs_pool_t pool); /* NULL for HS_BF16 */
/* Device addresses of the host arena's mapping (the addresses the resolve
 * reads misses through), for the caller's own kernels that read the arena.
 * NULL when the pool has no host arena (scales: also for HS_BF16). */
void *hs_host_rows_device(hs_pool_t pool);
float *hs_host_scales_device(hs_pool_t pool);

/* Snapshot / restore of the hot-buffer state of all requests (clock, slot_tag,
 * slot_stamp, lru_order, pos_to_slot) to / from host memory. Synchronous.
 * hs_pool_snapshot with host_dst NULL reports the size in *used. */
hs_status hs_pool_snapshot(hs_pool_t pool, void *host_dst, size_t cap, size_t *used);
hs_status hs_pool_restore(hs_pool_t pool, const void *host_src, size_t n);

/* Synchronises the pool's stream, returns the device error word and clears it. */
hs_status hs_pool_get_error(hs_pool_t pool, uint32_t *device_error_bits);

/* ---- hot path: no allocation, no host synchronisation, fixed launch shape
 *      for a given (B, K); capturable in a CUDA graph ------------------------ */

/* Resolves one decode step's top-K lists in one fused launch (混合 HiSparse 的
 * 技术实现, item 2; 融合内核与CUDA图兼容).
 *   d_req_ids   int32 [B]    distinct request ids
 *   d_topk_idx  int32 [B][K] token positions, -1 = padding; any order
 *   d_resolved  int32 [B][K] out: pool row id of each entry, -1 if unresolved
 *   d_gathered  [B][K][row_bytes] out: the rows, packed in list order (zeros
 *               for unresolved entries); 16-byte aligned. NULL: no gathered
 *               copy; the rows stay in the pool for hs_sparse_mla_decode to
 *               read in place (resolved ids only, misses still copied into
 *               their hot slots)
 *   d_gathered_scale float [B][K] out (FP8 pools with d_gathered; NULL for
 *               BF16 pools and whenever d_gathered is NULL)
 *   d_counts    int32 [B][3] out: entries resolved as (resident, hot, miss)
 * Per request, with clock c = previous clock + 1: an entry whose page is
 * resident resolves in place; one held in the hot buffer resolves to its slot
 * and gets stamp c; all hits are stamped before any miss is placed. Misses, in
 * ascending position, take the unprotected slots (stamp < c) with the smallest
 * (stamp, slot) keys; each miss row (and scale) is read from the pinned host
 * arena into its slot (and into d_gathered). A repeated missing position is
 * served once (first in list order). Requires 1 <= K <= min(max_topk, hot_rows). */
hs_status hs_resolve_topk(hs_pool_t pool, int32_t B, const int32_t *d_req_ids,
                          const int32_t *d_topk_idx, int32_t K, int32_t *d_resolved,
                          void *d_gathered, float *d_gathered_scale, int32_t *d_counts,
                          void *stream);

/* hs_resolve_topk for several top-K lists per request resolved against the
 * request's one hot state (推测性解码: each step's resolve plan is shared by the
 * request's speculative tokens). d_topk_idx [B][K] holds, per request, the
 * concatenation of its tokens' lists (K = tokens x per-token top-K; each token's
 * list holds distinct positions, lists may overlap). Results, layouts and
 * errors are those of hs_resolve_topk except for repeated positions: every
 * occurrence of a position resolves to the same row and counts in d_counts;
 * for a missing position the first occurrence in list order takes the LRU
 * slot and copies the row, the later ones share it (or are all rejected with
 * it). No HS_DEVERR_DUPLICATE is raised. Requires 1 <= K <= max_topk; distinct
 * missing positions beyond the free slots are rejected (HS_DEVERR_CAPACITY). */
hs_status hs_resolve_topk_union(hs_pool_t pool, int32_t B, const int32_t *d_req_ids,
                                const int32_t *d_topk_idx, int32_t K, int32_t *d_resolved,
                                void *d_gathered, float *d_gathered_scale, int32_t *d_counts,
                                void *stream);

/* Several sparse-MLA layers resolved in one launch ([A] 关键架构细节, 轻量级执行:
 * all sparse-MLA layers are launched at once, in the model stream's order).
 * Each layer has its own pool (rows, page table, hot buffers, LRU state); the
 * pools of a group share dtype, hot_rows and max_topk and live on the current
 * device. hs_layer_group_create copies the pools' table addresses to the
 * device once (synchronous); the pools must outlive the group, which owns
 * nothing else. */
hs_status hs_layer_group_create(const hs_pool_t *pools, int32_t L, hs_layer_group_t *out);
hs_status hs_layer_group_destroy(hs_layer_group_t group);

/* hs_resolve_topk for every layer of a group in one launch: one cluster per
 * (request, layer), each layer exactly as hs_resolve_topk would resolve it
 * (its own clock, LRU state and error word).
 *   d_req_ids [B] (the same requests in every layer); d_topk_idx and
 *   d_resolved [L][B][K]; d_gathered [L][B][K][row_bytes] or NULL;
 *   d_gathered_scale [L][B][K] (FP8 with gathered rows) or NULL;
 *   d_counts [L][B][3]. Requires 1 <= K <= min(max_topk, hot_rows). */
hs_status hs_resolve_topk_layers(hs_layer_group_t group, int32_t B, const int32_t *d_req_ids,
                                 const int32_t *d_topk_idx, int32_t K, int32_t *d_resolved,
                                 void *d_gathered, float *d_gathered_scale, int32_t *d_counts,
                                 void *stream);

/* Sparse MLA decode over the gathered rows: attention restricted to the K
 * selected latent rows (解决 KV 缓存内存压力; 稀疏MLA的核心思想). Query token t of request b sits at position L_b - T + t
 * (L_b = ctx_len of d_req_ids[b]) and attends to entry j iff d_resolved[b][j]
 * >= 0 and d_topk_idx[b][j] <= L_b - T + t.
 *   d_gathered / d_gathered_scale: as written by hs_resolve_topk; or both
 *           NULL to read each entry's row (and FP8 scale) in place from the
 *           pool by its d_resolved id (entries with id -1 read a zero row)
 *   d_q     bf16 [B][T][H][576]
 *   d_out   bf16 [B][T][H][512] = softmax(sm_scale * q.k_j) weighted sum of k_j[0:512]
 *   d_lse   float [B][T][H]      = ln sum_j exp(sm_scale * q.k_j); -inf if none valid
 *   d_workspace / ws_bytes: at least hs_decode_workspace_bytes(B, T, H, K)
 *   bytes of device memory, 256-byte aligned (may be NULL when that is 0).
 * Requires 1 <= T <= 32767, H*T <= 128*65535, B <= 65535 and K >= 1; q, gathered
 * and out 16-byte aligned. */
hs_status hs_sparse_mla_decode(hs_pool_t pool, int32_t B, int32_t T, int32_t H, int32_t K,
                               const void *d_q, const void *d_gathered,
                               const float *d_gathered_scale, const int32_t *d_resolved,
                               const int32_t *d_topk_idx, const int32_t *d_req_ids,
                               float sm_scale, void *d_out, float *d_lse, void *d_workspace,
                               size_t ws_bytes, void *stream);
size_t hs_decode_workspace_bytes(int32_t B, int32_t T, int32_t H, int32_t K);

/* hs_sparse_mla_decode with one top-K list per query token (the lists that
 * hs_resolve_topk_union resolved). List (b, t) of K entries is row b*T + t of
 * d_resolved / d_topk_idx ([B][T][K]) and of d_gathered ([B][T][K][row_bytes],
 * scales [B][T][K]) or, with both NULL, read in place from the pool. Query
 * token t of request b sits at position L_b - T + t and attends to entry j of
 * its own list iff d_resolved[b][t][j] >= 0 and d_topk_idx[b][t][j] <= L_b - T + t.
 * q, out and lse are laid out as in hs_sparse_mla_decode. The workspace needs
 * hs_decode_workspace_bytes(B * T, 1, H, K) bytes. Requires B * T <= 65535,
 * H <= 128*65535; other requirements as hs_sparse_mla_decode. */
hs_status hs_sparse_mla_decode_per_token(hs_pool_t pool, int32_t B, int32_t T, int32_t H,
                                         int32_t K, const void *d_q, const void *d_gathered,
                                         const float *d_gathered_scale, const int32_t *d_resolved,
                                         const int32_t *d_topk_idx, const int32_t *d_req_ids,
                                         float sm_scale, void *d_out, float *d_lse,
                                         void *d_workspace, size_t ws_bytes, void *stream);

/* hs_sparse_mla_decode without a caller-provided workspace. This entry point
 * has no counterpart in the pages; it exists for callers that cannot allocate
 * device memory: a host engine that has reserved the device's memory for its
 * own KV pool and passes this library only tensors it already owns, or a C
 * plugin that receives device pointers but has no allocator to call.
 * The split-KV partials go to one array of HS_STATIC_DECODE_WS_BYTES bytes
 * that lives in this library's device memory; every GPU that loads the
 * library holds it until the process exits. The function itself allocates
 * nothing. Arguments, layouts and results are those of hs_sparse_mla_decode.
 *  - Shapes whose workspace (hs_decode_workspace_bytes) exceeds
 *    HS_STATIC_DECODE_WS_BYTES return HS_ERR_CAPACITY and launch nothing.
 *  - The first call on a device looks up that device's address of the array
 *    (with that device current); make that first call before any stream
 *    capture on the device.
 *  - All calls share the one array and it keeps the last call's contents;
 *    each call writes every entry it later reads, so nothing needs clearing.
 *    Calls whose kernels overlap on the GPU (different streams without
 *    ordering) race on the array: order them on one stream. */
#define HS_STATIC_DECODE_WS_BYTES (24u << 20)
hs_status hs_sparse_mla_decode_static_ws(hs_pool_t pool, int32_t B, int32_t T, int32_t H,
                                         int32_t K, const void *d_q, const void *d_gathered,
                                         const float *d_gathered_scale, const int32_t *d_resolved,
                                         const int32_t *d_topk_idx, const int32_t *d_req_ids,
                                         float sm_scale, void *d_out, float *d_lse, void *stream);

/* ---- residency transitions on the device -------------------------------- */

/* Active copy ([A] 混合 HiSparse 的技术实现 item 1; 关键架构细节, 主动复制): for each
 * of n triples (d_req[i], d_page[i], d_host_block[i]) the page's 64 rows (and
 * FP8 scales) are copied from its GPU block into that block of the pinned host
 * arena, then the page table records the host copy; the page stays resident
 * and keeps being served from the GPU. One launch, asynchronous on `stream`;
 * it touches only the host half of page-table entries, which the resolve reads
 * for non-resident pages only, so it may run on a side stream next to the
 * decode path. A triple whose request, page or host block is out of range, or
 * whose page has no GPU block, is skipped and sets HS_DEVERR_BAD_PAGE. The
 * caller owns host-block allocation. */
hs_status hs_active_copy(hs_pool_t pool, int32_t n, const int32_t *d_req, const int32_t *d_page,
                         const int32_t *d_host_block, void *stream);

/* Demotion under pressure ([A] 混合 HiSparse 的技术实现 item 2; [B] 分级内存的运作机制):
 * request d_req[i] keeps its last d_keep_tail[i] tokens on the GPU and releases
 * its coldest pages, read as its oldest: every page p with (p+1)*64 <=
 * ctx_len - keep_tail that is resident and has a host copy loses its GPU
 * block. Pages without a host copy stay resident. The freed GPU blocks go to
 * d_freed[i][0 .. d_n_freed[i]) in ascending page order (d_freed is
 * [n][max_pages] int32, d_n_freed [n] int32) for the caller's allocator. One
 * launch, asynchronous on `stream`; order it with the resolve calls of the
 * same requests. A bad request id sets HS_DEVERR_BAD_REQUEST, a negative tail
 * HS_DEVERR_BAD_PAGE (that request frees nothing). */
hs_status hs_demote_cold_pages(hs_pool_t pool, int32_t n, const int32_t *d_req,
                               const int32_t *d_keep_tail, int32_t *d_freed, int32_t *d_n_freed,
                               void *stream);

/* Failure-detection check: launches one device wait on a barrier phase that
 * nothing completes, bounded by limit_us (1 .. 2,000,000) exactly like the
 * decode pipeline's waits. The wait gives up, sets HS_DEVERR_TIMEOUT in the
 * pool's device error word (read it with hs_pool_get_error) and the kernel
 * returns, leaving the context usable. Asynchronous on `stream`. */
hs_status hs_pool_check_bounded_wait(hs_pool_t pool, uint32_t limit_us, void *stream);

/* Human-readable name of a status. */
const char *hs_status_string(hs_status s);

#ifdef __cplusplus
}
#endif
#endif /* HS_H */
