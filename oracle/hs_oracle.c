/*
 * hs_oracle.c -- plain, slow CPU oracle for the tiered sparse-MLA decode path.
 *
 * TEST INFRASTRUCTURE. Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg load this library. It shares no code, header or
 * constant table with the CUDA path; both sides read only the seeded inputs.
 *
 * What it follows ("vLLM GLM 5.3 优化：混合 HiSparse 卸载", section 混合 HiSparse
 * 的技术实现, item 2, and section 关键架构细节; "vLLM Hybrid HiSparse：稀疏MLA破解
 * 长上下文显存瓶颈", sections 稀疏MLA的核心思想 and 融合内核与CUDA图兼容):
 *
 *   resolve, per request and decode step, for every selected token row:
 *     - a row whose page is GPU-resident is read in place;
 *     - a row held in the request's hot buffer is read and its LRU entry is
 *       refreshed;
 *     - any other row is copied, on its own, from pinned host memory into the
 *       least recently used hot-buffer slot.
 *   The pages leave the order of these actions open. The readings taken here:
 *     (1) all hits are stamped with the step's clock first; then the misses,
 *         in ascending token position, each take the slot with the smallest
 *         (stamp, slot) key among slots whose stamp is older than this step's
 *         clock, so a row used in this step is never evicted in this step;
 *     (2) residency is checked before the hot buffer;
 *     (3) a token position repeated in one list as a miss is served once (its
 *         first occurrence in list order); later repeats are rejected;
 *     (4) out-of-range positions, pages with neither a GPU block nor a host
 *         copy, and unknown request ids are rejected with an error bit and an
 *         unresolved (-1) entry.
 *
 *   attention (sparse MLA decode), per query row (request, token t, head h):
 *     s_j = sm_scale * <q, k_j> over the 576-wide latent row k_j of every
 *     selected row j that resolved and whose position is <= L - T + t;
 *     out = sum_j softmax(s)_j * k_j[0:512];  lse = ln sum_j exp(s_j).
 *   Computed in float64 after exact dequantisation (BF16 widened, FP8 e4m3
 *   decoded from the OCP 8-bit floating point format and multiplied by the
 *   row's fp32 scale).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* device-error bits, as the C ABI of the CUDA path specifies them */
#define OR_ERR_INDEX_RANGE 1u
#define OR_ERR_DUPLICATE   2u
#define OR_ERR_NO_HOST     4u
#define OR_ERR_BAD_REQUEST 8u
#define OR_ERR_CAPACITY    16u

#define OR_PAGE 64
#define OR_DIM 576
#define OR_NOPE 512

typedef struct {
    int32_t max_req, max_pages, max_ctx, hot_rows, row_bytes, fp8;
    const int32_t *page_gpu;   /* [max_req][max_pages], -1 = not resident */
    const int32_t *page_host;  /* [max_req][max_pages], -1 = no host copy  */
    const int32_t *hot_blocks; /* [max_req][hot_rows / 64]                 */
    int32_t *tag;              /* [max_req][hot_rows], -1 = empty          */
    int32_t *stamp;            /* [max_req][hot_rows], -1 = never used     */
    int32_t *pos_to_slot;      /* [max_req][max_ctx], -1 = not in hot buf  */
    int32_t *clock;            /* [max_req]                                */
    const int32_t *ctx_len;    /* [max_req]                                */
    uint8_t *pool_rows;        /* [n_gpu_blocks*64][row_bytes]             */
    float *pool_scales;        /* [n_gpu_blocks*64] or NULL (BF16)         */
    const uint8_t *host_rows;  /* [n_host_blocks*64][row_bytes]            */
    const float *host_scales;  /* [n_host_blocks*64] or NULL               */
} or_state;

/* ------------------------------------------------------------ number formats */
double or_bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP FP8 E4M3 ("fn" variant): 1 sign bit, 4 exponent bits with bias 7,
 * 3 mantissa bits; exponent 0 is subnormal; S.1111.111 is NaN; no infinities. */
double or_e4m3_to_double(uint8_t v)
{
    int sign = (v >> 7) & 1, e = (v >> 3) & 15, m = v & 7;
    double x;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        x = ldexp((double)m, -9);          /* m/8 * 2^(1-7) */
    else
        x = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
    return sign ? -x : x;
}

/* ------------------------------------------------------------ resolve */
typedef struct { int32_t p, j; } or_miss;

static int or_cmp_miss(const void *a, const void *b)
{
    const or_miss *x = a, *y = b;
    if (x->p != y->p) return x->p < y->p ? -1 : 1;
    return x->j < y->j ? -1 : (x->j > y->j);
}

typedef struct { int32_t stamp, slot; } or_key;

static int or_cmp_key(const void *a, const void *b)
{
    const or_key *x = a, *y = b;
    if (x->stamp != y->stamp) return x->stamp < y->stamp ? -1 : 1;
    return x->slot < y->slot ? -1 : (x->slot > y->slot);
}

static int64_t or_hot_row(const or_state *S, int32_t r, int32_t slot)
{
    int32_t per_req = (S->hot_rows + OR_PAGE - 1) / OR_PAGE; /* blocks leased per request */
    int32_t blk = S->hot_blocks[(int64_t)r * per_req + slot / OR_PAGE];
    return (int64_t)blk * OR_PAGE + slot % OR_PAGE;
}

/* Resolve one request's list. Bit 0 of `formulation` picks the LRU rule's
 * form: 0, each miss scans for the argmin (stamp, slot) unprotected slot; 1,
 * the unprotected keys are sorted once and the i-th miss takes the i-th key.
 * Bit 1 set: the list is the union of several lists sharing one hot state
 * (the MTP draft tokens' own lists, [A] 与 vLLM 栈的集成, speculative
 * decoding), so a missing position repeated in it is served once and every
 * occurrence resolves to that row (or is rejected with it); without bit 1 the
 * repeats are rejected as errors. */
static uint32_t or_resolve_one(const or_state *S, int32_t r, const int32_t *topk, int32_t K,
                               int formulation, int32_t *resolved, uint8_t *gathered,
                               float *gathered_scale, int32_t *counts)
{
    const int32_t rb = S->row_bytes;
    uint32_t err = 0;
    counts[0] = counts[1] = counts[2] = 0;
    for (int32_t j = 0; j < K; ++j) resolved[j] = -1;
    if (r < 0 || r >= S->max_req) {
        memset(gathered, 0, (size_t)K * rb);
        if (gathered_scale) memset(gathered_scale, 0, sizeof(float) * K);
        return OR_ERR_BAD_REQUEST;
    }
    const int32_t C = S->hot_rows;
    int32_t *tag = S->tag + (int64_t)r * C;
    int32_t *stamp = S->stamp + (int64_t)r * C;
    int32_t *p2s = S->pos_to_slot + (int64_t)r * S->max_ctx;
    const int32_t *pg_gpu = S->page_gpu + (int64_t)r * S->max_pages;
    const int32_t *pg_host = S->page_host + (int64_t)r * S->max_pages;
    const int32_t L = S->ctx_len[r];
    const int32_t c = ++S->clock[r];

    /* phase 1: resident rows, hot rows (stamped now), misses collected */
    or_miss *miss = malloc(sizeof(or_miss) * (K > 0 ? K : 1));
    int32_t n_miss = 0;
    for (int32_t j = 0; j < K; ++j) {
        int32_t p = topk[j];
        if (p == -1) continue;
        if (p < 0 || p >= L || p >= S->max_ctx) { err |= OR_ERR_INDEX_RANGE; continue; }
        int32_t g = pg_gpu[p / OR_PAGE];
        if (g >= 0) {
            resolved[j] = (int32_t)((int64_t)g * OR_PAGE + p % OR_PAGE);
            counts[0]++;
            continue;
        }
        int32_t s = p2s[p];
        if (s >= 0) {
            resolved[j] = (int32_t)or_hot_row(S, r, s);
            stamp[s] = c;
            counts[1]++;
            continue;
        }
        if (pg_host[p / OR_PAGE] < 0) { err |= OR_ERR_NO_HOST; continue; }
        miss[n_miss].p = p;
        miss[n_miss].j = j;
        n_miss++;
    }

    /* phase 2: misses in ascending position; repeats after the first rejected */
    qsort(miss, n_miss, sizeof(or_miss), or_cmp_miss);
    or_key *keys = NULL;
    int32_t n_keys = 0, next_key = 0;
    if (formulation & 1) {
        keys = malloc(sizeof(or_key) * C);
        for (int32_t s = 0; s < C; ++s)
            if (stamp[s] < c) { keys[n_keys].stamp = stamp[s]; keys[n_keys].slot = s; n_keys++; }
        qsort(keys, n_keys, sizeof(or_key), or_cmp_key);
    }
    const int uni = (formulation & 2) != 0;
    int32_t last_row = -1; /* row the previous distinct missing position got (-1 = rejected) */
    for (int32_t i = 0; i < n_miss; ++i) {
        int32_t p = miss[i].p, j = miss[i].j;
        if (i > 0 && miss[i - 1].p == p) {
            if (!uni) { err |= OR_ERR_DUPLICATE; continue; }
            if (last_row >= 0) { resolved[j] = last_row; counts[2]++; }
            continue;
        }
        last_row = -1;
        int32_t v = -1;
        if ((formulation & 1) == 0) {
            for (int32_t s = 0; s < C; ++s) {
                if (stamp[s] >= c) continue;
                if (v < 0 || stamp[s] < stamp[v]) v = s; /* ties keep the lower slot */
            }
        } else if (next_key < n_keys) {
            v = keys[next_key++].slot;
        }
        if (v < 0) { err |= OR_ERR_CAPACITY; continue; }
        if (tag[v] >= 0) p2s[tag[v]] = -1;
        tag[v] = p;
        stamp[v] = c;
        p2s[p] = v;
        /* the single-row copy from pinned host memory into the slot */
        int64_t hrow = (int64_t)pg_host[p / OR_PAGE] * OR_PAGE + p % OR_PAGE;
        int64_t drow = or_hot_row(S, r, v);
        memcpy(S->pool_rows + drow * rb, S->host_rows + hrow * rb, rb);
        if (S->pool_scales) S->pool_scales[drow] = S->host_scales[hrow];
        resolved[j] = (int32_t)drow;
        last_row = (int32_t)drow;
        counts[2]++;
    }
    free(keys);
    free(miss);

    /* gathered row j = the pool row that resolved[j] names after this step */
    for (int32_t j = 0; j < K; ++j) {
        uint8_t *dst = gathered + (int64_t)j * rb;
        if (resolved[j] >= 0) {
            memcpy(dst, S->pool_rows + (int64_t)resolved[j] * rb, rb);
            if (gathered_scale) gathered_scale[j] = S->pool_scales[resolved[j]];
        } else {
            memset(dst, 0, rb);
            if (gathered_scale) gathered_scale[j] = 0.0f;
        }
    }
    return err;
}

uint32_t or_resolve(const or_state *S, int32_t B, const int32_t *req_ids, const int32_t *topk,
                    int32_t K, int32_t formulation, int32_t *resolved, uint8_t *gathered,
                    float *gathered_scale, int32_t *counts, int32_t nthreads)
{
    uint32_t err = 0;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1) reduction(| : err)
#endif
    for (int32_t b = 0; b < B; ++b) {
        err |= or_resolve_one(S, req_ids[b], topk + (int64_t)b * K, K, formulation,
                              resolved + (int64_t)b * K,
                              gathered + (int64_t)b * K * S->row_bytes,
                              gathered_scale ? gathered_scale + (int64_t)b * K : NULL,
                              counts + 3 * b);
    }
    return err;
}

/* ------------------------------------------------------------ attention */
/* Rows (b, t, h) listed in `sel` (n_sel triples; all B*T*H rows in order when
 * sel is NULL). out: [n][512] float64, lse: [n] float64. */
void or_sparse_mla_decode(int32_t B, int32_t T, int32_t H, int32_t K, int32_t fp8,
                          const uint16_t *q, const uint8_t *gathered, const float *gscale,
                          const int32_t *resolved, const int32_t *topk, const int32_t *L_b,
                          double sm_scale, int32_t n_sel, const int32_t *sel,
                          double *out, double *lse, int32_t nthreads)
{
    const int64_t rb = fp8 ? OR_DIM : 2 * OR_DIM;
    int32_t n = sel ? n_sel : B * T * H;
#ifdef _OPENMP
    if (nthreads < 1) nthreads = 1;
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1)
#endif
    for (int32_t i = 0; i < n; ++i) {
        int32_t b, t, h;
        if (sel) { b = sel[3 * i]; t = sel[3 * i + 1]; h = sel[3 * i + 2]; }
        else { b = i / (T * H); t = (i / H) % T; h = i % H; }
        const uint16_t *qr = q + (((int64_t)b * T + t) * H + h) * OR_DIM;
        double qd[OR_DIM];
        for (int d = 0; d < OR_DIM; ++d) qd[d] = or_bf16_to_double(qr[d]);
        const int32_t pos = L_b[b] - T + t;
        double *s = malloc(sizeof(double) * (K > 0 ? K : 1));
        double m = -INFINITY;
        int32_t n_valid = 0;
        for (int32_t j = 0; j < K; ++j) {
            int64_t bj = (int64_t)b * K + j;
            s[j] = NAN;
            if (resolved[bj] < 0 || topk[bj] > pos) continue;
            const uint8_t *row = gathered + bj * rb;
            double acc = 0.0;
            for (int d = 0; d < OR_DIM; ++d) {
                double kd;
                if (fp8) kd = or_e4m3_to_double(row[d]) * (double)gscale[bj];
                else { uint16_t hb; memcpy(&hb, row + 2 * d, 2); kd = or_bf16_to_double(hb); }
                acc += qd[d] * kd;
            }
            s[j] = sm_scale * acc;
            if (s[j] > m) m = s[j];
            n_valid++;
        }
        double *o = out + (int64_t)i * OR_NOPE;
        for (int d = 0; d < OR_NOPE; ++d) o[d] = 0.0;
        if (n_valid == 0) { lse[i] = -INFINITY; free(s); continue; }
        double l = 0.0;
        for (int32_t j = 0; j < K; ++j)
            if (!isnan(s[j])) l += exp(s[j] - m);
        for (int32_t j = 0; j < K; ++j) {
            if (isnan(s[j])) continue;
            int64_t bj = (int64_t)b * K + j;
            double w = exp(s[j] - m) / l;
            const uint8_t *row = gathered + bj * rb;
            for (int d = 0; d < OR_NOPE; ++d) {
                double vd;
                if (fp8) vd = or_e4m3_to_double(row[d]) * (double)gscale[bj];
                else { uint16_t hb; memcpy(&hb, row + 2 * d, 2); vd = or_bf16_to_double(hb); }
                o[d] += w * vd;
            }
        }
        lse[i] = m + log(l);
        free(s);
    }
}

int32_t or_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
