// hs_resolve.cu -- the fused top-K resolve kernel.
//
// One launch resolves a decode step's top-K lists against the tiered cache
// ("vLLM GLM 5.3 优化：混合 HiSparse 卸载", section 混合 HiSparse 的技术实现, item 2;
// "vLLM Hybrid HiSparse：稀疏MLA破解长上下文显存瓶颈", section 融合内核与CUDA图兼容):
// a row in a resident page is read in place, a row in the request's hot buffer
// is read and its LRU entry refreshed, and a missing row is copied by itself
// from pinned host memory into the least recently used hot slot. The launch
// shape depends only on (B, K), so the kernel replays inside a CUDA graph; the
// LRU clock lives in device memory and advances on every replay.
//
// Orders the pages leave open (same readings as the oracle): hits are stamped
// before any miss is placed; misses in ascending position take the unprotected
// slots (stamp < clock) with the smallest (stamp, slot) keys; residency is
// checked before the hot buffer; a missing position repeated in one list is
// served once (first in list order). When a request's list is the union of its
// speculative tokens' lists (推测性解码 shares the request's hot state), every
// repeat of a missing position resolves to the row its first occurrence took;
// only the first occurrence updates the LRU state and copies the row.
//
// Design (GB300): one thread-block cluster of G CTAs per request (and layer,
// when a launch covers several layers' pools). Rank 0 keeps the request's LRU
// bookkeeping; ranks 1..G-1 ("workers") own K/(G-1) list entries each.
//   start    cluster barrier (every CTA's shared memory is live);
//   phase 1  workers classify their entries (page table, then pos_to_slot),
//            stamp their hot hits, and push each miss's (position, list index)
//            key into rank 0's key array (slots taken by one remote atomic per
//            warp). In a union the first occurrence to mark pos_to_slot is the
//            position's reader and the only one to push a key; -> barrier A
//   rank 0   sorts the keys (bitonic, shared memory or registers), ranks the
//            distinct positions, stages the persistent LRU order (slots kept
//            sorted by (stamp, slot), so the i-th unprotected entry is the
//            i-th victim) in shared memory, places the misses (tag / stamp /
//            pos_to_slot / LRU order) and writes each miss's slot into its
//            owner's shared memory;
//   phase 2  meanwhile workers copy every row whose gathered position is known
//            -- resident and hot rows from the pool, miss rows they read from
//            the device-mapped pinned host arena -- into the gathered buffer
//            (rows kept in the pool: the miss rows into shared memory), so the
//            host-link reads overlap rank 0's bookkeeping; -> barrier B
//   phase 3  a union's other occurrences take their reader's slot (through
//            distributed shared memory; -> barrier C before any CTA exits);
//            readers copy each placed miss row into its hot slot and rejected
//            entries get zeros.
// Barriers are hardware cluster barriers: no spin loops.
#include <algorithm>
#include <cstdint>
#include <new>
#include <vector>

#include "hs_internal.cuh"

namespace {

constexpr int NT = 512;       // threads per CTA
constexpr int UNROLL = 4;     // 16-byte vectors in flight per thread and round
constexpr int UNROLL_H = 8;   // the same for loops that read rows over the host link
constexpr int KIND_NONE = 0, KIND_RES = 1, KIND_HOT = 2, KIND_MISS = 3;

// Dynamic shared memory layout (bytes), identical in every CTA. Rank 0 holds
// no list entries, so its part overlaps the workers' part.
struct Smem {
    int chunk, kpad, K, C;
    // misc: [0] local misses, [1] resident, [2] hot, [3] staged rows (workers)
    //       or placed misses (rank 0), [4] keys received (rank 0), [8..9]
    //       totals, [20..52) warp scan scratch, [64 + 4g + 0..2] {misses,
    //       resident, hot} of worker g (rank 0)
    __host__ __device__ size_t off_misc() const { return 0; }
    // worker part
    __host__ __device__ size_t off_src() const { return 512; }
    __host__ __device__ size_t off_hrow() const { return off_src() + 4 * (size_t)chunk; }
    __host__ __device__ size_t off_kind() const { return off_hrow() + 4 * (size_t)chunk; }
    __host__ __device__ size_t off_mj() const { return off_kind() + 4 * (size_t)chunk; }
    // claim: for a miss, the request-level list index of the occurrence that
    // reads its row from the host (itself, unless a union repeats the position)
    __host__ __device__ size_t off_claim() const { return off_mj() + 4 * (size_t)chunk; }
    // rows read from the host wait here for their slot (rows kept in the pool)
    __host__ __device__ size_t off_stage() const {
        return (off_claim() + 4 * (size_t)chunk + 15) & ~size_t(15);
    }
    // rank-0 part: miss keys (position << 32 | rank+1 << 13 | list index), the
    // victims (one per distinct miss, at most one per slot), the LRU order and
    // each slot's protection
    __host__ __device__ size_t off_keys() const { return 512; }
    __host__ __device__ size_t off_victim() const { return off_keys() + 8 * (size_t)kpad; }
    __host__ __device__ size_t off_lru() const { return off_victim() + 4 * (size_t)(K < C ? K : C); }
    __host__ __device__ size_t off_prot() const { return off_lru() + 4 * (size_t)C; }
    // rank 0: the counts of block_rank8
    __host__ __device__ size_t off_rank() const { return (off_prot() + (size_t)C + 15) & ~size_t(15); }
    __host__ __device__ size_t total() const {
        const size_t r0 = off_rank() + 4 * (size_t)(8 * NT / 32 + 1);
        return r0 > off_stage() ? r0 : off_stage();
    }
};

__host__ __device__ inline int next_pow2(int x) {
    int p = 1;
    while (p < x) p <<= 1;
    return p;
}

// Ranks, in block order, of up to 8 * NT flags: flag (it, t) stands for
// element it * NT + t, and rank[it] counts the set flags before it. Each warp
// ballots its 8 rows of flags, one warp scans the 8 * NT / 32 counts (four per
// lane), so 8 * NT elements take two __syncthreads instead of one block-wide
// scan per NT. Returns the number of set flags; s_cnt holds 8 * NT / 32 + 1
// ints and may be reused after the caller's next __syncthreads.
__device__ __forceinline__ int block_rank8(const bool (&f)[8], int (&rank)[8], int *s_cnt, int tid) {
    constexpr int NW = NT / 32;
    static_assert(8 * NW == 4 * 32, "one warp scans the counts, four per lane");
    const int lane = tid & 31, w = tid >> 5;
    unsigned bal[8];
#pragma unroll
    for (int it = 0; it < 8; ++it) bal[it] = __ballot_sync(0xffffffffu, f[it]);
    if (lane == 0)
#pragma unroll
        for (int it = 0; it < 8; ++it) s_cnt[it * NW + w] = __popc(bal[it]);
    __syncthreads();
    if (w == 0) {
        int v[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = s_cnt[4 * lane + e];
        const int t4 = (v[0] + v[1]) + (v[2] + v[3]);
        int incl = t4;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        int run = incl - t4;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            s_cnt[4 * lane + e] = run;
            run += v[e];
        }
        if (lane == 31) s_cnt[8 * NW] = incl;
    }
    __syncthreads();
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll
    for (int it = 0; it < 8; ++it) rank[it] = s_cnt[it * NW + w] + __popc(bal[it] & lt);
    return s_cnt[8 * NW];
}

__device__ __forceinline__ void dsmem_st64(uint32_t a, unsigned long long v) {
    asm volatile("st.shared::cluster.u64 [%0], %1;\n" ::"r"(a), "l"(v) : "memory");
}

__device__ __forceinline__ int dsmem_atom_add(uint32_t a, int v) {
    int r;
    asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;\n" : "=r"(r) : "r"(a), "r"(v) : "memory");
    return r;
}

__device__ __forceinline__ void st_shared_v4(void *p, uint4 v) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(const void *p) {
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(p));
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a)
                 : "memory");
    return v;
}

__device__ __forceinline__ uint32_t dyn_smem_bytes() {
    uint32_t n;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(n));
    return n;
}

// ---------------------------------------------------------------- key sort
// Bitonic sort of up to 4096 64-bit keys held in registers, 8 per thread
// (element e = 8t + r of thread t). Strides below 8 pair registers of one
// thread, strides 8..128 pair threads of one warp (shuffles), larger strides
// go through shared memory. Element e lives in shared memory at swz(e), which
// spreads a warp's accesses over the banks.
__device__ __forceinline__ int swz8(int e) { return (e & ~7) | ((e ^ (e >> 3)) & 7); }

__device__ __forceinline__ void cmpx(unsigned long long &a, unsigned long long &b, bool asc) {
    const bool sw = (a > b) == asc;
    const unsigned long long lo = sw ? b : a, hi = sw ? a : b;
    a = lo;
    b = hi;
}

template <int JJ>
__device__ __forceinline__ void reg_stage(unsigned long long (&x)[8], int t, int k) {
#pragma unroll
    for (int r = 0; r < 8; ++r)
        if ((r & JJ) == 0) cmpx(x[r], x[r | JJ], ((t * 8 + r) & k) == 0);
}

// s: the keys at swz(e), e < n2 (a power of two, 8 <= n2 <= 8 * NT); sorted in place.
__device__ __forceinline__ void sort_keys_reg(unsigned long long *s, int n2, int tid) {
    const int T = n2 >> 3;  // threads holding keys
    const bool act = tid < T;
    unsigned long long x[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) x[r] = act ? s[swz8(tid * 8 + r)] : ~0ull;
    for (int k = 2; k <= n2; k <<= 1) {
        for (int jj = k >> 1; jj > 0; jj >>= 1) {
            if (jj >= 256) {
                __syncthreads();  // previous readers of s are done
                if (act) {
#pragma unroll
                    for (int r = 0; r < 8; ++r) s[swz8(tid * 8 + r)] = x[r];
                }
                __syncthreads();
                if (act) {
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        const int e = tid * 8 + r;
                        const unsigned long long y = s[swz8(e ^ jj)];
                        const bool keep_min = ((e & jj) == 0) == ((e & k) == 0);
                        x[r] = keep_min ? (x[r] < y ? x[r] : y) : (x[r] > y ? x[r] : y);
                    }
                }
            } else if (jj >= 8) {
                const int m = jj >> 3;  // partner lane offset (xor)
#pragma unroll
                for (int r = 0; r < 8; ++r) {
                    const int e = tid * 8 + r;
                    const unsigned lo = __shfl_xor_sync(0xffffffffu, (unsigned)x[r], m);
                    const unsigned hi = __shfl_xor_sync(0xffffffffu, (unsigned)(x[r] >> 32), m);
                    const unsigned long long y = ((unsigned long long)hi << 32) | lo;
                    const bool keep_min = ((e & jj) == 0) == ((e & k) == 0);
                    x[r] = keep_min ? (x[r] < y ? x[r] : y) : (x[r] > y ? x[r] : y);
                }
            } else if (jj == 4) {
                reg_stage<4>(x, tid, k);
            } else if (jj == 2) {
                reg_stage<2>(x, tid, k);
            } else {
                reg_stage<1>(x, tid, k);
            }
        }
    }
    __syncthreads();
    if (act) {
#pragma unroll
        for (int r = 0; r < 8; ++r) s[swz8(tid * 8 + r)] = x[r];
    }
    __syncthreads();
}

// The same sort for any power-of-two count, by a shared-memory bitonic
// network, keys stored at e. A pair of a stage with stride jj <= 32 stays
// inside the 64 keys of its 32-aligned group of pairs, which one warp owns
// across such stages: those stages sync the warp only.
__device__ __forceinline__ void sort_keys_smem(unsigned long long *s, int n2, int tid) {
    for (int k = 2; k <= n2; k <<= 1) {
        for (int jj = k >> 1; jj > 0; jj >>= 1) {
            for (int i = tid; i < (n2 >> 1); i += NT) {
                const int lo = ((i & ~(jj - 1)) << 1) | (i & (jj - 1)), hi = lo + jj;
                const unsigned long long a = s[lo], b = s[hi];
                if ((a > b) == ((lo & k) == 0)) {
                    s[lo] = b;
                    s[hi] = a;
                }
            }
            const int next = jj > 1 ? jj >> 1 : k;  // stride of the next stage
            if (jj >= 64 || next >= 64)
                __syncthreads();
            else
                __syncwarp();
        }
    }
    __syncthreads();
}

// Dynamic shared memory of a launch: the layout; with rows kept in the pool,
// grown (while two CTAs still fit on an SM) so that a worker can stage every
// row of its share of the list.
constexpr size_t kStageSmemCap = 110 * 1024;

// BIG: lists longer than 2048 entries (up to 4096 misses sort in registers).
// Shorter lists use the kernel without that path, which holds fewer registers.
// PT: the pool as a kernel parameter (hs::DevPool, one layer) or as a
// reference into device memory (const hs::DevPool &, a layer of a group).
template <int RB, bool BIG, typename PT>
__device__ __forceinline__ void resolve_body(PT P, const int32_t *__restrict__ req_ids,
                                             const int32_t *__restrict__ topk, int K, int chunk,
                                             int G, int32_t *__restrict__ resolved,
                                             uint8_t *__restrict__ gathered,
                                             float *__restrict__ gscale,
                                             int32_t *__restrict__ counts, int uni) {
    constexpr int V = RB / 16;  // 16-byte vectors per row
    // the step's decode may be scheduled as soon as every CTA of this grid runs
    // (it waits for this grid to complete before reading what it wrote)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ __align__(16) unsigned char smem[];
    const int W = G - 1;
    const Smem L{chunk, max(8, next_pow2(K)), K, P.C};
    int32_t *s_src = reinterpret_cast<int32_t *>(smem + L.off_src());
    int32_t *s_hrow = reinterpret_cast<int32_t *>(smem + L.off_hrow());
    int32_t *s_kind = reinterpret_cast<int32_t *>(smem + L.off_kind());
    int32_t *s_mj = reinterpret_cast<int32_t *>(smem + L.off_mj());
    int32_t *s_claim = reinterpret_cast<int32_t *>(smem + L.off_claim());
    int32_t *s_misc = reinterpret_cast<int32_t *>(smem + L.off_misc());
    int32_t *s_warp = s_misc + 20;
    int32_t *s_wcnt = s_misc + 64;  // [G][4], filled by the workers (rank 0 only)
    unsigned long long *s_keys = reinterpret_cast<unsigned long long *>(smem + L.off_keys());
    int32_t *s_victim = reinterpret_cast<int32_t *>(smem + L.off_victim());
    int32_t *s_lru = reinterpret_cast<int32_t *>(smem + L.off_lru());
    uint8_t *s_prot = smem + L.off_prot();
    int32_t *s_rank = reinterpret_cast<int32_t *>(smem + L.off_rank());
    // workers: the end of their shared memory stages the miss rows they read
    // from the host (rows beyond its capacity are read directly)
    uint8_t *s_stage = smem + L.off_stage();
    const int ncap = static_cast<int>((dyn_smem_bytes() - L.off_stage()) / RB);

    const int tid = threadIdx.x;
    const int g = static_cast<int>(hs::cluster_ctarank());
    const int bi = blockIdx.y;
    const int j0 = (g - 1) * chunk;  // first list entry of a worker
    const int nloc = g == 0 ? 0 : max(0, min(K, j0 + chunk) - j0);
    const size_t row0 = (size_t)bi * K + (g == 0 ? 0 : j0);  // first gathered row of this CTA
    // a worker's first list entry is loaded before anything else: its latency
    // overlaps the request's loads and the cluster barrier below
    const int p_first = tid < nloc ? topk[row0 + tid] : -1;
    const int r = req_ids[bi];
    const bool fp8 = P.scales != nullptr;
    const bool gath = gathered != nullptr;  // else rows are read in place by attention

    if (r < 0 || r >= P.max_req) {
        // the whole cluster takes this branch (same request), so no barrier waits
        for (int l = tid; l < nloc; l += NT) {
            resolved[row0 + l] = -1;
            if (gath && fp8) gscale[row0 + l] = 0.f;
        }
        if (gath)
            for (int i = tid; i < nloc * V; i += NT)
                hs::st_v4(gathered + row0 * RB + (size_t)i * 16, make_uint4(0, 0, 0, 0));
        if (g == 0 && tid < 3) counts[bi * 3 + tid] = 0;
        if (g == 0 && tid == 0) atomicOr(P.err, HS_DEVERR_BAD_REQUEST);
        return;
    }

    const int C = P.C;
    const int c = P.clock[r] + 1;  // this step's clock (rank 0 stores it after barrier A)
    const int Lr = P.ctx[r];
    const int2 *page = P.page + (size_t)r * P.max_pages;
    const int32_t *hblk = P.hot_blocks + (size_t)r * P.HB;
    int32_t *tag = P.tag + (size_t)r * C;
    int32_t *stamp = P.stamp + (size_t)r * C;
    int32_t *lru = P.lru + (size_t)r * C;
    int32_t *p2s = P.p2s + (size_t)r * P.max_ctx;
    // the first entry's page-table entry, also before the barrier
    const int2 e_first = (p_first >= 0 && p_first < P.max_ctx) ? page[p_first >> 6] : make_int2(-1, -1);

    if (tid == 0) s_misc[0] = s_misc[1] = s_misc[2] = s_misc[3] = s_misc[4] = 0;
    // every CTA of the cluster is running (and has set up its shared memory)
    // before any distributed-shared-memory store below; rank 0 releases its
    // counters, a worker publishes nothing here, so its arrive does not wait
    // for the loads above
    __syncthreads();
    if (g == 0)
        hs::cluster_arrive();
    else
        asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
    hs::cluster_wait();

    uint32_t err = 0;
    if (g != 0) {
        // ------------------------------------------------------------ phase 1
        // keys go straight into rank 0's key array, at slots taken (one remote
        // atomic per warp) from its counter
        const uint32_t keys0 = hs::dsmem_map(s_keys, 0);
        const uint32_t nkeys0 = hs::dsmem_map(&s_misc[4], 0);
        const int lane = tid & 31;
        int n_res = 0, n_hot = 0;
        for (int lb = 0; lb < nloc; lb += NT) {  // warp-uniform trip count
            const int l = lb + tid;
            const int p = lb == 0 ? p_first : (l < nloc ? topk[row0 + l] : -1);
            int kind = KIND_NONE, src = -1, hrow = -1;
            if (l >= nloc || p == -1) {
            } else if (p < 0 || p >= Lr || p >= P.max_ctx) {
                err |= HS_DEVERR_INDEX_RANGE;
            } else {
                const int2 e = lb == 0 ? e_first : page[p >> 6];
                if (e.x >= 0) {
                    kind = KIND_RES;
                    src = e.x * hs::kPage + (p & 63);
                    ++n_res;
                } else {
                    const int s = p2s[p];
                    if (s >= 0) {
                        kind = KIND_HOT;
                        src = hblk[s >> 6] * hs::kPage + (s & 63);
                        stamp[s] = c;
                        ++n_hot;
                    } else if (e.y < 0) {
                        err |= HS_DEVERR_NO_HOST;
                    } else {
                        kind = KIND_MISS;
                        hrow = e.y * hs::kPage + (p & 63);
                        int cj = j0 + l;
                        if (uni) {
                            // a union repeats positions across its lists: the
                            // first occurrence to mark pos_to_slot (-2 - its
                            // index) reads the row from the host, the others
                            // take its bytes (rank 0 replaces the mark)
                            const int old = atomicCAS(&p2s[p], -1, -2 - cj);
                            if (old <= -2) cj = -2 - old;
                        }
                        s_claim[l] = cj;
                        if (!gath && cj == j0 + l) {
                            // rows stay in the pool: this occurrence reads the
                            // row and keeps it in shared memory until its slot
                            // is known, if there is room (kind bits 4.. = stage + 1)
                            const int st = atomicAdd(&s_misc[3], 1);
                            if (st < ncap) kind |= (st + 1) << 4;
                        }
                        const int m = atomicAdd(&s_misc[0], 1);
                        s_mj[m] = l;
                    }
                }
            }
            // a union sends rank 0 one key per distinct position (its reader's);
            // the other occurrences take the reader's slot after barrier B
            const bool miss = (kind & 15) == KIND_MISS && (!uni || s_claim[l] == j0 + l);
            const unsigned bal = __ballot_sync(0xffffffffu, miss);
            if (bal) {
                const int leader = __ffs(bal) - 1;
                int kb = 0;
                if (lane == leader) kb = dsmem_atom_add(nkeys0, __popc(bal));
                kb = __shfl_sync(0xffffffffu, kb, leader);
                if (miss)
                    dsmem_st64(keys0 + 8u * (uint32_t)(kb + __popc(bal & ((1u << lane) - 1u))),
                               ((unsigned long long)(uint32_t)p << 32) | (uint32_t)(j0 + l));
            }
            if (l < nloc) {
                s_kind[l] = kind;
                s_src[l] = src;
                s_hrow[l] = hrow;
            }
        }
        if (n_res) atomicAdd(&s_misc[1], n_res);
        if (n_hot) atomicAdd(&s_misc[2], n_hot);
        __syncthreads();
        // this worker's totals into rank 0 (one writer per slot)
        if (tid < 3) hs::dsmem_st(hs::dsmem_map(&s_wcnt[4 * g + tid], 0), s_misc[tid]);
        __syncthreads();
        // the arrive releases (cluster scope) the hot-hit stamps, the keys and
        // the totals to rank 0, which acquires them in its wait
        hs::cluster_arrive();  // barrier A

        // ------------------------------------------------------------ phase 2
        const int nm = s_misc[0];
        if (gath) {
            // every gathered row whose bytes are at hand: pool rows for hits,
            // host rows for the misses this CTA reads (its claimed occurrences),
            // zeros for absent entries. Host and pool loads share each round.
            // Other occurrences of a union's miss copy their reader's row in
            // phase 3.
            const int nunits = nloc * V;
            uint8_t *gdst = gathered + row0 * RB;
            for (int base = tid; base < nunits; base += NT * UNROLL_H) {
                uint4 v[UNROLL_H];
                unsigned w = 0;  // bit u: store vector u
#pragma unroll
                for (int u = 0; u < UNROLL_H; ++u) {
                    const int i = base + u * NT;
                    v[u] = make_uint4(0, 0, 0, 0);
                    if (i < nunits) {
                        const int l = i / V, part = i - l * V;
                        const int kd = s_kind[l];
                        if (kd == KIND_RES || kd == KIND_HOT) {
                            v[u] = hs::ld_stream_v4(P.rows + (size_t)s_src[l] * RB + part * 16);
                            w |= 1u << u;
                        } else if (kd == KIND_MISS) {
                            if (s_claim[l] == j0 + l) {
                                v[u] = hs::ld_v4(P.host_rows + (size_t)s_hrow[l] * RB + part * 16);
                                w |= 1u << u;
                            }
                        } else {
                            w |= 1u << u;
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < UNROLL_H; ++u)
                    if (w >> u & 1u) hs::st_v4(gdst + (size_t)(base + u * NT) * 16, v[u]);
            }
        } else {
            // rows stay in the pool: each miss row this CTA reads goes to
            // shared memory until its slot is known (rows beyond the staging
            // room are read again in phase 3)
            for (int base = tid; base < nm * V; base += NT * UNROLL_H) {
                uint4 v[UNROLL_H];
                int at[UNROLL_H];  // staging unit, -1 = none
#pragma unroll
                for (int u = 0; u < UNROLL_H; ++u) {
                    const int i = base + u * NT;
                    at[u] = -1;
                    if (i < nm * V) {
                        const int mi = i / V, part = i - mi * V;
                        const int l = s_mj[mi];
                        const int st = (s_kind[l] >> 4) - 1;
                        if (st >= 0) {
                            v[u] = hs::ld_v4(P.host_rows + (size_t)s_hrow[l] * RB + part * 16);
                            at[u] = st * V + part;
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < UNROLL_H; ++u)
                    if (at[u] >= 0) st_shared_v4(s_stage + (size_t)at[u] * 16, v[u]);
            }
        }
        for (int l = tid; l < nloc; l += NT) {
            const int kd = s_kind[l] & 15;
            if (kd != KIND_MISS) resolved[row0 + l] = kd == KIND_NONE ? -1 : s_src[l];
            if (gath && fp8) {
                float sc = 0.f;
                if (kd == KIND_RES || kd == KIND_HOT) sc = P.scales[s_src[l]];
                else if (kd == KIND_MISS) sc = P.host_scales[s_hrow[l]];
                gscale[row0 + l] = sc;
            }
        }
        hs::cluster_wait();    // barrier A (long complete)
        hs::cluster_arrive();  // barrier B
        hs::cluster_wait();    // barrier B: rank 0 has placed every miss

        if (uni) {
            // occurrences that did not read their row: the reader's slot row,
            // from the reader's owner (-2 - row, as repeats are encoded; -1
            // when the position was rejected); each placed one counts as a miss
            int placed = 0;
            for (int mi = tid; mi < nm; mi += NT) {
                const int l = s_mj[mi];
                const int cj = s_claim[l];
                if (cj == j0 + l) continue;
                const int owner = 1 + cj / chunk;
                const int d = hs::dsmem_ld(hs::dsmem_map(&s_src[cj - (owner - 1) * chunk], owner));
                s_src[l] = d >= 0 ? -2 - d : -1;
                placed += d >= 0;
            }
            if (placed) atomicAdd(&counts[bi * 3 + 2], placed);
            __syncthreads();
            // barrier C: this CTA has finished reading its peers' shared
            // memory; no CTA exits before every CTA has arrived here
            hs::cluster_arrive();
        }

        // ------------------------------------------------------------ phase 3
        // Each placed position's row goes into its hot slot once, written by
        // the occurrence that read it (from shared memory, or the gathered
        // buffer / host arena when it was not staged); every other occurrence
        // of a union takes the row id (and, with gathered rows, copies the
        // reader's gathered row into its own). Rejected entries: zeros.
        {
            const uint8_t *greq = gath ? gathered + (size_t)bi * K * RB : nullptr;
            for (int base = tid; base < nm * V; base += NT * UNROLL) {
                uint4 v[UNROLL];
                size_t slot[UNROLL], gdst[UNROLL];
                bool tos[UNROLL], tog[UNROLL];
#pragma unroll
                for (int u = 0; u < UNROLL; ++u) {
                    const int i = base + u * NT;
                    tos[u] = tog[u] = false;
                    slot[u] = 0;
                    gdst[u] = 0;
                    if (i < nm * V) {
                        const int mi = i / V, part = i - mi * V;
                        const int l = s_mj[mi];
                        const int cj = s_claim[l];
                        const int d = s_src[l];
                        const bool own = cj == j0 + l;
                        const int sl = d >= 0 ? d : (d <= -2 ? -2 - d : -1);
                        const int st = (s_kind[l] >> 4) - 1;
                        gdst[u] = (row0 + l) * RB + part * 16;
                        slot[u] = (size_t)(sl < 0 ? 0 : sl) * RB + part * 16;
                        if (sl >= 0 && own) {
                            tos[u] = true;
                            v[u] = gath     ? hs::ld_v4(greq + (size_t)cj * RB + part * 16)
                                 : st >= 0 ? ld_shared_v4(s_stage + (size_t)st * RB + part * 16)
                                           : hs::ld_v4(P.host_rows + (size_t)s_hrow[l] * RB + part * 16);
                        } else if (gath && sl >= 0) {
                            tog[u] = true;
                            v[u] = hs::ld_v4(greq + (size_t)cj * RB + part * 16);
                        } else if (gath && sl < 0) {
                            tog[u] = true;
                            v[u] = make_uint4(0, 0, 0, 0);
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < UNROLL; ++u) {
                    if (tos[u]) hs::st_v4(P.rows + (size_t)slot[u], v[u]);
                    if (tog[u]) hs::st_v4(gathered + gdst[u], v[u]);
                }
            }
            for (int mi = tid; mi < nm; mi += NT) {
                const int l = s_mj[mi];
                const int d = s_src[l];
                if (d <= -2) {
                    // a union's repeat: the row its first occurrence placed
                    // (gathered row and scale already hold the host's bytes)
                    resolved[row0 + l] = -2 - d;
                    continue;
                }
                resolved[row0 + l] = d;
                if (fp8) {
                    if (!gath) {
                        if (d >= 0) P.scales[d] = P.host_scales[s_hrow[l]];
                    } else if (d >= 0) {
                        P.scales[d] = gscale[row0 + l];
                    } else {
                        gscale[row0 + l] = 0.f;
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------------ rank 0
        hs::cluster_arrive();  // barrier A
        hs::cluster_wait();
        if (tid == 0) {
            int res = 0, hot = 0;
            for (int q = 1; q <= W; ++q) {
                res += s_wcnt[4 * q + 1];
                hot += s_wcnt[4 * q + 2];
            }
            s_misc[8] = res;
            s_misc[9] = hot;
        }
        __syncthreads();
        // the workers' keys are in s_keys[0, n_miss), in arrival order
        const int n_miss = s_misc[4], tot_res = s_misc[8], tot_hot = s_misc[9];
        const bool leased = hblk[0] >= 0;
        int served = 0;
        if (n_miss > 0 || tot_hot > 0) {
            // sort the keys by (position, list index), ascending. 4096 keys
            // (a union of per-token lists): in registers, stored at swz8(i);
            // otherwise in shared memory, stored at i. (Measured: the register
            // network wins at 4096 keys and loses at 1024.)
            const int n2 = max(8, next_pow2(n_miss));
            for (int i = n_miss + tid; i < n2; i += NT) s_keys[i] = ~0ull;
            __syncthreads();
            const bool regsort = BIG && n2 == 8 * NT;
            if (regsort) {
                sort_keys_reg(s_keys, n2, tid);
            } else {
                sort_keys_smem(s_keys, n2, tid);
            }
            // sorted key i sits at kat(i)
            auto kat = [regsort](int i) { return regsort ? swz8(i) : i; };
            // rank of each miss among distinct positions (repeats: none; in a
            // union, their first occurrence's), stored as rank + 1 in key bits 13..26
            int m = 0;
            for (int base = 0; base < n_miss; base += NT) {
                const int i = base + tid;
                int first = 0;
                if (i < n_miss)
                    first = (i == 0) || ((s_keys[kat(i)] >> 32) != (s_keys[kat(i - 1)] >> 32));
                int tot;
                const int pre = hs::block_scan_flag<NT>(first, s_warp, tot);
                if (i < n_miss) {
                    const int rk = first ? m + pre : (uni ? m + pre - 1 : -1);
                    unsigned long long &key = s_keys[kat(i)];
                    key = (key & ~0xffffffffull) | ((unsigned long long)(rk + 1) << 13) | (key & 0x1fffull);
                }
                m += tot;
            }
            // stage the LRU order with each slot's protection in shared memory
            // (all loads in flight at once): bit 31 set = unprotected
            for (int i0 = 0; i0 < C; i0 += NT * 8) {
                int o[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int i = i0 + e * NT + tid;
                    o[e] = i < C ? lru[i] : 0;
                }
                int st[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) st[e] = (i0 + e * NT + tid) < C ? stamp[o[e]] : 0;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int i = i0 + e * NT + tid;
                    if (i < C) {
                        const int u = st[e] < c;
                        s_lru[i] = o[e] | (u ? int(0x80000000u) : 0);
                        s_prot[o[e]] = u ? 0 : 1;
                    }
                }
            }
            __syncthreads();
            // walk the LRU order: the first m unprotected slots are the victims,
            // the remaining unprotected slots move to the front
            int nu = 0;
            const int mv = leased ? m : 0;
            for (int c0 = 0; c0 < C; c0 += 8 * NT) {
                bool u[8];
                int o[8], rk[8];
#pragma unroll
                for (int it = 0; it < 8; ++it) {
                    const int i = c0 + it * NT + tid;
                    const int v = i < C ? s_lru[i] : 0;
                    o[it] = v & 0x7fffffff;
                    u[it] = v < 0;
                }
                const int tot = block_rank8(u, rk, s_rank, tid);
#pragma unroll
                for (int it = 0; it < 8; ++it) {
                    if (!u[it]) continue;
                    const int k = nu + rk[it];
                    if (k < mv) {
                        s_victim[k] = o[it];
                        s_prot[o[it]] = 1;  // stamped this step once placed
                    } else {
                        lru[k - mv] = o[it];
                    }
                }
                nu += tot;
                __syncthreads();  // s_rank is reused
            }
            const int mvict = min(mv, nu);
            __syncthreads();
            // place the misses; tell each owner worker its slot row (-1 =
            // rejected; in a union, -2 - row = a repeat of a placed miss, whose
            // row the first occurrence copies)
            if (tid == 0) s_misc[3] = 0;
            __syncthreads();
            int placed = 0;
            for (int i = tid; i < n_miss; i += NT) {
                const unsigned long long key = s_keys[kat(i)];
                const int p = static_cast<int>(key >> 32), j = static_cast<int>(key & 0x1fffu);
                const int rk = static_cast<int>((key >> 13) & 0x3fffu) - 1;
                const bool first = (i == 0) || ((s_keys[kat(i - 1)] >> 32) != (key >> 32));
                int dst = -1;
                if (rk < 0) {
                    err |= HS_DEVERR_DUPLICATE;
                } else if (rk >= mvict) {
                    err |= HS_DEVERR_CAPACITY;
                    if (uni && first) p2s[p] = -1;  // drop the workers' mark
                } else {
                    const int v = s_victim[rk];
                    if (first) {
                        const int old = tag[v];
                        if (old >= 0) p2s[old] = -1;
                        tag[v] = p;
                        stamp[v] = c;
                        p2s[p] = v;
                    }
                    dst = hblk[v >> 6] * hs::kPage + (v & 63);
                    ++placed;
                    if (!first) dst = -2 - dst;
                }
                const int owner = 1 + j / chunk;
                hs::dsmem_st(hs::dsmem_map(&s_src[j - (owner - 1) * chunk], owner), dst);
            }
            if (placed) atomicAdd(&s_misc[3], placed);
            __syncthreads();
            // the slots stamped this step, in slot order, close the LRU order
            int out = nu - mvict;
            for (int c0 = 0; c0 < C; c0 += 8 * NT) {
                bool f[8];
                int rk[8];
#pragma unroll
                for (int it = 0; it < 8; ++it) {
                    const int sl = c0 + it * NT + tid;
                    f[it] = sl < C && s_prot[sl];
                }
                const int tot = block_rank8(f, rk, s_rank, tid);
#pragma unroll
                for (int it = 0; it < 8; ++it)
                    if (f[it]) lru[out + rk[it]] = c0 + it * NT + tid;
                out += tot;
                __syncthreads();  // s_rank is reused
            }
            served = s_misc[3];  // misses resolved, counting the repeats of a union
        }
        if (tid == 0) {
            P.clock[r] = c;
            counts[bi * 3 + 0] = tot_res;
            counts[bi * 3 + 1] = tot_hot;
            counts[bi * 3 + 2] = served;
        }
        __syncthreads();
        hs::cluster_arrive();  // barrier B: miss slots (and counts) released to the workers
        hs::cluster_wait();
        if (uni) hs::cluster_arrive();  // barrier C (see the workers)
    }
    if (uni) {
        // a union's workers read each other's shared memory after barrier B:
        // wait until all of them are done before this CTA's memory goes away
        __syncthreads();
        hs::cluster_wait();  // barrier C
    }
    if (err) atomicOr(P.err, err);
}

template <int RB, bool BIG>
__global__ void __launch_bounds__(NT, 2)
resolve_kernel(const hs::DevPool P, const int32_t *__restrict__ req_ids,
               const int32_t *__restrict__ topk, int K, int chunk, int G,
               int32_t *__restrict__ resolved, uint8_t *__restrict__ gathered,
               float *__restrict__ gscale, int32_t *__restrict__ counts, int uni) {
    resolve_body<RB, BIG, hs::DevPool>(P, req_ids, topk, K, chunk, G, resolved, gathered, gscale,
                                       counts, uni);
}

// One launch over (request, layer) pairs: layer z = blockIdx.z has its own pool
// (its table addresses, copied to the device when the layer group was made)
// and its own slice of every per-entry array.
template <int RB, bool BIG>
__global__ void __launch_bounds__(NT, 2)
resolve_layers_kernel(const hs::DevPool *__restrict__ layers, const int32_t *__restrict__ req_ids,
               const int32_t *__restrict__ topk, int K, int chunk, int G,
               int32_t *__restrict__ resolved, uint8_t *__restrict__ gathered,
               float *__restrict__ gscale, int32_t *__restrict__ counts, int uni) {
    const size_t ents = (size_t)blockIdx.z * gridDim.y * K;
    resolve_body<RB, BIG, const hs::DevPool &>(
        layers[blockIdx.z], req_ids, topk + ents, K, chunk, G, resolved + ents,
        gathered ? gathered + ents * RB : nullptr, gscale ? gscale + ents : nullptr,
        counts + (size_t)blockIdx.z * gridDim.y * 3, uni);
}

int pick_cluster(int K) {
    // one bookkeeping CTA + up to 7 workers (portable cluster size), each
    // worker owning at least 32 entries. (16-CTA clusters for long unions were
    // measured slower: 108 -> 119 us on the MTP workload.)
    int W = 7;
    while (W > 1 && (K + W - 1) / W < 32) --W;
    return W + 1;
}

}  // namespace

size_t hs_resolve_smem_bytes(int K, int G, int C, int RB, bool stage) {
    const int chunk = (K + G - 2) / (G - 1);
    Smem L{chunk, std::max(8, next_pow2(K)), K, C};
    const size_t want = stage ? std::min(kStageSmemCap, L.off_stage() + (size_t)chunk * RB) : 0;
    return (std::max(L.total(), want) + 15) & ~size_t(15);
}

hs_status hs_resolve_prepare(hs_pool *pool) {
    size_t mx = 0;
    for (int K = 1; K <= pool->cfg.max_topk; ++K) {
        const size_t b = hs_resolve_smem_bytes(K, pick_cluster(K), pool->cfg.hot_rows,
                                               pool->row_bytes, true);
        if (b > mx) mx = b;
    }
    if (mx > 232448) return HS_ERR_UNSUPPORTED;  // shared memory per block on sm_103
    HS_CUDA_TRY(cudaFuncSetAttribute(resolve_kernel<1152, false>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)mx));
    HS_CUDA_TRY(cudaFuncSetAttribute(resolve_kernel<576, false>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)mx));
    HS_CUDA_TRY(cudaFuncSetAttribute(resolve_kernel<1152, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)mx));
    HS_CUDA_TRY(cudaFuncSetAttribute(resolve_kernel<576, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)mx));
    HS_CUDA_TRY(cudaFuncSetAttribute(resolve_layers_kernel<1152, false>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)mx));
    HS_CUDA_TRY(cudaFuncSetAttribute(resolve_layers_kernel<576, false>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)mx));
    HS_CUDA_TRY(cudaFuncSetAttribute(resolve_layers_kernel<1152, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)mx));
    HS_CUDA_TRY(cudaFuncSetAttribute(resolve_layers_kernel<576, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)mx));
    return HS_OK;
}

hs_status hs_launch_resolve(hs_pool *pool, int32_t B, const int32_t *req_ids, const int32_t *topk,
                            int32_t K, int32_t *resolved, void *gathered, float *gscale,
                            int32_t *counts, cudaStream_t stream, int uni,
                            const hs::DevPool *layers, int nlayers) {
    const int G = pick_cluster(K);
    const int chunk = (K + G - 2) / (G - 1);
    const size_t smem =
        hs_resolve_smem_bytes(K, G, pool->cfg.hot_rows, pool->row_bytes, gathered == nullptr);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(G, B, nlayers);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = G;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    auto *uc = static_cast<uint8_t *>(gathered);
    const bool big = K > 2048;
    const int Ki = K;
    if (layers) {
        if (pool->row_bytes == 1152)
            e = big ? cudaLaunchKernelEx(&cfg, resolve_layers_kernel<1152, true>, layers, req_ids,
                                         topk, Ki, chunk, G, resolved, uc, gscale, counts, uni)
                    : cudaLaunchKernelEx(&cfg, resolve_layers_kernel<1152, false>, layers, req_ids,
                                         topk, Ki, chunk, G, resolved, uc, gscale, counts, uni);
        else
            e = big ? cudaLaunchKernelEx(&cfg, resolve_layers_kernel<576, true>, layers, req_ids,
                                         topk, Ki, chunk, G, resolved, uc, gscale, counts, uni)
                    : cudaLaunchKernelEx(&cfg, resolve_layers_kernel<576, false>, layers, req_ids,
                                         topk, Ki, chunk, G, resolved, uc, gscale, counts, uni);
    } else {
        const hs::DevPool P = pool->dev();
        if (pool->row_bytes == 1152)
            e = big ? cudaLaunchKernelEx(&cfg, resolve_kernel<1152, true>, P, req_ids, topk, Ki,
                                         chunk, G, resolved, uc, gscale, counts, uni)
                    : cudaLaunchKernelEx(&cfg, resolve_kernel<1152, false>, P, req_ids, topk, Ki,
                                         chunk, G, resolved, uc, gscale, counts, uni);
        else
            e = big ? cudaLaunchKernelEx(&cfg, resolve_kernel<576, true>, P, req_ids, topk, Ki,
                                         chunk, G, resolved, uc, gscale, counts, uni)
                    : cudaLaunchKernelEx(&cfg, resolve_kernel<576, false>, P, req_ids, topk, Ki,
                                         chunk, G, resolved, uc, gscale, counts, uni);
    }
    return e == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}

namespace {
hs_status resolve_entry(hs_pool_t pool, int32_t B, const int32_t *d_req_ids,
                        const int32_t *d_topk_idx, int32_t K, int32_t *d_resolved,
                        void *d_gathered, float *d_gathered_scale, int32_t *d_counts,
                        void *stream, int uni) {
    if (!pool || B < 0 || !d_req_ids || !d_topk_idx || !d_resolved || !d_counts)
        return HS_ERR_INVALID_ARG;
    // one list: at most one entry per slot; a union: its distinct misses are
    // checked against the free slots on the device
    if (K < 1 || K > pool->cfg.max_topk || (!uni && K > pool->cfg.hot_rows)) return HS_ERR_CAPACITY;
    if (B > 65535) return HS_ERR_INVALID_ARG;
    const bool fp8 = pool->cfg.dtype == HS_FP8_E4M3_ROWSCALE;
    // gathered rows (and, for FP8 pools, their scales) or neither
    if (d_gathered ? fp8 != (d_gathered_scale != nullptr) : d_gathered_scale != nullptr)
        return HS_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(d_gathered) & 15u) != 0) return HS_ERR_INVALID_ARG;
    if (B == 0) return HS_OK;
    return hs_launch_resolve(pool, B, d_req_ids, d_topk_idx, K, d_resolved, d_gathered,
                             d_gathered_scale, d_counts, static_cast<cudaStream_t>(stream), uni,
                             nullptr, 1);
}
}  // namespace

extern "C" hs_status hs_resolve_topk(hs_pool_t pool, int32_t B, const int32_t *d_req_ids,
                                     const int32_t *d_topk_idx, int32_t K, int32_t *d_resolved,
                                     void *d_gathered, float *d_gathered_scale, int32_t *d_counts,
                                     void *stream) {
    return resolve_entry(pool, B, d_req_ids, d_topk_idx, K, d_resolved, d_gathered,
                         d_gathered_scale, d_counts, stream, 0);
}

// Several top-K lists per request (one per speculative query token) resolved
// as their union against the request's one hot state.
extern "C" hs_status hs_resolve_topk_union(hs_pool_t pool, int32_t B, const int32_t *d_req_ids,
                                           const int32_t *d_topk_idx, int32_t K,
                                           int32_t *d_resolved, void *d_gathered,
                                           float *d_gathered_scale, int32_t *d_counts,
                                           void *stream) {
    return resolve_entry(pool, B, d_req_ids, d_topk_idx, K, d_resolved, d_gathered,
                         d_gathered_scale, d_counts, stream, 1);
}

// ---------------------------------------------------------------- layer groups
// The pools of several sparse-MLA layers, resolved in one launch whose grid
// spans (request, layer) pairs ("vLLM GLM 5.3 优化：混合 HiSparse 卸载", 关键架构细节,
// 轻量级执行: all sparse-MLA layers launched at once, in stream order).
struct hs_layer_group {
    int L = 0;
    hs_pool *first = nullptr;
    hs::DevPool *d_pools = nullptr;  // [L] device copies of the pools' table pointers
};

extern "C" hs_status hs_layer_group_create(const hs_pool_t *pools, int32_t L,
                                           hs_layer_group_t *out) {
    if (!pools || !out || L < 1 || L > 65535) return HS_ERR_INVALID_ARG;
    *out = nullptr;
    const hs_pool *p0 = pools[0];
    if (!p0) return HS_ERR_INVALID_ARG;
    std::vector<hs::DevPool> host(L);
    for (int l = 0; l < L; ++l) {
        const hs_pool *p = pools[l];
        if (!p || p->device != p0->device || p->cfg.dtype != p0->cfg.dtype ||
            p->cfg.hot_rows != p0->cfg.hot_rows || p->cfg.max_topk != p0->cfg.max_topk)
            return HS_ERR_INVALID_ARG;
        host[l] = p->dev();
    }
    int cur = 0;
    HS_CUDA_TRY(cudaGetDevice(&cur));
    if (cur != p0->device) return HS_ERR_INVALID_ARG;
    auto *g = new (std::nothrow) hs_layer_group;
    if (!g) return HS_ERR_OUT_OF_MEMORY;
    if (cudaMalloc(&g->d_pools, L * sizeof(hs::DevPool)) != cudaSuccess) {
        delete g;
        return HS_ERR_OUT_OF_MEMORY;
    }
    if (cudaMemcpy(g->d_pools, host.data(), L * sizeof(hs::DevPool), cudaMemcpyHostToDevice) !=
        cudaSuccess) {
        cudaFree(g->d_pools);
        delete g;
        return HS_ERR_CUDA;
    }
    g->L = L;
    g->first = pools[0];
    *out = g;
    return HS_OK;
}

extern "C" hs_status hs_layer_group_destroy(hs_layer_group_t g) {
    if (!g) return HS_ERR_INVALID_ARG;
    cudaFree(g->d_pools);
    delete g;
    return HS_OK;
}

extern "C" hs_status hs_resolve_topk_layers(hs_layer_group_t g, int32_t B, const int32_t *d_req_ids,
                                            const int32_t *d_topk_idx, int32_t K,
                                            int32_t *d_resolved, void *d_gathered,
                                            float *d_gathered_scale, int32_t *d_counts,
                                            void *stream) {
    if (!g || B < 0 || !d_req_ids || !d_topk_idx || !d_resolved || !d_counts)
        return HS_ERR_INVALID_ARG;
    hs_pool *pool = g->first;
    if (K < 1 || K > pool->cfg.max_topk || K > pool->cfg.hot_rows) return HS_ERR_CAPACITY;
    if (B > 65535) return HS_ERR_INVALID_ARG;
    const bool fp8 = pool->cfg.dtype == HS_FP8_E4M3_ROWSCALE;
    if (d_gathered ? fp8 != (d_gathered_scale != nullptr) : d_gathered_scale != nullptr)
        return HS_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(d_gathered) & 15u) != 0) return HS_ERR_INVALID_ARG;
    if (B == 0) return HS_OK;
    return hs_launch_resolve(pool, B, d_req_ids, d_topk_idx, K, d_resolved, d_gathered,
                             d_gathered_scale, d_counts, static_cast<cudaStream_t>(stream), 0,
                             g->d_pools, g->L);
}
