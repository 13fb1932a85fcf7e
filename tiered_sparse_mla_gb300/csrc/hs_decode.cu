// hs_decode.cu -- sparse MLA decode over the selected top-K latent rows, on
// tcgen05 tensor cores (sm_103a).
//
// Attention restricted to the K rows the indexer selected ("vLLM GLM 5.3 优化：
// 混合 HiSparse 卸载", section 解决 KV 缓存内存压力; "vLLM Hybrid HiSparse：稀疏MLA
// 破解长上下文显存瓶颈", section 稀疏MLA的核心思想). MLA keeps one 576-wide latent
// row per token: the key is the whole row, the value its first 512 elements.
// Query token t of a request sits at position L - T + t and sees entries whose
// position is <= that (MTP draft tokens share one top-K list, 与 vLLM 栈的集成).
//
// All H*T query rows of a request share the same K rows, so QK^T and PV are
// dense contractions: S[128 x 64] = Q[128 x 576] K^T, O[128 x 512] = P V.
//
// Work unit: (request, 128-row M tile, KV split), run by a cluster of two CTAs.
// The 576-wide rows are nine 64-column chunks: eight value chunks and the rope
// chunk 8. CTA h (h = 0, 1):
//   - loads, per 64-key tile, its four value chunks 4h..4h+3 and the rope
//     chunk (40 KB of BF16 rows, 20 KB of FP8 codes; rows read in place from
//     the pool bring only the half of the rope chunk this CTA uses);
//   - holds Q in tensor memory for those value chunks and for its half of the
//     rope chunk (columns 32h..32h+31 of it), so that each CTA computes S over
//     288 of the 576 depth columns;
//   - writes its partial S of each half tile (32 keys), in f32 and already
//     multiplied by sm_scale*log2(e) (times the row scale for FP8), to shared
//     memory, sends it to the peer with one 16 KB bulk copy, and adds the
//     peer's partial; f32 addition is commutative, so both CTAs hold
//     bit-identical S and take identical softmax decisions;
//   - accumulates O for output columns [256h, 256h + 256) (its value chunks)
//     with P in tensor memory.
// FP8 rows: the codes are turned into BF16 exactly (each code's bits placed as
// a BF16 of value code * 2^-120, then multiplied by 2^120); the row's fp32
// scale multiplies the scores of that key in f32, and its probability before
// P is rounded to BF16 (the sum of probabilities stays unscaled). So Q stays
// BF16 on both paths and no operand is rounded beyond BF16.
// Roles inside a CTA (384 threads):
//   warp 0      producer: Q once by TMA, into the space of tile groups 2-3
//               (their first loads wait until Q has moved to TMEM), then per
//               tile one TMA box of the four value chunks and one of the rope
//               chunk; rows read in place are copied from the pool in 16-byte
//               cp.async pieces (keys 0-31 of each tile);
//   warp 1      MMA issuer (one thread): S_j = Q K_j^T into the TMEM S buffer
//               once tile j is ready and S_{j-1} has been read; O += P_u V_u
//               per half tile u (V read from the same smem chunks as K through
//               an MN-major descriptor) once P_u is written; PV first when both
//               can go;
//   warp 2      per tile: the lowest query token that sees each key, and for
//               FP8 the key's row scale, into shared rings, so that no row
//               thread waits on a global load; rows read in place: the
//               copies of keys 32-63, with the ids and scales loaded a tile
//               ahead;
//   warp 3      courier (one thread): the bulk copies of the partial S to the
//               peer, each once the peer has read the half tile sent two
//               before into the same buffer;
//   warps 4-7   stagers, one thread per query row (TMEM lane): read S_j, free
//               it for the next QK, scale it and write both halves to the
//               outgoing buffers; FP8: also convert each landed tile of codes
//               to BF16 in place, two tiles ahead of its QK; BF16: output
//               columns 128-255 of the epilogue;
//   warps 8-11  softmax, one thread per query row, per half tile: add the two
//               partials, mask, online softmax with a conditional rescale, P
//               to TMEM; then the epilogue (O / l through shared memory and
//               TMA stores; BF16 rows: columns 0-127).
// TMEM (512 columns): O half 256 | S 64 | P 32 | Q 144.
// Every mbarrier wait is bounded in time; on expiry the kernel sets
// HS_DEVERR_TIMEOUT, drains its own copies and MMAs and returns. Roles hand
// over through mbarriers, so one that gives up leaves no other waiting on a
// hardware barrier (the FP8 stagers' named barrier is reached by all four
// stager warps on every path).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <climits>
#include <cstdint>
#include <mutex>

#include "hs_internal.cuh"
#include "hs_tc.cuh"

namespace {

using namespace hs::tc;

constexpr int NSTG = 128;            // stager threads (warps 4-7)
constexpr int NSFT = 128;            // softmax threads (warps 8-11)
constexpr int NCVT = NSTG;           // FP8: the stagers also convert the codes
constexpr int BM = 128, BN = 64;
constexpr int NLC = 5;               // chunks a CTA loads per 64-key tile: 4 value + rope
constexpr int NG = 4;                // tile groups in flight
constexpr int NQC = 5;               // Q chunks staged per CTA (4 value + rope)
constexpr int QCH_BYTES = BM * 128;  // 128 rows x 64 columns x 2 B
constexpr int KCH_BYTES = BN * 128;  // 64 keys x 64 columns x 2 B
constexpr int FCH_BYTES = BN * 64;   // 64 keys x 64 e4m3 codes
constexpr int GRP_BYTES = NLC * KCH_BYTES;
constexpr int CVT_UNITS = NLC * FCH_BYTES / 16 / NCVT;  // 16-byte code units per converter per tile
constexpr int X_BYTES = BM * 32 * 4; // 128 rows x 32 f32 partial scores (half a tile)
constexpr float TAU2 = 8.f;          // rescale threshold, log2 units
constexpr uint32_t TMEM_COLS = 512, TM_O = 0, TM_S = 256, TM_P = 320, TM_Q = 352;
static_assert(TM_Q + 4 * 32 + 16 <= TMEM_COLS, "tensor memory");

template <bool FP8>
struct Threads {
    static constexpr int N = 384;
};

struct Cfg {
    static constexpr int OFF_RING = 0;
    static constexpr int OFF_QSTAGE = OFF_RING + 2 * GRP_BYTES;       // tile groups 2-3
    static constexpr int OFF_XIN = OFF_RING + NG * GRP_BYTES;         // [2] the peer's partial S
    static constexpr int OFF_XOUT = OFF_XIN + 2 * X_BYTES;            // [2] own partial S
    static constexpr int OFF_KVIS = OFF_XOUT + 2 * X_BYTES;           // int16 [NG][64]
    static constexpr int OFF_KSC = OFF_KVIS + NG * BN * 2;            // f32 [NG][64] FP8 row scales
    static constexpr int OFF_TDMAX = OFF_KSC + NG * BN * 4;           // int32 [NG][2]
    static constexpr int OFF_BAR = OFF_TDMAX + NG * 8;
    static constexpr int B_QFULL = 0, B_QREADY = 1, B_DRAIN = 2, B_GFULL = 3;
    static constexpr int B_GEMPTY = B_GFULL + NG, B_GLANDED = B_GEMPTY + NG;
    static constexpr int B_SFULL = B_GLANDED + NG, B_SFREE = B_SFULL + 1;
    static constexpr int B_PFULL = B_SFREE + 1;     // [2] P of a half tile (columns 16h..) written
    static constexpr int B_PVDONE = B_PFULL + 2;    // [2] PV of a half tile done
    static constexpr int B_XFULL = B_PVDONE + 2;    // [2] the peer's partial has landed
    static constexpr int B_XTAKEN = B_XFULL + 2;    // [2] the peer has read what this CTA sent
    static constexpr int B_STAGED = B_XTAKEN + 2;   // [2] own partial written, ready to send
    static constexpr int B_READ = B_STAGED + 2;     // [2] both partials of a half tile read here
    static constexpr int B_XOUTDONE = B_READ + 2;   // [2] the courier's copy has read X_out
    static constexpr int B_KVIS = B_XOUTDONE + 2;   // [NG] key visibility (and scales) of a tile
    static constexpr int NBAR = B_KVIS + NG;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // [0] TMEM base, [1] abort flag
    static constexpr int SMEM = OFF_MISC + 16;
    static constexpr int SMEM_ALLOC = SMEM + 1024;       // room to align the base to 1 KiB
    static_assert(OFF_QSTAGE % 1024 == 0 && OFF_XIN % 1024 == 0 && OFF_XOUT % 1024 == 0,
                  "alignment");
    static_assert(NQC * QCH_BYTES <= (NG - 2) * GRP_BYTES, "Q staging space");
    static_assert(SMEM_ALLOC <= 232448, "shared memory");
};

// Programmatic dependent launch: this grid may start while the previous kernel
// on the stream (the step's resolve) is still running; a thread waits here for
// that kernel's completion and memory before reading anything it wrote.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel on the stream (the split merge) be scheduled early.
__device__ __forceinline__ void grid_dep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

struct DecParams {
    const int32_t *resolved, *topk, *req_ids, *ctx;
    const float *gscale;        // gathered row scales (FP8, gathered rows)
    const float *pool_scales;   // pool row scales (FP8, rows read in place)
    const uint8_t *pool_rows;   // the pool's rows (rows read in place)
    int zero_row;               // pool row of zeros read for absent entries (in place)
    __nv_bfloat16 *out;
    float *lse, *ws_lse;
    __nv_bfloat16 *ws_o;  // split partials: normalised O of one split (a weighted mean of value rows)
    uint32_t *err;
    int B, T, H, K, M, nsplit, kps, max_req;
    int tpl;  // lists per request: list b is token b % tpl of request b / tpl
    float scale_log2;
};

__device__ __forceinline__ void st_shared_v4(uint32_t a, uint32_t x, uint32_t y, uint32_t z,
                                             uint32_t w) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w)
                 : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a)
                 : "memory");
    return v;
}
__device__ __forceinline__ float4 ld_shared_f4(uint32_t a) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(a)
                 : "memory");
    return v;
}
// TMEM load of 32 columns whose registers only become valid after the wait;
// the wait takes them as operands so no use can be scheduled before it.
#define HS_TMEM_LD32(taddr, r)                                                                    \
    asm volatile(                                                                                 \
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"  \
        "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"        \
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),    \
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),             \
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),          \
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),          \
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),          \
          "=r"(r[31])                                                                             \
        : "r"(taddr)                                                                              \
        : "memory")
#define HS_TMEM_WAIT_LD32(r)                                                                      \
    asm volatile("tcgen05.wait::ld.sync.aligned;"                                                 \
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),        \
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),      \
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),  \
                   "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),  \
                   "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),  \
                   "+r"(r[30]), "+r"(r[31])::"memory")
// TMEM store of 32 (16) columns of 32-bit words from this thread's lane.
#define HS_TMEM_ST32(taddr, r)                                                                    \
    asm volatile(                                                                                 \
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"   \
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"      \
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),           \
        "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),          \
        "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]),      \
        "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),      \
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])                               \
        : "memory")
#define HS_TMEM_ST16(taddr, r)                                                                    \
    asm volatile(                                                                                 \
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"   \
        "%13,%14,%15,%16};" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]),  \
        "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]),           \
        "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])                                           \
        : "memory")

// A box of a 4-D tensor map (coordinates innermost first).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const void *tmap, int c0, int c1, int c2, int c3,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

// Shared memory to a box of a 3-D tensor map (bulk async group of this thread).
__device__ __forceinline__ void tma_store_3d(const void *tmap, uint32_t src, int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(tmap)),
        "r"(src), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Four e4m3 codes (the bytes of w, lowest first) to four BF16 values, exactly.
// A code's sign, four exponent bits and three mantissa bits, placed at the
// BF16 sign, the low four exponent bits and the top three mantissa bits, form
// a BF16 whose value is the code's times 2^-120: a normal code 2^(e-7)(1+m/8)
// becomes 2^(e-127)(1+m/8), a subnormal code 2^-6 (m/8) the BF16 subnormal
// 2^-126 (m/8). Multiplying by 2^120 (exact) gives the code's value.
__device__ __forceinline__ void e4m3x4_to_bf16(uint32_t w, uint32_t &lo, uint32_t &hi) {
    const uint32_t t0 = __byte_perm(w, 0u, 0x1404);  // bytes (c1, 0, c0, 0), high to low
    const uint32_t t1 = __byte_perm(w, 0u, 0x3424);  // bytes (c3, 0, c2, 0)
    uint32_t a = (t0 & 0x80008000u) | ((t0 >> 4) & 0x07F007F0u);
    uint32_t b = (t1 & 0x80008000u) | ((t1 >> 4) & 0x07F007F0u);
    const uint32_t two120 = 0x7B807B80u;  // (2^120, 2^120) in BF16
    asm("mul.rn.bf16x2 %0, %0, %1;" : "+r"(a) : "r"(two120));
    asm("mul.rn.bf16x2 %0, %0, %1;" : "+r"(b) : "r"(two120));
    lo = a;
    hi = b;
}

// One kind::f16 MMA with A from TMEM; the B descriptor comes as two 32-bit
// halves (only the low half changes between the MMAs of one operand walk) and
// the accumulate flag is a constant, so that issuing costs a few instructions.
template <bool ACC>
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint32_t blo, uint32_t bhi,
                                       uint32_t idesc) {
    if (ACC)
        asm volatile(
            "{\n .reg .b64 bd;\n mov.b64 bd, {%2, %3};\n"
            " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, 1;\n}\n" ::"r"(d),
            "r"(a), "r"(blo), "r"(bhi), "r"(idesc)
            : "memory");
    else
        asm volatile(
            "{\n .reg .b64 bd;\n mov.b64 bd, {%2, %3};\n"
            " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, 0;\n}\n" ::"r"(d),
            "r"(a), "r"(blo), "r"(bhi), "r"(idesc)
            : "memory");
}

// S = Q K^T over this CTA's 288 depth columns: the four value chunks (A = Q
// chunk c at TMEM columns aq + 32 c, B = local chunk c) and its half of the
// rope chunk (A at aq + 128, B = K steps 2h, 2h + 1 of local chunk 4).
// Straight-line: 18 MMAs of K = 16.
__device__ __forceinline__ void issue_qk(uint32_t dS, uint32_t aq, uint32_t blo, uint32_t bhi,
                                         uint32_t idesc, int half) {
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t a = aq + 32u * c + 8u * k;
            const uint32_t lo = blo + (uint32_t)((c * KCH_BYTES + 32 * k) >> 4);
            if (c == 0 && k == 0)
                mma_ts<false>(dS, a, lo, bhi, idesc);
            else
                mma_ts<true>(dS, a, lo, bhi, idesc);
        }
#pragma unroll
    for (int k = 0; k < 2; ++k)
        mma_ts<true>(dS, aq + 128u + 8u * k,
                     blo + (uint32_t)((4 * KCH_BYTES + 32 * (2 * half + k)) >> 4), bhi, idesc);
}

// Row r, 16-byte chunk c of a 128-byte-per-row tile with the 128-byte swizzle
// (the TMA layout of Q and K).
__device__ __forceinline__ uint32_t x_off(int r, int c) {
    return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}
template <bool FP8, bool INPLACE>
__global__ void __launch_bounds__(Threads<FP8>::N, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_kv,
                 const __grid_constant__ CUtensorMap tm_kr, const __grid_constant__ CUtensorMap tm_o,
                 const DecParams p) {
    using C = Cfg;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = hs::smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (base - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = static_cast<int>(hs::cluster_ctarank());
    const uint32_t peer = static_cast<uint32_t>(half ^ 1);
    const int split = blockIdx.x >> 1, mt = blockIdx.y, b = blockIdx.z;
    const int k0 = split * p.kps, k1 = min(p.K, k0 + p.kps);
    const int ntiles = (k1 - k0 + BN - 1) / BN;
    const int nunits = 2 * ntiles;  // half tiles of 32 keys: the exchange and softmax unit
    volatile int32_t *misc = reinterpret_cast<volatile int32_t *>(smem + C::OFF_MISC);
    const uint32_t sR = base + C::OFF_RING, sQst = base + C::OFF_QSTAGE;
    const uint32_t sXin = base + C::OFF_XIN, sXout = base + C::OFF_XOUT;
    const uint32_t sKvis = base + C::OFF_KVIS, sKsc = base + C::OFF_KSC;
    volatile int32_t *tdmax = reinterpret_cast<volatile int32_t *>(smem + C::OFF_TDMAX);
    auto bar = [&](int i) { return base + C::OFF_BAR + 8u * (uint32_t)i; };
    auto slot = [&](int g, int lc) { return sR + (uint32_t)(g * GRP_BYTES + lc * KCH_BYTES); };
    // FP8: the e4m3 codes of local chunk lc, packed in the upper half of the tile group
    auto codes = [&](int g, int lc) {
        return sR + (uint32_t)(g * GRP_BYTES + NLC * FCH_BYTES + lc * FCH_BYTES);
    };
    auto fail = [&]() {
        misc[1] = 1;
        atomicOr(p.err, HS_DEVERR_TIMEOUT);
    };
    // Rows read in place: keys kb..kb + 31 of a tile (lane i holds the pool row
    // of key kb + i in `rows`) copied from the pool in 16-byte pieces with
    // cp.async, the value half of one row (BF16) or of two (FP8 codes) per
    // instruction, then the half of the rope chunk this CTA's QK reads. BF16
    // pieces land in the 128-byte-swizzled layout the MMA reads, FP8 codes
    // packed [chunk][row][64 B] for the converters. Called by a whole warp.
    auto gather_keys = [&](int g, int rows, int kb) {
        constexpr int RB = FP8 ? hs::kDim : 2 * hs::kDim;  // row bytes
        constexpr int VP = FP8 ? 16 : 32;                  // 16-byte pieces of a value half
        constexpr int RH = FP8 ? 2 : 4;                    // 16-byte pieces of half the rope chunk
        const uint8_t *pool = p.pool_rows;
#pragma unroll 4
        for (int m = 0; m < VP; ++m) {
            const int kk = m * (32 / VP) + lane / VP, pc = lane % VP;
            const int r = __shfl_sync(0xffffffffu, rows, kk);
            const int k = kb + kk;
            const uint8_t *src = pool + (size_t)r * RB + half * (RB / 9 * 4) + pc * 16;
            const uint32_t dst = FP8 ? codes(g, pc >> 2) + (uint32_t)(k * 64 + (pc & 3) * 16)
                                     : slot(g, pc >> 3) + (uint32_t)(k * 128 + (((pc & 7) ^ (k & 7)) << 4));
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
        }
#pragma unroll
        for (int m = 0; m < RH; ++m) {
            const int kk = m * (32 / RH) + lane / RH, pc = RH * half + lane % RH;
            const int r = __shfl_sync(0xffffffffu, rows, kk);
            const int k = kb + kk;
            const uint8_t *src = pool + (size_t)r * RB + (RB / 9 * 8) + pc * 16;
            const uint32_t dst = FP8 ? codes(g, 4) + (uint32_t)(k * 64 + pc * 16)
                                     : slot(g, 4) + (uint32_t)(k * 128 + ((pc ^ (k & 7)) << 4));
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
        }
    };

    if (threadIdx.x == 0) {
        mbar_init(bar(C::B_QFULL), 1);
        mbar_init(bar(C::B_QREADY), NSTG + NSFT);
        mbar_init(bar(C::B_DRAIN), 1);
        for (int g = 0; g < NG; ++g) {
            // TMA loads complete a tile with one arrive and its bytes; rows read
            // in place arrive once per producer lane (cp.async completion)
            mbar_init(bar(C::B_GFULL + g), FP8 ? NCVT : (INPLACE ? 64 : 1));
            mbar_init(bar(C::B_GEMPTY + g), 1);
            mbar_init(bar(C::B_GLANDED + g), INPLACE ? 64 : 1);
            mbar_init(bar(C::B_KVIS + g), 32);
        }
        mbar_init(bar(C::B_SFULL), 1);
        mbar_init(bar(C::B_SFREE), NSTG);
        for (int x = 0; x < 2; ++x) {
            mbar_init(bar(C::B_PFULL + x), NSFT);
            mbar_init(bar(C::B_PVDONE + x), 1);
            mbar_init(bar(C::B_XFULL + x), 1);  // own arm + the peer's bulk copy bytes
            mbar_init(bar(C::B_XTAKEN + x), NSFT / 32);  // one arrive per peer softmax warp
            mbar_init(bar(C::B_STAGED + x), NSTG);
            mbar_init(bar(C::B_READ + x), NSFT / 32);    // one arrive per softmax warp
            mbar_init(bar(C::B_XOUTDONE + x), 1);
        }
        misc[1] = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(base + C::OFF_MISC, TMEM_COLS);
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_q);
        if (!INPLACE) {
            prefetch_tmap(&tm_kv);
            prefetch_tmap(&tm_kr);
        }
        prefetch_tmap(&tm_o);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync_all();  // the peer's barriers are initialised before any remote arrive
    const uint32_t tmem = static_cast<uint32_t>(misc[0]);
    grid_dep_launch();
    // the producer first issues the Q loads (Q does not come from the resolve)
    if (warp != 0) grid_dep_wait();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // Lane 0 loads Q and takes each slot; a tile read from the gathered
        // buffer is two boxes (lane 0), a tile read in place from the pool is
        // copied by all 32 lanes with cp.async.
        if (lane == 0) {
            mbar_expect_tx(bar(C::B_QFULL), NQC * QCH_BYTES);
            for (int c = 0; c < NQC; ++c)
                tma_load_3d(sQst + c * QCH_BYTES, &tm_q, 64 * (c < 4 ? 4 * half + c : 8), mt * BM, b,
                            bar(C::B_QFULL));
        }
        grid_dep_wait();
        // in place: pool row id of key lane of a tile, loaded a tile ahead
        // (absent entries read the pool's zero row)
        auto row_id = [&](int i) {
            const int j = k0 + i * BN + lane;
            return (INPLACE && i < ntiles && j < k1) ? p.resolved[(size_t)b * p.K + j] : -1;
        };
        int nxt_lo = row_id(0);
        int issued = 0;
        bool ok = true;
        for (int i = 0; i < ntiles; ++i) {
            const int g = i % NG;
            int go = 0;
            if (lane == 0) {
                const uint32_t ph = (uint32_t)(i / NG) & 1u;
                // tile groups 2-3 hold the staged Q until it has moved to TMEM
                go = (i != 2 || mbar_wait(bar(C::B_QREADY), 0)) &&
                     mbar_wait(bar(C::B_GEMPTY + g), ph ^ 1u) && !misc[1];
            }
            if (!__shfl_sync(0xffffffffu, go, 0)) {
                ok = false;
                break;
            }
            const uint32_t done = bar((FP8 ? C::B_GLANDED : C::B_GFULL) + g);
            if (INPLACE) {
                // keys 0-31 here, keys 32-63 by the key-visibility warp
                const int lo = nxt_lo >= 0 ? nxt_lo : p.zero_row;
                nxt_lo = row_id(i + 1);
                gather_keys(g, lo, 0);
                // arrives on the tile's barrier once this lane's copies have landed
                asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(done) : "memory");
            } else if (lane == 0) {
                // the four value chunks of the tile's 64 rows in one box
                // ([chunk][row][64]), the rope chunk in another
                mbar_expect_tx(done, NLC * (FP8 ? FCH_BYTES : KCH_BYTES));
                tma_load_4d(FP8 ? codes(g, 0) : slot(g, 0), &tm_kv, 0, k0 + i * BN, 4 * half, b, done);
                tma_load_4d(FP8 ? codes(g, 4) : slot(g, 4), &tm_kr, 0, k0 + i * BN, 8, b, done);
            }
            ++issued;
        }
        if (!ok && lane == 0) {
            fail();
            // let the copies this warp started land before the CTA exits
            mbar_wait(bar(C::B_QFULL), 0);
            for (int i = issued - 1; i >= 0 && i >= issued - NG; --i)
                mbar_wait(bar((FP8 ? C::B_GLANDED : C::B_GFULL) + i % NG), (i / NG) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID_QK = idesc_f16(1u, 0, BM, BN);
            constexpr uint32_t ID_PV = idesc_f16(1u, 1, BM, 256);
            bool ok = mbar_wait(bar(C::B_QREADY), 0);
            tc_fence_after();
            // PV of half tile u as soon as its P is ready (the second half
            // frees tile group u / 2 % NG for the next load); otherwise QK_j
            // once tile j is ready and the stagers have read S_{j-1}. Each
            // test is on the next phase of its barrier (the previous one has
            // completed, or the MMA that needs it would not have been
            // issued), so a parity test cannot see a stale phase. An idle
            // spell longer than 2 s gives up like every other wait.
            int u = 0, j = 0;
            uint64_t idle0 = 0;
            while (ok && u < nunits) {
                if (misc[1]) {
                    ok = false;
                    break;
                }
                if ((u >> 1) < j && mbar_test(bar(C::B_PFULL + (u & 1)), (uint32_t)(u >> 1) & 1u)) {
                    // O[128 x 256] += P_u[128 x 32] V_u[32 x 256]: keys 32h..32h+31 of the tile
                    tc_fence_after();
                    const int g = (u >> 1) % NG, h = u & 1;
                    const uint64_t vb = desc_sw128(slot(g, 0), KCH_BYTES, 1024);
                    const uint32_t lo = (uint32_t)vb + 256u * (uint32_t)h, hi = (uint32_t)(vb >> 32);
                    const uint32_t ap = tmem + TM_P + 16u * (uint32_t)h;
                    if (u == 0)
                        mma_ts<false>(tmem + TM_O, ap, lo, hi, ID_PV);
                    else
                        mma_ts<true>(tmem + TM_O, ap, lo, hi, ID_PV);
                    mma_ts<true>(tmem + TM_O, ap + 8u, lo + 128u, hi, ID_PV);  // 16 keys = 2 KB of V
                    if (h) mma_commit(bar(C::B_GEMPTY + g));
                    mma_commit(bar(C::B_PVDONE + h));
                    ++u;
                    idle0 = 0;
                    continue;
                }
                if (j < ntiles && mbar_test(bar(C::B_GFULL + j % NG), (uint32_t)(j / NG) & 1u) &&
                    (j == 0 || mbar_test(bar(C::B_SFREE), (uint32_t)(j - 1) & 1u))) {
                    // rows gathered by cp.async were written through the generic
                    // proxy; the MMA reads shared memory through the async proxy
                    if (INPLACE) fence_proxy_async();
                    tc_fence_after();
                    const uint64_t b0 = desc_sw128(slot(j % NG, 0), 16, 1024);
                    issue_qk(tmem + TM_S, tmem + TM_Q, (uint32_t)b0, (uint32_t)(b0 >> 32), ID_QK, half);
                    mma_commit(bar(C::B_SFULL));
                    ++j;
                    idle0 = 0;
                    continue;
                }
                const uint64_t now = globaltimer();
                if (!idle0)
                    idle0 = now;
                else if (now - idle0 > 2000000000ull)
                    ok = false;
                __nanosleep(32);
            }
            if (!ok) fail();
            // every MMA issued above has finished before TMEM and smem are released
            mma_commit(bar(C::B_DRAIN));
            mbar_wait(bar(C::B_DRAIN), 0);
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------ key visibility, row scales
        // Key j of a tile is seen by query token t iff its position is at most
        // L - T + t: store d = clamp(position - (L - T), 0, T), and d = T (seen
        // by none) for unresolved or absent entries; row t then masks d > t.
        // With one list per token (tpl > 1, T = 1) list b serves token b % tpl
        // of the request's tpl tokens, whose position is L - tpl + b % tpl.
        const int r = p.req_ids[b / p.tpl];
        const long long first = (long long)((r >= 0 && r < p.max_req) ? p.ctx[r] : 0) - p.T -
                                (p.tpl - 1 - b % p.tpl);
        const int32_t *res_b = p.resolved + (size_t)b * p.K;
        const int32_t *top_b = p.topk + (size_t)b * p.K;
        const float *gs = (FP8 && !INPLACE) ? p.gscale + (size_t)b * p.K : nullptr;
        int16_t *kvis = reinterpret_cast<int16_t *>(smem + C::OFF_KVIS);
        float *ksc = reinterpret_cast<float *>(smem + C::OFF_KSC);
        // Rows read in place: the row ids and positions of tile i + 1, and its
        // row scales (FP8, found through the row ids), are loaded while tile i
        // is written and copied, so no global-load latency sits between two
        // tiles of this warp. From the gathered buffer each tile's entries are
        // loaded after its slot is free (measured faster there).
        auto load_ids = [&](int i, int (&res)[2], int (&top)[2]) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // keys lane and lane + 32
                const int j = k0 + i * BN + lane + 32 * h;
                const bool in = i < ntiles && j < k1;
                res[h] = in ? res_b[j] : -1;
                top[h] = in ? top_b[j] : 0;
            }
        };
        auto load_scales = [&](int i, const int (&res)[2], float (&sc)[2]) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                sc[h] = 0.f;
                if (FP8 && res[h] >= 0) sc[h] = INPLACE ? p.pool_scales[res[h]] : gs[k0 + i * BN + lane + 32 * h];
            }
        };
        int nres[2] = {-1, -1}, ntop[2] = {0, 0};
        float nsc[2] = {0.f, 0.f};
        if (INPLACE) {
            load_ids(0, nres, ntop);
            load_scales(0, nres, nsc);
        }
        bool ok = true;
        for (int i = 0; i < ntiles; ++i) {
            const int g = i % NG;
            const uint32_t ph = (uint32_t)(i / NG) & 1u;
            int cres[2] = {nres[0], nres[1]}, ctop[2] = {ntop[0], ntop[1]};
            float csc[2] = {nsc[0], nsc[1]};
            if (INPLACE) load_ids(i + 1, nres, ntop);
            // the slot's previous tile is finished (its stagers and softmax read these rings)
            if (ok) ok = mbar_wait(bar(C::B_GEMPTY + g), ph ^ 1u) && !misc[1];
            if (!INPLACE) {
                load_ids(i, cres, ctop);
                load_scales(i, cres, csc);
            }
            int dm[2] = {0, 0}, rr[2] = {-1, -1};
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                long long d = (long long)ctop[h] - first;
                d = d < 0 ? 0 : (d > p.T ? p.T : d);
                const int v = cres[h] >= 0 ? (int)d : p.T;
                dm[h] = v;
                rr[h] = cres[h];
                if (ok) {
                    kvis[g * BN + lane + 32 * h] = (int16_t)v;
                    if (FP8) ksc[g * BN + lane + 32 * h] = csc[h];
                }
            }
            if (INPLACE) {
                // keys 32-63 of the tile from the pool (keys 0-31: the producer);
                // tile groups 2-3 hold the staged Q until it has moved to TMEM
                if (ok && i == 2) ok = mbar_wait(bar(C::B_QREADY), 0);
                if (__all_sync(0xffffffffu, ok)) {
                    gather_keys(g, rr[1] >= 0 ? rr[1] : p.zero_row, 32);
                    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(
                                     bar((FP8 ? C::B_GLANDED : C::B_GFULL) + g))
                                 : "memory");
                }
            }
            // the largest d of each half tile: rows with t >= it skip the mask
            const int d0 = __reduce_max_sync(0xffffffffu, dm[0]);
            const int d1 = __reduce_max_sync(0xffffffffu, dm[1]);
            if (ok && lane == 0) {
                tdmax[2 * g] = d0;
                tdmax[2 * g + 1] = d1;
            }
            mbar_arrive(bar(C::B_KVIS + g));
            if (INPLACE && FP8) load_scales(i + 1, nres, nsc);
        }
        if (INPLACE) asm volatile("cp.async.wait_all;" ::: "memory");  // own copies landed before exit
        if (!ok) fail();
    } else if (warp == 3) {
        // ------------------------------------------------------------ courier
        // Sends each staged half tile to the peer, in order, once the peer has
        // read the half tile sent two before into the same buffer; arms this
        // CTA's barrier for the peer's partial of the same half tile; tells
        // the stagers when the copy has read X_out.
        if (lane == 0) {
            const uint32_t peer_xin = hs::dsmem_map(smem + C::OFF_XIN, peer);
            const uint32_t peer_xfull = hs::dsmem_map(smem + C::OFF_BAR + 8 * C::B_XFULL, peer);
            bool ok = true;
            for (int u = 0; u < nunits; ++u) {
                const uint32_t x = (uint32_t)(u & 1);
                if (ok) ok = mbar_wait(bar(C::B_STAGED + x), (uint32_t)(u >> 1) & 1u);
                if (ok && u >= 2)
                    ok = mbar_wait_cluster(bar(C::B_XTAKEN + x), (uint32_t)((u - 2) >> 1) & 1u);
                if (ok && !misc[1]) {
                    mbar_expect_tx(bar(C::B_XFULL + x), X_BYTES);  // arms this CTA's receive of u
                    asm volatile(
                        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes"
                        " [%0], [%1], %2, [%3];" ::"r"(peer_xin + x * X_BYTES),
                        "r"(sXout + x * X_BYTES), "r"((uint32_t)X_BYTES), "r"(peer_xfull + 8u * x)
                        : "memory");
                    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                }
                mbar_arrive(bar(C::B_XOUTDONE + x));
            }
            if (!ok) fail();
        }
    } else {
        // ------------------------------------------------------------ stagers and softmax
        // Thread row = TMEM lane (warp w reaches lanes 32 (w % 4) .. + 31).
        const bool stager = warp < 8;
        const int wq = warp & 3;
        const int row = wq * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
        bool ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_QFULL), 0));
        if (ok) {
            // this thread's row of the staged Q into its TMEM lane: stagers
            // value chunks 0 and 2 and this CTA's half of the rope chunk,
            // softmax threads value chunks 1 and 3
            for (int c = stager ? 0 : 1; c < 4; c += 2) {
                uint32_t q[32];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const uint4 v = ld_shared_v4(sQst + c * QCH_BYTES + x_off(row, u));
                    q[4 * u] = v.x;
                    q[4 * u + 1] = v.y;
                    q[4 * u + 2] = v.z;
                    q[4 * u + 3] = v.w;
                }
                HS_TMEM_ST32(tmem + lane_off + TM_Q + 32u * (uint32_t)c, q);
            }
            if (stager) {
                uint32_t q[16];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint4 v = ld_shared_v4(sQst + 4 * QCH_BYTES + x_off(row, 4 * half + u));
                    q[4 * u] = v.x;
                    q[4 * u + 1] = v.y;
                    q[4 * u + 2] = v.z;
                    q[4 * u + 3] = v.w;
                }
                HS_TMEM_ST16(tmem + lane_off + TM_Q + 128u, q);
            }
            tmem_wait_st();
        }
        fence_proxy_async();  // the staging space is refilled by TMA next
        tc_fence_before();
        mbar_arrive(bar(C::B_QREADY));

        // Epilogue: O / l as BF16 through shared memory (the ring is idle once
        // the last PV is done): 32-column TMEM loads into 64-column boxes of
        // the 128-byte-swizzled layout, then one TMA store per box (rows past
        // M are clipped by the tensor map). BF16 rows: the softmax warp of a
        // lane quarter writes columns 0-127 of its 32 rows and the stager warp
        // of the same quarter, idle by then, columns 128-255; the softmax warp
        // hands 1/l (-1 after a failed wait) to it through shared memory and a
        // named barrier of the two warps. FP8 rows: the stagers may still be
        // converting codes, so the softmax warp writes all 256 columns.
        float *s_inv = reinterpret_cast<float *>(smem + C::OFF_RING + 65536);  // [BM], past the staging
        auto store_o = [&](int cc0, int ncc, float inv) {
            const uint32_t stg = sR + (uint32_t)wq * 16384u;
#pragma unroll 1
            for (int cc = cc0; cc < cc0 + ncc; ++cc) {
                uint32_t o[32];
                HS_TMEM_LD32(tmem + lane_off + TM_O + 32 * cc, o);
                HS_TMEM_WAIT_LD32(o);
                const uint32_t box = stg + (uint32_t)(cc >> 1) * 4096u + (uint32_t)lane * 128u;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w[e] = pack_bf16(__uint_as_float(o[8 * q + 2 * e]) * inv,
                                         __uint_as_float(o[8 * q + 2 * e + 1]) * inv);
                    const int c = (cc & 1) * 4 + q;
                    st_shared_v4(box + (uint32_t)((c ^ (lane & 7)) << 4), w[0], w[1], w[2], w[3]);
                }
            }
            fence_proxy_async();  // the TMA stores read what the threads wrote
            __syncwarp();
            if (lane == 0) {
                const int zb = p.nsplit == 1 ? b : split * p.B + b;
                for (int cg = cc0 >> 1; cg < (cc0 + ncc) >> 1; ++cg)
                    tma_store_3d(&tm_o, stg + (uint32_t)cg * 4096u, half * 256 + cg * 64,
                                 mt * BM + wq * 32, zb);
                asm volatile("cp.async.bulk.commit_group;" ::: "memory");
                // the stores have read shared memory before the CTA may exit
                asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
            }
            __syncwarp();
        };

        if (stager) {
            // ------------------------------------------------ stagers (FP8: and converters)
            // FP8, tile i: read every code of the group (20 KB, ten 16-byte
            // units per thread), wait until all stagers have read theirs,
            // then write the BF16 rows of all five chunks over the group (the
            // rows of a chunk overlap the codes of that chunk and of lower
            // ones). Tiles 0 and 1 are converted first, tile j + 2 after tile
            // j has been staged, so a tile is ready two tiles before its QK.
            // Every stager reaches the named barrier on every converted tile.
            auto convert = [&](int i) {
                const int g = i % NG;
                if (ok) ok = __all_sync(0xffffffffu,
                                        mbar_wait(bar(C::B_GLANDED + g), (uint32_t)(i / NG) & 1u) &&
                                            !misc[1]);
                uint4 cw[CVT_UNITS];
                if (ok) {
#pragma unroll
                    for (int k = 0; k < CVT_UNITS; ++k)
                        cw[k] = ld_shared_v4(codes(g, 0) + 16u * (row + NCVT * k));
                }
                named_bar_sync(3, NCVT);
                if (ok) {
#pragma unroll
                    for (int k = 0; k < CVT_UNITS; ++k) {
                        const int u = row + NCVT * k;  // 16-byte unit of codes: chunk, key, part
                        const int lc = u >> 8, key = (u >> 2) & 63, part = u & 3;
                        uint32_t o[8];
                        e4m3x4_to_bf16(cw[k].x, o[0], o[1]);
                        e4m3x4_to_bf16(cw[k].y, o[2], o[3]);
                        e4m3x4_to_bf16(cw[k].z, o[4], o[5]);
                        e4m3x4_to_bf16(cw[k].w, o[6], o[7]);
                        const uint32_t dst = slot(g, lc) + key * 128;
                        st_shared_v4(dst + (((2 * part) ^ (key & 7)) << 4), o[0], o[1], o[2], o[3]);
                        st_shared_v4(dst + (((2 * part + 1) ^ (key & 7)) << 4), o[4], o[5], o[6], o[7]);
                    }
                    fence_proxy_async();  // the MMAs read these rows
                }
                mbar_arrive(bar(C::B_GFULL + g));
            };
            if (FP8) {
                for (int i = 0; i < 2 && i < ntiles; ++i) convert(i);
            }
            // Tile j: read the partial S from TMEM, free S, and write each
            // half (32 keys) as f32 of S * sm_scale * log2(e) (times the row
            // scale for FP8) to X_out[u & 1] once half tile u - 2 is done
            // with that buffer (read by this CTA's softmax and copied out).
            for (int j = 0; j < ntiles; ++j) {
                const int g = j % NG;
                float sv[64];
                if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_SFULL), (uint32_t)j & 1u));
                if (ok) {
                    tc_fence_after();
                    uint32_t ra[32], rb[32];
                    HS_TMEM_LD32(tmem + lane_off + TM_S, ra);
                    HS_TMEM_LD32(tmem + lane_off + TM_S + 32, rb);
                    HS_TMEM_WAIT_LD32(ra);
                    HS_TMEM_WAIT_LD32(rb);
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        sv[e] = __uint_as_float(ra[e]);
                        sv[32 + e] = __uint_as_float(rb[e]);
                    }
                }
                tc_fence_before();
                mbar_arrive(bar(C::B_SFREE));  // QK of tile j + 1 may overwrite S
                if (FP8 && ok)
                    ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_KVIS + g), (uint32_t)(j / NG) & 1u));
                if (ok) {
                    if (FP8) {
#pragma unroll
                        for (int q = 0; q < 16; ++q) {
                            const float4 s4 = ld_shared_f4(sKsc + (uint32_t)(g * BN * 4 + 16 * q));
                            sv[4 * q] *= p.scale_log2 * s4.x;
                            sv[4 * q + 1] *= p.scale_log2 * s4.y;
                            sv[4 * q + 2] *= p.scale_log2 * s4.z;
                            sv[4 * q + 3] *= p.scale_log2 * s4.w;
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 64; ++e) sv[e] *= p.scale_log2;
                    }
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int u = 2 * j + h;
                    const uint32_t x = (uint32_t)(u & 1);
                    if (ok && u >= 2) {
                        // X_out[x] was read by this CTA's softmax and by the copy to the peer
                        const uint32_t ph = (uint32_t)((u - 2) >> 1) & 1u;
                        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_READ + x), ph) &&
                                                         mbar_wait(bar(C::B_XOUTDONE + x), ph));
                    }
                    if (ok) {
                        const uint32_t xo = sXout + x * X_BYTES;
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            st_shared_v4(xo + x_off(row, c), __float_as_uint(sv[32 * h + 4 * c]),
                                         __float_as_uint(sv[32 * h + 4 * c + 1]),
                                         __float_as_uint(sv[32 * h + 4 * c + 2]),
                                         __float_as_uint(sv[32 * h + 4 * c + 3]));
                        fence_proxy_async();  // the courier's bulk copy reads it
                    }
                    mbar_arrive(bar(C::B_STAGED + x));
                }
                if (FP8 && j + 2 < ntiles) convert(j + 2);
            }
            if (!FP8) {
                named_bar_sync(4 + wq, 64);  // 1/l of this quarter's rows from its softmax warp
                const float inv = s_inv[row];
                if (inv >= 0.f) {
                    tc_fence_after();
                    store_o(4, 4, inv);
                }
            }
        } else {
            // ------------------------------------------------ softmax, PV, epilogue
            const int mg = mt * BM + row;
            const bool vrow = mg < p.M;
            const int t = vrow ? mg / p.H : 0;  // query token of this row
            const uint32_t peer_xtaken = hs::dsmem_map(smem + C::OFF_BAR + 8 * C::B_XTAKEN, peer);
            float m2 = -INFINITY, l = 0.f;
            // Every softmax thread runs every half tile; after a failed wait
            // the remaining work is skipped.
            for (int u = 0; u < nunits; ++u) {
                const uint32_t x = (uint32_t)(u & 1);
                const int j = u >> 1, h = u & 1, g = j % NG;
                float s[32];
                if (ok) ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_XFULL + x), (u >> 1) & 1));
                if (ok) {
                    // S = own partial + the peer's partial; f32 addition is
                    // commutative, so the peer, adding them the other way
                    // round, gets the same bits
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const float4 a = ld_shared_f4(sXout + x * X_BYTES + x_off(row, c));
                        const float4 v = ld_shared_f4(sXin + x * X_BYTES + x_off(row, c));
                        s[4 * c] = a.x + v.x;
                        s[4 * c + 1] = a.y + v.y;
                        s[4 * c + 2] = a.z + v.z;
                        s[4 * c + 3] = a.w + v.w;
                    }
                }
                // X_in[x] and X_out[x] read by this warp: lane 0 frees them for the
                // stagers and the peer, one arrive per warp (the reads above have
                // returned their values, so an arrive without a cluster-scope
                // release is enough to let the peer overwrite)
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(bar(C::B_READ + x));
                    mbar_arrive_peer(peer_xtaken + 8u * x);
                }
                if (ok && h == 0)
                    ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_KVIS + g), (uint32_t)(j / NG) & 1u));
                uint32_t pk[16];
                float alpha = 1.f;
                bool need = false;
                if (ok) {
                    if (!__all_sync(0xffffffffu, tdmax[2 * g + h] <= t)) {
                        // some key of this half tile is hidden from some row of this warp
#pragma unroll
                        for (int q = 0; q < 4; ++q) {  // 8 keys per 16 bytes, lower key in the low half
                            const uint4 kv = ld_shared_v4(sKvis + (uint32_t)(g * BN * 2 + 64 * h + 16 * q));
                            const uint32_t w[4] = {kv.x, kv.y, kv.z, kv.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int d0 = (int)(w[e] & 0xffffu), d1 = (int)(w[e] >> 16);
                                s[8 * q + 2 * e] = d0 <= t ? s[8 * q + 2 * e] : -INFINITY;
                                s[8 * q + 2 * e + 1] = d1 <= t ? s[8 * q + 2 * e + 1] : -INFINITY;
                            }
                        }
                    }
                    // tree reduction: no long dependency chain
                    float mx[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        mx[e] = fmaxf(fmaxf(s[e], s[e + 8]), fmaxf(s[e + 16], s[e + 24]));
#pragma unroll
                    for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
                        for (int e = 0; e < w; ++e) mx[e] = fmaxf(mx[e], mx[e + w]);
                    const float tmax = mx[0];
                    if (u == 0) {
                        m2 = tmax;
                    } else if (tmax > m2 + TAU2) {
                        need = true;
                        alpha = exp2f(m2 - tmax);
                        l *= alpha;
                        m2 = tmax;
                    }
                    const float mref = (m2 == -INFINITY) ? 0.f : m2;
                    float ls[4] = {0.f, 0.f, 0.f, 0.f};
                    if (FP8) {
                        // P = probability x the key's row scale (the value rows are codes)
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float4 s4 = ld_shared_f4(sKsc + (uint32_t)(g * BN * 4 + 128 * h + 16 * q));
                            const float a0 = exp2f(s[4 * q] - mref), a1 = exp2f(s[4 * q + 1] - mref);
                            const float a2 = exp2f(s[4 * q + 2] - mref), a3 = exp2f(s[4 * q + 3] - mref);
                            ls[q & 3] += (a0 + a1) + (a2 + a3);
                            pk[2 * q] = pack_bf16(a0 * s4.x, a1 * s4.y);
                            pk[2 * q + 1] = pack_bf16(a2 * s4.z, a3 * s4.w);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float a = exp2f(s[2 * e] - mref), c = exp2f(s[2 * e + 1] - mref);
                            ls[e & 3] += a + c;
                            pk[e] = pack_bf16(a, c);
                        }
                    }
                    l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                    // this half's P columns were last read by PV of u - 2
                    if (u >= 2)
                        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_PVDONE + h),
                                                               (uint32_t)((u - 2) >> 1) & 1u));
                    // a rescale of O needs every earlier PV done (PV of u - 1 is the last)
                    if (ok && u >= 1 && __any_sync(0xffffffffu, need))
                        ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_PVDONE + (h ^ 1)),
                                                               (uint32_t)((u - 1) >> 1) & 1u));
                }
                if (ok) {
                    tc_fence_after();
                    HS_TMEM_ST16(tmem + lane_off + TM_P + 16u * (uint32_t)h, pk);
                    if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
                        for (int cc = 0; cc < 8; ++cc) {
                            uint32_t o[32];
                            const uint32_t tO = tmem + lane_off + TM_O + 32 * cc;
                            HS_TMEM_LD32(tO, o);
                            HS_TMEM_WAIT_LD32(o);
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            HS_TMEM_ST32(tO, o);
                        }
                    }
                    tmem_wait_st();
                }
                tc_fence_before();
                mbar_arrive(bar(C::B_PFULL + h));  // P_u (and a rescaled O) complete in TMEM
            }
            if (ok && nunits > 0) {
                // the last PV's completion covers every earlier one
                ok = __all_sync(0xffffffffu, mbar_wait(bar(C::B_PVDONE + ((nunits - 1) & 1)),
                                                       (uint32_t)((nunits - 1) >> 1) & 1u));
                tc_fence_after();
            }
            if (!ok) fail();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const size_t orow = (size_t)b * p.M + mg;
            if (!FP8) {
                s_inv[row] = ok ? inv : -1.f;
                named_bar_sync(4 + wq, 64);
            }
            if (ok) store_o(0, FP8 ? 8 : 4, inv);
            if (vrow && half == 0) {
                const float lse = (ok && l > 0.f) ? (m2 + __log2f(l)) * 0.69314718055994531f : -INFINITY;
                if (p.nsplit == 1)
                    p.lse[orow] = lse;
                else
                    p.ws_lse[((size_t)split * p.B + b) * p.M + mg] = lse;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
    cluster_sync_all();  // no CTA leaves while its peer may still write to it
}

// Merges the KV-split partials: out = sum_s w_s O_s / sum_s w_s, w_s = exp(lse_s - max).
// One task per 8 output columns of a row (64 tasks per row), two tasks per
// thread a grid apart: every load of both is issued before any is used, so the
// whole merge is about one round trip to memory, with half as many blocks to
// place once the decode's CTAs leave their SMs.
constexpr int CMB_TPT = 2;
__device__ __forceinline__ void combine_store(__nv_bfloat16 *__restrict__ out, float *__restrict__ lse,
                                              int row, int c8, const float (&acc)[8], float wsum, float mx) {
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    *reinterpret_cast<uint4 *>(out + (size_t)row * 512 + c8) =
        make_uint4(pack_bf16(acc[0] * inv, acc[1] * inv), pack_bf16(acc[2] * inv, acc[3] * inv),
                   pack_bf16(acc[4] * inv, acc[5] * inv), pack_bf16(acc[6] * inv, acc[7] * inv));
    if (c8 == 0) lse[row] = wsum > 0.f ? mx + __logf(wsum) : -INFINITY;
}
__global__ void __launch_bounds__(256)
combine_kernel(const __nv_bfloat16 *__restrict__ ws_o, const float *__restrict__ ws_lse, int nsplit,
               int rows, __nv_bfloat16 *__restrict__ out, float *__restrict__ lse) {
    grid_dep_wait();  // the decode grid's partials are complete
    const int t0 = blockIdx.x * 256 + threadIdx.x, stride = gridDim.x * 256;
    constexpr int MAXS = 4;
    if (nsplit <= MAXS) {
        float ls[CMB_TPT][MAXS];
        uint4 u[CMB_TPT][MAXS];
#pragma unroll
        for (int q = 0; q < CMB_TPT; ++q) {
            const int t = t0 + q * stride, row = t >> 6, c8 = (t & 63) * 8;
#pragma unroll
            for (int s = 0; s < MAXS; ++s) {
                ls[q][s] = -INFINITY;
                u[q][s] = make_uint4(0u, 0u, 0u, 0u);
                if (row < rows && s < nsplit) {
                    ls[q][s] = ws_lse[(size_t)s * rows + row];
                    u[q][s] = *reinterpret_cast<const uint4 *>(ws_o + ((size_t)s * rows + row) * 512 + c8);
                }
            }
        }
#pragma unroll
        for (int q = 0; q < CMB_TPT; ++q) {
            const int t = t0 + q * stride, row = t >> 6, c8 = (t & 63) * 8;
            if (row >= rows) continue;
            float acc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = 0.f;
            float wsum = 0.f, mx = -INFINITY;
#pragma unroll
            for (int s = 0; s < MAXS; ++s) mx = fmaxf(mx, ls[q][s]);
            if (mx != -INFINITY) {
#pragma unroll
                for (int s = 0; s < MAXS; ++s) {
                    const float w = ls[q][s] == -INFINITY ? 0.f : __expf(ls[q][s] - mx);
                    wsum += w;
                    const uint32_t v[4] = {u[q][s].x, u[q][s].y, u[q][s].z, u[q][s].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        acc[2 * e] += w * __uint_as_float(v[e] << 16);
                        acc[2 * e + 1] += w * __uint_as_float(v[e] & 0xffff0000u);
                    }
                }
            }
            combine_store(out, lse, row, c8, acc, wsum, mx);
        }
    } else {
        for (int q = 0; q < CMB_TPT; ++q) {
            const int t = t0 + q * stride, row = t >> 6, c8 = (t & 63) * 8;
            if (row >= rows) continue;
            float acc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = 0.f;
            float wsum = 0.f, mx = -INFINITY;
            for (int s = 0; s < nsplit; ++s) mx = fmaxf(mx, ws_lse[(size_t)s * rows + row]);
            if (mx != -INFINITY) {
#pragma unroll 4
                for (int s = 0; s < nsplit; ++s) {
                    const float l = ws_lse[(size_t)s * rows + row];
                    const uint4 v4 = *reinterpret_cast<const uint4 *>(ws_o + ((size_t)s * rows + row) * 512 + c8);
                    const float w = l == -INFINITY ? 0.f : __expf(l - mx);
                    wsum += w;
                    const uint32_t v[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        acc[2 * e] += w * __uint_as_float(v[e] << 16);
                        acc[2 * e + 1] += w * __uint_as_float(v[e] & 0xffff0000u);
                    }
                }
            }
            combine_store(out, lse, row, c8, acc, wsum, mx);
        }
    }
}

// ---------------------------------------------------------------- host side
struct Plan {
    int M, mtiles, nsplit, kps;
    size_t ws_o_bytes, ws_bytes;
};

int sm_count() {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (!n) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 148;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

Plan make_plan(int B, int T, int H, int K) {
    Plan pl{};
    pl.M = T * H;
    pl.mtiles = (pl.M + BM - 1) / BM;
    const int tiles = (K + BN - 1) / BN;
    const int base = B * pl.mtiles * 2;
    int ns = base > 0 ? sm_count() / base : 1;
    if (ns < 1) ns = 1;
    const int max_ns = tiles / 2 > 1 ? tiles / 2 : 1;  // at least two key tiles per split
    if (ns > max_ns) ns = max_ns;
    const int per = (tiles + ns - 1) / ns;
    pl.kps = per * BN;
    pl.nsplit = (K + pl.kps - 1) / pl.kps;
    if (pl.nsplit > 1) {
        const size_t rows = (size_t)pl.nsplit * B * pl.M;
        pl.ws_o_bytes = (rows * 512 * sizeof(__nv_bfloat16) + 255) & ~size_t(255);
        pl.ws_bytes = pl.ws_o_bytes + ((rows * sizeof(float) + 255) & ~size_t(255));
    }
    return pl;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

// Map [batch][rows][inner] (rank 3) or [rows][inner] (rank 2, batch 1) with a
// (box_inner x box_rows) box.
bool make_map(CUtensorMap *m, CUtensorMapDataType dt, const void *ptr, uint64_t inner,
              uint64_t rows, uint64_t batch, uint64_t row_bytes, uint32_t box_inner,
              uint32_t box_rows, CUtensorMapSwizzle sw, uint32_t rank = 3) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {inner, rows, batch};
    cuuint64_t strides[2] = {row_bytes, row_bytes * rows};
    cuuint32_t box[3] = {box_inner, box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(m, dt, rank, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Rows of 9 chunks of 64 elements, as a 4-D map (element, row, chunk,
// request) with a (64 x BN x nchunks x 1) box.
bool make_chunk_map(CUtensorMap *m, CUtensorMapDataType dt, const void *ptr, uint64_t rows,
                    uint64_t batch, uint64_t row_bytes, uint64_t chunk_bytes, CUtensorMapSwizzle sw,
                    uint32_t nchunks) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {64, rows, 9, batch};
    cuuint64_t strides[3] = {row_bytes, chunk_bytes, row_bytes * rows};
    cuuint32_t box[4] = {64, (cuuint32_t)BN, nchunks, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return fn(m, dt, 4, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// cudaFuncSetAttribute once per device and kernel variant (the opt-in to
// more than 48 KB of shared memory is per device).
template <bool FP8, bool INPLACE>
hs_status set_smem_attr(int dev) {
    static std::atomic<int> state[64];  // 0 unknown, 1 set
    if (dev < 0 || dev >= 64) return HS_ERR_UNSUPPORTED;
    if (state[dev].load(std::memory_order_acquire) == 1) return HS_OK;
    HS_CUDA_TRY(cudaFuncSetAttribute(decode_tc_kernel<FP8, INPLACE>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_ALLOC));
    state[dev].store(1, std::memory_order_release);
    return HS_OK;
}

template <bool FP8, bool INPLACE>
hs_status launch_decode(dim3 grid, cudaStream_t s, const CUtensorMap &tq, const CUtensorMap &tkv,
                        const CUtensorMap &tkr, const CUtensorMap &to, const DecParams &p) {
    int dev = 0;
    HS_CUDA_TRY(cudaGetDevice(&dev));
    const hs_status st = set_smem_attr<FP8, INPLACE>(dev);
    if (st != HS_OK) return st;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(Threads<FP8>::N, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_ALLOC;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;  // the two output halves of one work unit
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // may start before the previous kernel ends (it waits in griddepcontrol.wait)
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, decode_tc_kernel<FP8, INPLACE>, tq, tkv, tkr, to, p) == cudaSuccess
               ? HS_OK
               : HS_ERR_CUDA;
}

}  // namespace

extern "C" size_t hs_decode_workspace_bytes(int32_t B, int32_t T, int32_t H, int32_t K) {
    if (B < 1 || T < 1 || H < 1 || K < 1) return 0;
    return make_plan(B, T, H, K).ws_bytes;
}

namespace {
// B lists of T query tokens each; tpl > 1 (with T = 1): B / tpl requests whose
// tpl tokens each have their own list.
hs_status decode_entry(hs_pool_t pool, int32_t B, int32_t T, int32_t tpl, int32_t H, int32_t K,
                       const void *d_q, const void *d_gathered, const float *d_gathered_scale,
                       const int32_t *d_resolved, const int32_t *d_topk_idx,
                       const int32_t *d_req_ids, float sm_scale, void *d_out, float *d_lse,
                       void *d_workspace, size_t ws_bytes, void *stream) {
    if (!pool || !d_q || !d_resolved || !d_topk_idx || !d_req_ids || !d_out || !d_lse)
        return HS_ERR_INVALID_ARG;
    if (B < 0 || T < 1 || T > 32767 || H < 1 || K < 1 || B > 65535 ||
        (int64_t)T * H > (int64_t)BM * 65535)
        return HS_ERR_INVALID_ARG;
    const bool fp8 = pool->cfg.dtype == HS_FP8_E4M3_ROWSCALE;
    // rows from the gathered buffer (with their scales for FP8), or in place
    // from the pool by row id (no gathered buffer and no scales)
    const bool inplace = d_gathered == nullptr;
    if (inplace ? d_gathered_scale != nullptr : fp8 != (d_gathered_scale != nullptr))
        return HS_ERR_INVALID_ARG;
    if (((uintptr_t)d_q | (uintptr_t)d_gathered | (uintptr_t)d_out) & 15u) return HS_ERR_INVALID_ARG;
    if (B == 0) return HS_OK;
    const Plan pl = make_plan(B, T, H, K);
    if (pl.nsplit > 1 && (!d_workspace || ws_bytes < pl.ws_bytes || ((uintptr_t)d_workspace & 255u)))
        return HS_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    CUtensorMap tq, tkv, tkr;
    if (!make_map(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, d_q, hs::kDim, pl.M, B, 2 * hs::kDim, 64,
                  BM, CU_TENSOR_MAP_SWIZZLE_128B))
        return HS_ERR_CUDA;
    bool ok_k;
    if (inplace) {
        // not read: rows read in place are copied from the pool with cp.async
        tkv = tq;
        tkr = tq;
        ok_k = true;
    } else {
        // [B][K][9 chunks][64] viewed as (column, row, chunk, request): one box
        // brings four value chunks of 64 rows (chunk-major in shared memory),
        // another the rope chunk
        const auto dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        const uint64_t rb = fp8 ? hs::kDim : 2 * hs::kDim, cb = fp8 ? 64 : 128;
        const auto sw = fp8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B;
        ok_k = make_chunk_map(&tkv, dt, d_gathered, K, B, rb, cb, sw, 4) &&
               make_chunk_map(&tkr, dt, d_gathered, K, B, rb, cb, sw, 1);
    }
    if (!ok_k) return HS_ERR_CUDA;

    DecParams p{};
    p.resolved = d_resolved;
    p.topk = d_topk_idx;
    p.req_ids = d_req_ids;
    p.ctx = pool->d_ctx;
    p.gscale = d_gathered_scale;
    p.pool_scales = pool->d_scales;
    p.zero_row = (int)(pool->cfg.n_gpu_blocks * hs::kPage);
    p.pool_rows = pool->d_rows;
    p.out = static_cast<__nv_bfloat16 *>(d_out);
    p.lse = d_lse;
    p.ws_o = pl.nsplit > 1 ? static_cast<__nv_bfloat16 *>(d_workspace) : nullptr;
    p.ws_lse = pl.nsplit > 1
                   ? reinterpret_cast<float *>(static_cast<uint8_t *>(d_workspace) + pl.ws_o_bytes)
                   : nullptr;
    p.err = pool->d_err;
    p.B = B;
    p.T = T;
    p.H = H;
    p.K = K;
    p.M = pl.M;
    p.nsplit = pl.nsplit;
    p.kps = pl.kps;
    p.max_req = pool->cfg.max_requests;
    p.tpl = tpl;
    p.scale_log2 = sm_scale * 1.4426950408889634f;

    const dim3 grid(2 * pl.nsplit, pl.mtiles, B);
    // the output (one split) or the split partials, [batch][M][512] BF16, in
    // 64-column x 32-row boxes
    CUtensorMap to;
    if (!make_map(&to, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, pl.nsplit == 1 ? d_out : d_workspace, 512,
                  pl.M, (uint64_t)B * pl.nsplit, 1024, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B))
        return HS_ERR_CUDA;
    const hs_status st = fp8 ? (inplace ? launch_decode<true, true>(grid, s, tq, tkv, tkr, to, p)
                                        : launch_decode<true, false>(grid, s, tq, tkv, tkr, to, p))
                             : (inplace ? launch_decode<false, true>(grid, s, tq, tkv, tkr, to, p)
                                        : launch_decode<false, false>(grid, s, tq, tkv, tkr, to, p));
    if (st != HS_OK) return st;
    if (pl.nsplit > 1) {
        const int rows = B * pl.M;
        cudaLaunchConfig_t cc = {};
        cc.gridDim = dim3((rows + 4 * CMB_TPT - 1) / (4 * CMB_TPT), 1, 1);  // 4 rows per block and task
        cc.blockDim = dim3(256, 1, 1);
        cc.stream = s;
        cudaLaunchAttribute ca[1];
        ca[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        ca[0].val.programmaticStreamSerializationAllowed = 1;
        cc.attrs = ca;
        cc.numAttrs = 1;
        if (cudaLaunchKernelEx(&cc, combine_kernel, (const __nv_bfloat16 *)p.ws_o, (const float *)p.ws_lse,
                               pl.nsplit, rows, p.out, d_lse) != cudaSuccess)
            return HS_ERR_CUDA;
    }
    return HS_OK;
}
}  // namespace

extern "C" hs_status hs_sparse_mla_decode(hs_pool_t pool, int32_t B, int32_t T, int32_t H, int32_t K,
                                          const void *d_q, const void *d_gathered,
                                          const float *d_gathered_scale, const int32_t *d_resolved,
                                          const int32_t *d_topk_idx, const int32_t *d_req_ids,
                                          float sm_scale, void *d_out, float *d_lse,
                                          void *d_workspace, size_t ws_bytes, void *stream) {
    return decode_entry(pool, B, T, 1, H, K, d_q, d_gathered, d_gathered_scale, d_resolved,
                        d_topk_idx, d_req_ids, sm_scale, d_out, d_lse, d_workspace, ws_bytes,
                        stream);
}

extern "C" hs_status hs_sparse_mla_decode_per_token(
    hs_pool_t pool, int32_t B, int32_t T, int32_t H, int32_t K, const void *d_q,
    const void *d_gathered, const float *d_gathered_scale, const int32_t *d_resolved,
    const int32_t *d_topk_idx, const int32_t *d_req_ids, float sm_scale, void *d_out, float *d_lse,
    void *d_workspace, size_t ws_bytes, void *stream) {
    if (B < 0 || T < 1 || (int64_t)B * T > 65535) return HS_ERR_INVALID_ARG;
    // request b's T lists are lists b*T .. b*T+T-1 of one query token each
    return decode_entry(pool, B * T, 1, T, H, K, d_q, d_gathered, d_gathered_scale, d_resolved,
                        d_topk_idx, d_req_ids, sm_scale, d_out, d_lse, d_workspace, ws_bytes,
                        stream);
}

// ---------------------------------------------------------------- no-allocation variant
// Decode for callers that cannot allocate device memory themselves: a host
// engine that has reserved the device's memory for its own KV pool and hands
// this library only the tensors it owns, or a C plugin that receives device
// pointers but has no allocator. The split-KV partials live in a fixed array in
// this module's device memory instead of a caller-provided workspace. Every
// GPU that loads the library holds the array until the process exits.
static __device__ __align__(256) unsigned char hs_static_decode_ws[HS_STATIC_DECODE_WS_BYTES];

namespace {
// device address of hs_static_decode_ws, looked up once per device (the
// lookup is idempotent, so two threads racing on a first call store the same
// address)
std::atomic<void *> g_static_ws[64];
}

extern "C" hs_status hs_sparse_mla_decode_static_ws(
    hs_pool_t pool, int32_t B, int32_t T, int32_t H, int32_t K, const void *d_q,
    const void *d_gathered, const float *d_gathered_scale, const int32_t *d_resolved,
    const int32_t *d_topk_idx, const int32_t *d_req_ids, float sm_scale, void *d_out, float *d_lse,
    void *stream) {
    if (!pool || B < 0 || T < 1 || H < 1 || K < 1) return HS_ERR_INVALID_ARG;
    if (B > 0 && hs_decode_workspace_bytes(B, T, H, K) > HS_STATIC_DECODE_WS_BYTES)
        return HS_ERR_CAPACITY;
    int dev = 0;
    HS_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return HS_ERR_UNSUPPORTED;
    void *ws = g_static_ws[dev].load(std::memory_order_acquire);
    if (!ws) {
        // host code cannot use the array's name as a device address: ask the
        // runtime for this device's copy (the current device)
        HS_CUDA_TRY(cudaGetSymbolAddress(&ws, hs_static_decode_ws));
        if (!ws) return HS_ERR_CUDA;
        g_static_ws[dev].store(ws, std::memory_order_release);
    }
    return hs_sparse_mla_decode(pool, B, T, H, K, d_q, d_gathered, d_gathered_scale, d_resolved,
                                d_topk_idx, d_req_ids, sm_scale, d_out, d_lse, ws,
                                HS_STATIC_DECODE_WS_BYTES, stream);
}

// ---------------------------------------------------------------- bounded-wait check
namespace {
// One thread waits on an mbarrier phase that nothing completes, with the same
// bounded wait the decode pipeline uses; it must give up after `limit_ns`.
__global__ void bounded_wait_check_kernel(uint32_t *err, unsigned long long limit_ns) {
    __shared__ __align__(8) unsigned long long bar;
    const uint32_t b = hs::smem_addr(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_mbar_init();
        if (!mbar_wait(b, 0, limit_ns)) atomicOr(err, HS_DEVERR_TIMEOUT);
    }
}
}  // namespace

extern "C" hs_status hs_pool_check_bounded_wait(hs_pool_t pool, uint32_t limit_us, void *stream) {
    if (!pool || limit_us == 0 || limit_us > 2000000) return HS_ERR_INVALID_ARG;
    bounded_wait_check_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
        pool->d_err, 1000ull * limit_us);
    return cudaGetLastError() == cudaSuccess ? HS_OK : HS_ERR_CUDA;
}
