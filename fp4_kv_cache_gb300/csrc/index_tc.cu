// index_tc.cu -- tensor-core CSA2 indexer (csa2_index_score fast path, sm_103a tcgen05).
//
// DeepSeek-V4.1-Flash report (aipaper.jasonlin.tech) §2.3 / §2.4.4: the indexer scores
// main-KV entries with FP4 (MXFP4) indexer queries and keys, which is what FP4 tensor
// cores accelerate.  Per query row, the positions are a dense contraction
//     D[t, h] = sum_d k_hat[t, d] * q_hat[h, d]      (t: 128-position tile, h: heads)
// run as block-scaled MMA (kind::mxf4, E2M1 x E2M1, UE8M0 scale per 32) with M = 128
// positions, N = 32 heads per query, K = 128 (two K = 64 steps).  The epilogue reads each
// position's 32 head dots from tensor memory and sums w_h * ReLU(D_h) over the heads.
//
// Precision.  The float32 score written out sums w_h * max(D_h, 0) in one fma chain in head
// order (decode) or in eight chains over the heads h = j mod 8 added in a fixed tree
// (prefill chunks), with D_h = RN32(exact dot); the selection kernels rank by the exact
// score and use this one through its error bound, which needs each D_h correctly rounded.
// Non-finite scores set CSA2_DEV_SCORE_RANGE.  The per-head dot D_h = RN32(exact dot).  Each K = 32 block adds an
// integer (< 2^13) times 2^(Xq + Xk - 2); when every term's exponent lies within 9 of the
// others and in the normal range, every partial sum is exactly representable, so the MMA's
// float32 accumulation returns the exact dot whatever its order.  That condition is checked
// conservatively per position and query from the scale bytes; a position outside it is
// re-scored on CUDA cores (per head, an integer dot of the E2M1 codes per block and one
// dyadic sum rounded once): in decode by the epilogue warp in place, in prefill chunks
// after the main loop for the stages the producer flagged.
//
// Roles: warp 0 = producer (TMA for the FP4 codes with the 64-byte swizzle; the scale
// bytes by one bulk copy per stage, or by cp.async straight into the 512-byte
// scale-factor atoms where a stage is not one contiguous run), warp 1 = MMA issuer (lays
// bulk-copied scales out as atoms, tcgen05.cp of scale factors to TMEM, tcgen05.mma,
// tcgen05.commit), then the epilogue warps (each reads its own TMEM lane quadrant).  A
// shared-memory ring of stages, accumulators rotating in TMEM.  A CTA scores QG queries of
// one sequence (N = QG x 32): QG = 1 in decode, where the CTAs of one query row share its
// stages; QG = 4 in prefill chunks, where one K tile feeds four queries' dots.
#include <cudaTypedefs.h>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "exact.cuh"
#include "tc_util.cuh"

namespace csa2 {
namespace {

constexpr int kD = 128;                // indexer head dim of this path
constexpr int kRowBytes = kD / 2;      // 64 bytes of codes per position
constexpr int kTile = 128;             // positions per tile (MMA M)
constexpr int kNPad = 32;              // heads per query, padded to 32

// A CTA scores QG queries of one sequence against the same key tiles: MMA N = QG x 32
// (queries x heads).  A stage holds kMB tiles of 128 positions (one MMA M block each).
//   QG = 1 (decode): two CTAs per SM, stages of two tiles, so the producer's and the MMA
//     issuer's per-stage costs cover 256 positions and each SM has four tiles in its
//     epilogues at once (two warps per TMEM lane quadrant, one per M block).
//   QG = 4 (prefill chunks): every query of a group sees nearly the same positions, so
//     one K tile feeds four queries' dots; one CTA per SM (its accumulators fill tensor
//     memory), two epilogue warps per lane quadrant, two queries each.
// Tensor-memory columns: accumulator (a, mb) at (a * kMB + mb) * N, then the scale-factor
// columns of A (4 per accumulator block) and of B (4).
template <int QG> struct Cfg;
// kDeferred: positions the MMA may round are found per stage by the producer and re-scored
// after the main loop (prefill: it keeps the re-scoring code out of the epilogue's loop);
// otherwise the epilogue checks each position's bounds and re-scores in place (decode).
template <> struct Cfg<1> {
    static constexpr bool kDeferred = false;
    static constexpr int kStages = 5, kAcc = 3, kMB = 2, kEpiPerQuad = 2, kCtasPerSm = 2;
    static constexpr uint32_t kTmemCols = 256, kColSfa = 192, kColSfb = 216;
};
template <> struct Cfg<4> {
    static constexpr bool kDeferred = true;
    static constexpr int kStages = 12, kAcc = 2, kMB = 1, kEpiPerQuad = 2, kCtasPerSm = 1;
    static constexpr uint32_t kTmemCols = 512, kColSfa = 256, kColSfb = 264;
};
template <int QG> constexpr int kThreadsOf = 64 + 128 * Cfg<QG>::kEpiPerQuad;
template <int QG> constexpr int kSpanOf = Cfg<QG>::kMB * 128;   // positions per stage
constexpr int kFlagWords = 512;        // stage flags: at most 16,384 stages per query group

struct TcParams {
    int32_t n_q, H, ratio_m, block, n_pool_blocks;
    int64_t n_keys, n_cand;
    const uint16_t *q;
    const float *w;
    const uint8_t *kc, *ks;
    const int32_t *q_pos, *pool;
    int pool_mode;
    float *scores;
    int32_t *row_len;
    uint32_t *gmax;          // optional [rows, G]: largest selection key of each 32-group
    int64_t G;
    uint32_t *tile_ctr;      // [units]: claims from each unit's shared tiles (zero at launch)
    uint32_t *tile_done;     // [units]: CTAs of the unit done (zero at launch)
    uint32_t *d_status;
    // fused selection (one query per CTA, FULL mode): the CTA keeps its scores' selection
    // keys on chip and writes a candidate list instead of scores (see fused_list)
    uint32_t *lst_key;       // [rows, CTAs per row, lst_cap] keys (null: write scores)
    int32_t *lst_pos;        // [rows, CTAs per row, lst_cap] positions
    uint32_t *lst_meta;      // [rows, CTAs per row, 4]: count, K-th key (0: K or fewer), non-finite
    int32_t lst_k;           // K
    int32_t lst_stages;      // stages per CTA (lst_cap = lst_stages x span)
    int64_t fresh_from;      // > 0: only positions >= fresh_from may come from the kernel before
};

constexpr int kFuseStages = 32;        // fused selection: stages a CTA keeps on chip
constexpr int kFuseRing = 4;           // fused selection: stage ring (its keys take the room)
// FU: the fused selection's layout (QG = 1 only): a shorter stage ring and the key buffer
template <int QG, bool FU = false>
struct TcSmem {
    static constexpr int kStages = FU ? kFuseRing : Cfg<QG>::kStages, kAcc = Cfg<QG>::kAcc, kSpan = kSpanOf<QG>;
    static constexpr int kFuseKeys = FU ? kFuseStages * kSpanOf<1> : 1;
    uint8_t a[kStages][kSpan * kRowBytes];     // K codes, 64-byte swizzle, 1024-aligned
    uint8_t b[QG * kNPad * kRowBytes];         // q codes (row = query x 32 + head), same layout
    uint32_t sfa[kStages][kSpan];              // scale-factor atoms of the K tiles (one per block)
    uint32_t sfb[kTile];                       // scale-factor atom of q (rows 0..QG*32-1)
    uint64_t full[kStages], empty[kStages], accf[kAcc], acce[kAcc], qready;
    int32_t tile[kStages];                     // stage number held by each stage (-1: no more)
    int32_t sf_raw[kStages];                   // 1: sfa holds the scales in position order
    uint32_t flag_bits[kFlagWords];            // stages with positions to re-check exactly
    int thr_span, thr_lo, thr_hi;              // key-exponent bounds safe for every query
    int32_t acc_tile[kAcc];                    // tile held by each accumulator
    alignas(16) float w[QG][kNPad];            // head weights, 0 for padded heads
    int hmin[QG][kNPad], hmax[QG][kNPad];
    unsigned long long len;                    // candidates of the group (its longest row)
    int64_t qlen[QG];                          // candidates of each query (0: no query)
    uint32_t tmem_base;
    int abort_flag, bad;
    int q_span[QG], q_min[QG], q_max[QG];
    uint32_t fkeys[kFuseKeys];                 // fused selection: the CTA's keys in position order
};
// Two decode CTAs per SM in either layout (the SM's 228 KB, less 1 KB reserved per CTA and
// the 1 KB alignment slack of each)
static_assert(2 * (sizeof(TcSmem<1>) + 1024 + 1024) <= 228 * 1024, "two decode CTAs per SM");
static_assert(2 * (sizeof(TcSmem<1, true>) + 1024 + 1024) <= 228 * 1024, "two fused decode CTAs per SM");

// instruction descriptor, kind::mxf4: A = B = E2M1 (1), UE8M0 scales, K-major A and B,
// N at bits 17-22 (N/8), M at bits 24-28 (M/16), scale-factor ids at bits 4-5 (B) and
// 29-30 (A) select the byte pair of the 32-bit scale column used by this K = 64 step.
template <int QG>
__device__ __forceinline__ uint32_t mxf4_idesc(int sf_id)
{
    return (1u << 7) | (1u << 10) | ((uint32_t)((QG * kNPad) >> 3) << 17) | (1u << 23) |
           ((uint32_t)(kTile >> 4) << 24) | ((uint32_t)sf_id << 4) | ((uint32_t)sf_id << 29);
}

__device__ __forceinline__ int64_t n_visible(const TcParams &P, int64_t row)
{
    if (!P.q_pos) return P.n_keys;
    const int64_t p = P.q_pos[row];
    int64_t v = (p + 1) / P.ratio_m;
    if (p + 1 < 0) v = 0;
    return v < 0 ? 0 : (v > P.n_keys ? P.n_keys : v);
}

// Four E2M1 codes (the low 16 bits, element 0 in the lowest nibble) as four int8 lanes of
// twice their values.
__device__ __forceinline__ int32_t twice4(uint32_t x)
{
    uint32_t r = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) r |= ((uint32_t)e2m1_twice((x >> (4 * i)) & 15u) & 0xffu) << (8 * i);
    return (int32_t)r;
}

// Exact D_h of one position for head h = this lane (the rare positions the tensor-core
// result cannot be proven exact for): per 32-value block the integer dot of twice the
// E2M1 values (dp4a) and its dyadic sum rounded once to float32.  The key row is read by
// all lanes at once; the query's codes and scales come from the B-operand copy in shared
// memory (64-byte rows, 16-byte chunks XOR-swizzled by bits 1-2 of the row within its
// group of 8).
__device__ __forceinline__ float exact_head_dot(const uint8_t *kc, uint32_t sfw, const uint8_t *qb,
                                                const uint8_t *qsf, int qi, int h)
{
    const int n = qi * kNPad + h, r8 = n & 7;               // B-operand row of (query, head)
    const uint8_t *qrow = qb + (n >> 3) * 512 + r8 * 64;
    int I[4], E[4];
#pragma unroll
    for (int kb = 0; kb < 4; ++kb) {
        const uint4 k = *reinterpret_cast<const uint4 *>(kc + 16 * kb);
        const uint4 q = *reinterpret_cast<const uint4 *>(qrow + ((kb ^ ((r8 >> 1) & 3)) << 4));
        const uint32_t k4[4] = {k.x, k.y, k.z, k.w}, q4[4] = {q.x, q.y, q.z, q.w};
        int acc = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            acc = __dp4a(twice4(q4[j] & 0xffffu), twice4(k4[j] & 0xffffu), acc);
            acc = __dp4a(twice4(q4[j] >> 16), twice4(k4[j] >> 16), acc);
        }
        I[kb] = acc;
        E[kb] = ((int)qsf[h * 16 + qi * 4 + kb] - 127) + ((int)((sfw >> (8 * kb)) & 255u) - 127) - 2;
    }
    return dyadic_sum_f32<4>(I, E);
}

// The warp re-scores its lanes flagged in `todo` exactly, one head per lane, summing the
// heads' terms in the order the calling kernel uses (split: the eight partial sums of the
// prefill-chunk epilogue, else one chain in head order); returns this lane's new score
// (or `score` when the lane was not flagged).  Out of line: the hot loop keeps only the
// call.
template <bool SPLIT>
__device__ __noinline__ float rescore_flagged(uint32_t todo, float score, uint32_t sfw, int64_t cand0,
                                              const uint8_t *kc_row0, const int32_t *pool, int pool_mode,
                                              int64_t n_keys, const uint8_t *qb, const uint8_t *qsf,
                                              const float *w, int qi, int H)
{
    const int lane = threadIdx.x & 31;
    while (todo) {
        const int src = __ffs(todo) - 1;
        todo &= todo - 1u;
        const int64_t pc = cand0 + src;
        int64_t pos = pc;
        if (pool_mode) {
            const int32_t id = pool[pc >> 3];
            pos = (int64_t)(id < 0 ? 0 : id) * 8 + (pc & 7);
            if (pos >= n_keys) pos = n_keys - 1;
        }
        const uint32_t psfw = __shfl_sync(0xffffffffu, sfw, src);
        const float Dh = lane < H ? exact_head_dot(kc_row0 + pos * kRowBytes, psfw, qb, qsf, qi, lane) : 0.0f;
        float e = 0.0f;
        if constexpr (SPLIT) {
            float p[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int h = 0; h < kNPad; ++h) {
                const float d = __shfl_sync(0xffffffffu, Dh, h);
                p[h & 7] = __fmaf_rn(h < H ? w[h] : 0.0f, d > 0.0f ? d : 0.0f, p[h & 7]);
            }
            e = __fadd_rn(__fadd_rn(__fadd_rn(p[0], p[1]), __fadd_rn(p[2], p[3])),
                          __fadd_rn(__fadd_rn(p[4], p[5]), __fadd_rn(p[6], p[7])));
        } else {
            for (int h = 0; h < H; ++h) {
                const float d = __shfl_sync(0xffffffffu, Dh, h);
                e = __fmaf_rn(w[h], d > 0.0f ? d : 0.0f, e);
            }
        }
        if (lane == src) score = e;
    }
    return score;
}

// Exact re-check of one flagged stage by one warp: per 32 positions and query, the
// positions whose key exponents break that query's exactness bounds are re-scored on CUDA
// cores (rescore_flagged) and their score and group maximum rewritten.  Runs after the main
// loop, so the loop itself carries no re-scoring code.
template <int QG, bool FU>
__device__ __noinline__ void recheck_stage(const TcParams &P, const TcSmem<QG, FU> &S, int t, int span, int64_t row0,
                                           int t0q, int64_t kbase, const int32_t *pool, int64_t n_blk_all)
{
    const int lane = threadIdx.x & 31;
#pragma unroll 1
    for (int c = 0; c < span / 32; ++c) {
        const int64_t g0 = (int64_t)t * span + c * 32, p = g0 + lane;
        int64_t pos = p;
        if (P.pool_mode) {
            const int64_t plen = (int64_t)P.n_pool_blocks * P.block;
            int64_t id = p < plen ? pool[p >> 3] : 0;
            id = id < 0 ? 0 : (id >= n_blk_all ? n_blk_all - 1 : id);
            pos = id * 8 + (p & 7);
        }
        if (pos >= P.n_keys) pos = P.n_keys - 1;
        const uint32_t kw = *reinterpret_cast<const uint32_t *>(P.ks + (kbase + pos) * 4);
        const int e0 = (int)(kw & 255u), e1 = (int)((kw >> 8) & 255u);
        const int e2 = (int)((kw >> 16) & 255u), e3 = (int)(kw >> 24);
        const int kmin = min(min(e0, e1), min(e2, e3)) - 127, kmax = max(max(e0, e1), max(e2, e3)) - 127;
#pragma unroll 1
        for (int qi = 0; qi < QG; ++qi) {
            if (t0q + qi >= P.n_q) break;
            const int64_t qlen = S.qlen[qi];
            const bool valid = p < qlen;
            const bool unsafe = valid && ((kmax - kmin) + S.q_span[qi] > 9 || S.q_min[qi] + kmin - 2 < -126 ||
                                          S.q_max[qi] + kmax - 2 > 100);
            const uint32_t todo = __ballot_sync(0xffffffffu, unsafe);
            if (!todo) continue;
            float *srow = P.scores + (row0 + qi) * P.n_cand;
            float sc = valid ? srow[p] : 0.0f;
            sc = rescore_flagged<Cfg<QG>::kDeferred>(todo, sc, kw, g0, P.kc + kbase * kRowBytes, pool, P.pool_mode, P.n_keys, S.b,
                                 reinterpret_cast<const uint8_t *>(S.sfb), S.w[qi], qi, P.H);
            if ((todo >> lane) & 1u) srow[p] = sc;
            if (__any_sync(0xffffffffu, ((todo >> lane) & 1u) && !(fabsf(sc) <= 3.4028234663852886e38f)) &&
                lane == 0)
                dev_flag(P.d_status, CSA2_DEV_SCORE_RANGE);
            if (P.gmax) {
                const uint32_t gk = __reduce_max_sync(0xffffffffu, valid ? score_key(sc) : 0u);
                if (lane == 0 && g0 < qlen) P.gmax[(row0 + qi) * P.G + (g0 >> 5)] = gk;
            }
        }
    }
}

// Registers: with QG = 1, two resident CTAs of 320 threads need every warp within its
// sub-partition's share of the register file (20 warps over 4 sub-partitions: at most 102
// registers a thread, 96 after rounding); the launch bound makes the compiler keep to it.
// Block-wide exclusive prefix sum of one value per thread (any multiple of 32 threads).
__device__ __forceinline__ uint32_t fused_scan(uint32_t v, uint32_t *s_warp, uint32_t &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const uint32_t w = lane < nw ? s_warp[lane] : 0u;
        uint32_t wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += t;
        }
        s_warp[lane] = wi - w;
        if (lane == 31) s_warp[32] = wi;
    }
    __syncthreads();
    const uint32_t r = s_warp[warp] + incl - v;
    total = s_warp[32];
    __syncthreads();
    return r;
}

// Fused selection at the end of a CTA: its V selection keys (positions pos0 .. pos0 + V - 1 of
// `row`, in S.fkeys) become its candidate list, in position order.  With K or fewer keys the
// list is all of them; otherwise tau is a lower bound of the K-th largest key (its top 22
// bits) and the list holds every key whose score is at least lo(tau), lo as in the exact
// Top-K's band (report §2.3 Top-K by the exact score): the row's K-th score is at least
// tau, so every candidate of the row's exact top K and of its band is here.  A row with a
// negative head weight (its bound needs the whole sequence's key scales) keeps every key; a
// CTA that met a non-finite score keeps the keys >= tau and says so (its row then goes by
// the float order, for which those suffice).
template <int QG, bool FU>
__device__ __noinline__ void fused_list(const TcParams &P, TcSmem<QG, FU> &S, int64_t row, int64_t pos0, int V)
{
    const int tid = threadIdx.x, lane = tid & 31;
    constexpr int NT = kThreadsOf<QG>;
    __shared__ uint32_t s_pick[2], s_warp[33];
    const uint32_t *keys = S.fkeys;
    const int64_t slot = row * gridDim.x + blockIdx.x;
    uint32_t *meta = P.lst_meta + slot * 4;
    const int64_t lbase = slot * (int64_t)P.lst_stages * kSpanOf<QG>;
    const uint32_t K = (uint32_t)P.lst_k;
    bool nf = false;
    for (int i = tid; i < V; i += NT) {
        const uint32_t k = keys[i];
        nf |= k >= 0xff800000u || k <= 0x007fffffu;
    }
    nf = __syncthreads_or(nf) != 0;
    uint32_t tau = 0u, lo_key = 0u;
    if ((uint32_t)V > K) {
        // tau: the top 22 bits of the K-th largest key, its low bits zero -- a lower bound,
        // enough to cut the list (lo rises with its argument): two digit passes of 11 bits,
        // one atomic per distinct digit and warp, in the stage buffers (free now)
        uint32_t *hist = reinterpret_cast<uint32_t *>(&S.a[0][0]);
        uint32_t *coarse = hist + 2048;
        uint32_t prefix = 0u, mask = 0u, remaining = K;
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
            const int shift = pass == 0 ? 21 : 10;
            for (int i = tid; i < 2048 + 64; i += NT) hist[i] = 0u;
            __syncthreads();
            for (int base = 0; base < V; base += NT) {
                const int i = base + tid;
                uint32_t key = 0u;
                bool act = false;
                if (i < V) {
                    key = keys[i];
                    act = (key & mask) == prefix;
                }
                const uint32_t am = __ballot_sync(0xffffffffu, act);
                if (act) {
                    const uint32_t digit = (key >> shift) & 2047u;
                    const uint32_t peers = __match_any_sync(am, digit);
                    if (lane == __ffs(peers) - 1) {
                        atomicAdd(&hist[digit], (uint32_t)__popc(peers));
                        atomicAdd(&coarse[digit >> 5], (uint32_t)__popc(peers));
                    }
                }
            }
            __syncthreads();
            if (tid < 32) {                      // the digit, from the top: coarse bins, then 32 bins
                const uint32_t c0 = coarse[63 - lane], c1 = coarse[31 - lane];
                uint32_t i0 = c0, i1 = c1;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t x = __shfl_up_sync(0xffffffffu, i0, o), y = __shfl_up_sync(0xffffffffu, i1, o);
                    if (lane >= o) { i0 += x; i1 += y; }
                }
                i1 += __shfl_sync(0xffffffffu, i0, 31);
                const uint32_t b0 = __ballot_sync(0xffffffffu, i0 >= remaining);
                const uint32_t b1 = __ballot_sync(0xffffffffu, i1 >= remaining);
                int cb;
                uint32_t above;
                if (b0) {
                    const int L = __ffs(b0) - 1;
                    cb = 63 - L;
                    above = __shfl_sync(0xffffffffu, i0 - c0, L);
                } else {
                    const int L = b1 ? __ffs(b1) - 1 : 31;
                    cb = 31 - L;
                    above = __shfl_sync(0xffffffffu, i1 - c1, L);
                }
                const uint32_t f = hist[cb * 32 + 31 - lane];
                uint32_t fi = f;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t x = __shfl_up_sync(0xffffffffu, fi, o);
                    if (lane >= o) fi += x;
                }
                fi += above;
                const uint32_t bf = __ballot_sync(0xffffffffu, fi >= remaining);
                const int Lf = bf ? __ffs(bf) - 1 : 31;
                const uint32_t fabove = __shfl_sync(0xffffffffu, fi - f, Lf);
                if (lane == 0) {
                    s_pick[0] = (uint32_t)(cb * 32 + 31 - Lf);
                    s_pick[1] = remaining - fabove;
                }
            }
            __syncthreads();
            prefix |= s_pick[0] << shift;
            mask |= 2047u << shift;
            remaining = s_pick[1];
            __syncthreads();                     // s_pick is read before the next pass writes it
        }
        tau = prefix;
        bool neg;
        const RowBound rb = row_bound_nonneg(S.w[0], P.H, neg);
        lo_key = neg ? 0u : (nf ? tau : score_key(rb.lo(key_value(tau))));
    }
    // the list: keys >= lo_key, each thread a contiguous run of positions
    const int run = (V + NT - 1) / NT;
    const int i0 = min(tid * run, V), i1 = min(i0 + run, V);
    uint32_t cnt = 0;
    for (int i = i0; i < i1; ++i) cnt += keys[i] >= lo_key;
    uint32_t total;
    uint32_t o = fused_scan(cnt, s_warp, total);
    for (int i = i0; i < i1; ++i) {
        const uint32_t key = keys[i];
        if (key >= lo_key) {
            P.lst_key[lbase + o] = key;
            P.lst_pos[lbase + o] = (int32_t)(pos0 + i);
            ++o;
        }
    }
    if (tid == 0) {
        meta[0] = total;
        meta[1] = tau;
        meta[2] = nf ? 1u : 0u;
        meta[3] = 0u;
    }
}

template <int QG, bool FU>
__global__ void __launch_bounds__(kThreadsOf<QG>, Cfg<QG>::kCtasPerSm)
index_score_tc_kernel(const __grid_constant__ CUtensorMap tmap, const TcParams P)
{
    using C = Cfg<QG>;
    constexpr int kStages = TcSmem<QG, FU>::kStages, kAcc = C::kAcc, kN = QG * kNPad, kMB = C::kMB;
    constexpr int kSpan = kSpanOf<QG>;
    constexpr int kEpiWarps = 4 * C::kEpiPerQuad, kQPerWarp = QG * kMB / C::kEpiPerQuad;
    extern __shared__ uint8_t smem_raw[];
    TcSmem<QG, FU> &S = *reinterpret_cast<TcSmem<QG, FU> *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                    ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // unit = the QG consecutive queries of one sequence this CTA scores (rows row0 ..)
    const int64_t unit = blockIdx.y;
    const int64_t groups = (P.n_q + QG - 1) / QG;
    const int64_t b = unit / groups;
    const int t0q = (int)(unit % groups) * QG;                 // first query of the group
    const int64_t row0 = b * P.n_q + t0q;
    const int H = P.H;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            tc::mbar_init(&S.full[s], 1 + 32);
            tc::mbar_init(&S.empty[s], 1);       // the MMA's commit
        }
        for (int i = 0; i < kAcc; ++i) {
            tc::mbar_init(&S.accf[i], 2);        // the MMA's commit + the issuer's own arrive
            tc::mbar_init(&S.acce[i], kEpiWarps);
        }
        tc::mbar_init(&S.qready, 1);
        S.abort_flag = 0;
        S.bad = 0;
        S.len = 0;
        tc::fence_mbar_init();
    }
    if (tid < QG * kNPad) { S.hmin[tid >> 5][tid & 31] = 1 << 20; S.hmax[tid >> 5][tid & 31] = -(1 << 20); }
    if (tid < kTile) S.sfb[tid] = 0x7f7f7f7fu;
    for (int i = tid; i < kFlagWords; i += kThreadsOf<QG>) S.flag_bits[i] = 0u;
    if (warp == 0 && lane == 0) tc::prefetch_tmap(&tmap);
    if (warp == 1) {
        tc::tmem_alloc(&S.tmem_base, C::kTmemCols);
        tc::tmem_relinquish();
    }
    // everything above touched no input: it overlaps the previous kernel's tail.  With
    // fresh_from, the positions below it (and q, w, q_pos) are not written by the kernel
    // before: the dependency wait is taken only before the first stage that holds a newer
    // position, before the first claim from the shared counters, and before the CTA ends.
    const bool early = !P.pool_mode && P.fresh_from > 0;
    if (!early) pdl_wait();
    pdl_allow_dependents();
    // ---- valid candidates of the group's rows (and pool checks): needed before streaming
    const int32_t *pool = P.pool_mode ? P.pool + row0 * (int64_t)P.n_pool_blocks : nullptr;
    const int64_t n_blk_all = (P.n_keys + P.block - 1) / P.block;
    __syncthreads();                                       // barrier init / len zero visible
    if (!P.pool_mode) {
        if (tid < QG) {
            const bool live = t0q + tid < P.n_q;
            const int64_t nv = live ? n_visible(P, row0 + tid) : 0;
            S.qlen[tid] = nv;
            atomicMax(&S.len, (unsigned long long)nv);
        }
    } else {                                               // QG == 1 here
        const int64_t n_vis = n_visible(P, row0);
        unsigned long long part = 0;
        int bad = 0;
        for (int i = tid; i < P.n_pool_blocks; i += kThreadsOf<QG>) {
            const int32_t id = pool[i];
            const int32_t prev = i > 0 ? pool[i - 1] : -1;
            if (id >= 0) {
                if (id >= n_blk_all || (i > 0 && (prev < 0 || prev >= id))) bad = 1;
                const int64_t c = n_vis - (int64_t)id * P.block;
                part += c <= 0 ? 0 : (c > P.block ? P.block : c);
            }
        }
        if (bad) atomicOr(&S.bad, 1);
        if (part) atomicAdd(&S.len, part);
    }
    __syncthreads();
    const int64_t len = (int64_t)S.len;
    if (P.pool_mode && tid == 0) S.qlen[0] = len;
    __syncthreads();
    if (blockIdx.x == 0 && tid < QG && t0q + tid < P.n_q) {
        if (P.row_len) P.row_len[row0 + tid] = (int32_t)S.qlen[tid];
        if (tid == 0 && S.bad) dev_flag(P.d_status, CSA2_DEV_BAD_POOL);
    }
    // Stages of the group (kSpan positions each): CTA c first takes the R consecutive
    // stages [cR, cR + R) (C CTAs per group, R two short of an even share; consecutive
    // stages keep the reads sequential); the rest are handed out one at a time from the
    // group's counter, so its CTAs finish together.  Each claim is made one stage ahead of
    // its use, which hides the atomic's latency.  A stage carries its number from the
    // producer to the MMA issuer (-1: no more), an accumulator carries it on to the
    // epilogue.
    const int ntr = len > 0 ? (int)((len + kSpan - 1) / kSpan) : 0;
    const int CT = (int)gridDim.x;
    // fused selection: CTA c takes the fixed run [c F, c F + F) of lst_stages stages
    constexpr bool fused = QG == 1 && FU;
    const int R = fused ? P.lst_stages : (ntr / CT > 2 ? ntr / CT - 2 : 0);
    const int64_t c1 = len;
    const uint32_t tmem = S.tmem_base;
    const int64_t kbase = b * P.n_keys;

    if (warp == 0) {
        // ================= producer
        // first the quantising warps' query reads enter the memory system (named barrier
        // 2), so they are not queued behind every CTA's first tile loads
        asm volatile("bar.sync 2, 160;" ::: "memory");
        // Exactness (see the file header): a position's MMA dot is exact for query q when its
        // key block exponents kmin..kmax satisfy kmax - kmin <= 9 - span_q, kmin >= -124 -
        // min_q and kmax <= 102 - max_q.  When the MMA has released a stage, the producer
        // reads its scale words back and flags the stage if any position breaks the bounds
        // of some query of this CTA; flagged stages are re-checked per query and re-scored
        // after the main loop, so neither the MMA issuer nor the epilogue carries that work.
        int thr_span = 0, thr_lo = 0, thr_hi = 0;
        bool have_thr = false;
        auto check_stage = [&](int st, int tp) {
            if (!have_thr) {
                if (!__all_sync(0xffffffffu, tc::mbar_wait(&S.qready, 0, &S.abort_flag))) return;
                thr_span = 1 << 20; thr_lo = -(1 << 20); thr_hi = 1 << 20;
#pragma unroll 1
                for (int qi = 0; qi < QG; ++qi) {
                    thr_span = min(thr_span, 9 - S.q_span[qi]);
                    thr_lo = max(thr_lo, -124 - S.q_min[qi]);
                    thr_hi = min(thr_hi, 102 - S.q_max[qi]);
                }
                have_thr = true;
            }
            bool uns = false;
#pragma unroll
            for (int j = 0; j < 4 * kMB; ++j) {
                const uint32_t x = S.sfa[st][j * 32 + lane];       // every word once, any order
                const int e0 = (int)(x & 255u), e1 = (int)((x >> 8) & 255u);
                const int e2 = (int)((x >> 16) & 255u), e3 = (int)(x >> 24);
                const int kmn = min(min(e0, e1), min(e2, e3)) - 127, kmx = max(max(e0, e1), max(e2, e3)) - 127;
                uns |= kmx - kmn > thr_span || kmn < thr_lo || kmx > thr_hi;
            }
            if (__any_sync(0xffffffffu, uns) && lane == 0) S.flag_bits[tp >> 5] |= 1u << (tp & 31);
        };
        int issued = 0;
        uint32_t claim = 0;                       // lane 0: the next claim from the counter
        bool waited = !early;
        auto wait_prev = [&]() {
            if (!waited) {
                pdl_wait();
                waited = true;
            }
        };
        if (R == 0 && !fused) wait_prev();
        if (lane == 0 && R == 0 && !fused) claim = atomicAdd(&P.tile_ctr[unit], 1u);
        for (int i = 0;; ++i) {
            const int s = i % kStages;
            const uint32_t ph = (uint32_t)(i / kStages) & 1u;
            if (!__all_sync(0xffffffffu, tc::mbar_wait(&S.empty[s], ph ^ 1u, &S.abort_flag))) {
                S.abort_flag = 1;
                break;
            }
            if (C::kDeferred && i >= kStages && !S.abort_flag) check_stage(s, S.tile[s]);   // its previous tile
            int t = 0;
            if (fused) {
                t = i < R ? (int)blockIdx.x * R + i : ntr;
            } else if (i < R) {
                t = (int)blockIdx.x * R + i;
                if (i == R - 1) wait_prev();
                if (lane == 0 && i == R - 1) claim = atomicAdd(&P.tile_ctr[unit], 1u);
            } else {
                if (lane == 0) {
                    t = R * CT + (int)claim;
                    if (t < ntr) claim = atomicAdd(&P.tile_ctr[unit], 1u);
                }
                t = __shfl_sync(0xffffffffu, t, 0);
            }
            if (t >= ntr) {                       // end marker: 1 + 32 plain arrivals, no bytes
                if (lane == 0) {
                    S.tile[s] = -1;
                    tc::mbar_arrive(&S.full[s]);
                }
                __syncwarp();
                tc::mbar_arrive(&S.full[s]);
                break;
            }
            const int64_t t0 = (int64_t)t * kSpan;
            if (t0 + kSpan > P.fresh_from) wait_prev();   // the stage holds a newer position
            // a whole stage of consecutive positions: its scale bytes are one contiguous run,
            // copied in position order by one bulk copy (the MMA warp rearranges them into
            // the scale-factor atoms); otherwise each lane copies its atom words
            const uint8_t *ks_run = P.ks + (kbase + t0) * 4;
            const bool sf_bulk = !P.pool_mode && t0 + kSpan <= c1 && ((uintptr_t)ks_run & 15u) == 0;
            if (lane == 0) {
                S.tile[s] = t;
                S.sf_raw[s] = sf_bulk ? 1 : 0;
                if (!P.pool_mode) {
                    tc::mbar_arrive_expect_tx(&S.full[s], kSpan * kRowBytes + (sf_bulk ? kSpan * 4 : 0));
                    tc::tma_load_2d(S.a[s], &tmap, &S.full[s], 0, (int32_t)(kbase + t0));
                    if (sf_bulk) tc::bulk_load(S.sfa[s], ks_run, kSpan * 4, &S.full[s]);
                }
            }
            // pool mode: lane j reads the stage's block id j (all at once) and loads that
            // block's 8 code rows with one TMA box
            int64_t blk_id = -1;
            if (P.pool_mode) {
                static_assert(QG != 1 || kSpanOf<1> / 8 == 32, "one pool block per lane");
                if (lane < kSpan / 8 && t0 + 8 * lane < c1) blk_id = pool[(t0 >> 3) + lane];
                const uint32_t have = __ballot_sync(0xffffffffu, blk_id >= 0);
                if (lane == 0) tc::mbar_arrive_expect_tx(&S.full[s], (uint32_t)__popc(have) * 8u * kRowBytes);
                __syncwarp();
                if (blk_id >= 0) {
                    const int64_t id = blk_id >= n_blk_all ? n_blk_all - 1 : blk_id;
                    tc::tma_load_2d(S.a[s] + lane * 8 * kRowBytes, &tmap, &S.full[s], 0, (int32_t)(kbase + id * 8));
                }
            }
            // scale atom of block mb: word lane * 4 + j holds position mb * 128 + lane + 32 j
#pragma unroll
            for (int j = 0; j < 4 * kMB; ++j) {
                if (sf_bulk) break;
                const int m = lane + 32 * j;
                const int64_t cand = t0 + m;
                uint32_t *dst = &S.sfa[s][(j >> 2) * kTile + lane * 4 + (j & 3)];
                const int64_t bid = P.pool_mode ? __shfl_sync(0xffffffffu, blk_id, (m >> 3) & 31) : 0;
                if (cand < c1) {
                    int64_t pos = cand;
                    if (P.pool_mode) {
                        int64_t id = bid;           // lane m / 8 read it above
                        id = id < 0 ? 0 : (id >= n_blk_all ? n_blk_all - 1 : id);
                        pos = id * 8 + (cand & 7);
                        if (pos >= P.n_keys) pos = P.n_keys - 1;
                    }
                    tc::cp_async_4(dst, P.ks + (kbase + pos) * 4);
                } else {
                    *dst = 0x7f7f7f7fu;
                }
            }
            // no proxy fence here: it would wait for this lane's copies in flight; the MMA
            // thread fences after it has seen the stage complete
            tc::cp_async_mbar_arrive_noinc(&S.full[s]);
            ++issued;
        }
        if (S.abort_flag) {       // let copies already in flight land before the CTA exits
            for (int i = issued - 1; i >= 0 && i >= issued - kStages; --i)
                tc::mbar_wait_bounded(&S.full[i % kStages], (uint32_t)(i / kStages) & 1u);
        } else if (C::kDeferred) {
            // the tiles still in stages: checked once the MMA has released them
#pragma unroll 1
            for (int j = issued - kStages + 1 > 0 ? issued - kStages + 1 : 0; j < issued; ++j) {
                const int st = j % kStages;
                if (!__all_sync(0xffffffffu, tc::mbar_wait(&S.empty[st], (uint32_t)(j / kStages) & 1u,
                                                           &S.abort_flag))) {
                    S.abort_flag = 1;
                    break;
                }
                check_stage(st, S.tile[st]);
            }
        }
        // joins the epilogue warps before their re-check of the flagged stages
        if (C::kDeferred) asm volatile("bar.sync 3, %0;" ::"r"((kEpiWarps + 1) * 32) : "memory");
    } else if (warp == 1) {
        // ================= MMA issuer (lane 0; the warp rearranges bulk-copied scales)
        const uint32_t sfb_t = tmem + C::kColSfb;
        bool ok = tc::mbar_wait(&S.qready, 0, &S.abort_flag);
        if (!__all_sync(0xffffffffu, ok)) S.abort_flag = 1;
        if (lane == 0) {
            tc::fence_proxy_async_smem();
            tc::tc_fence_after();
            if (!S.abort_flag)
                tc::tc_cp_32x128b_warpx4(sfb_t, tc::smem_desc(tc::smem_u32(S.sfb), 512, 128, tc::kSwizzleNone));
        }
        __syncwarp();
        for (int i = 0;; ++i) {
            if (__any_sync(0xffffffffu, S.abort_flag != 0)) break;    // the warp leaves together
            const int s = i % kStages, acc = i % kAcc;
            ok = tc::mbar_wait(&S.acce[acc], ((uint32_t)(i / kAcc) & 1u) ^ 1u, &S.abort_flag) &&
                 tc::mbar_wait(&S.full[s], (uint32_t)(i / kStages) & 1u, &S.abort_flag);
            if (!__all_sync(0xffffffffu, ok)) {
                S.abort_flag = 1;
                break;
            }
            const int t = S.tile[s];
            if (t < 0) {                          // pass the end marker to the epilogue
                if (lane == 0) {
                    S.acc_tile[acc] = t;
                    tc::mbar_arrive(&S.accf[acc]);
                    tc::mbar_arrive(&S.accf[acc]);
                }
                break;
            }
            const bool raw = S.sf_raw[s] != 0;
            if (raw) {
                // position-ordered scale words -> atoms (word lane * 4 + j of block mb holds
                // position mb * 128 + lane + 32 j): all reads, then all writes
                uint32_t v[4 * kMB];
#pragma unroll
                for (int j = 0; j < 4 * kMB; ++j) v[j] = S.sfa[s][(j >> 2) * kTile + lane + 32 * (j & 3)];
                __syncwarp();
#pragma unroll
                for (int mb = 0; mb < kMB; ++mb)
                    *reinterpret_cast<uint4 *>(&S.sfa[s][mb * kTile + lane * 4]) =
                        make_uint4(v[4 * mb], v[4 * mb + 1], v[4 * mb + 2], v[4 * mb + 3]);
                tc::fence_proxy_async_smem();
                __syncwarp();
            }
            if (lane == 0) {
                S.acc_tile[acc] = t;
                // atoms the producer's lanes copied (cp.async) are seen by the tensor core's
                // copy after this fence; rearranged atoms were fenced by the writing lanes
                if (!raw) tc::fence_proxy_async_smem();
                tc::tc_fence_after();
#pragma unroll
                for (int mb = 0; mb < kMB; ++mb) {
                    const uint32_t sfa_t = tmem + C::kColSfa + 4 * (acc * kMB + mb);
                    tc::tc_cp_32x128b_warpx4(sfa_t, tc::smem_desc(tc::smem_u32(S.sfa[s] + mb * kTile), 512, 128,
                                                                  tc::kSwizzleNone));
                    const uint32_t d_t = tmem + (acc * kMB + mb) * kN;
                    const uint32_t a0 = tc::smem_u32(S.a[s]) + mb * kTile * kRowBytes;
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk) {
                        const uint64_t ad = tc::smem_desc(a0 + kk * 32, 16, 512, tc::kSwizzle64B);
                        const uint64_t bd = tc::smem_desc(tc::smem_u32(S.b) + kk * 32, 16, 512, tc::kSwizzle64B);
                        tc::tc_mma_mxf4(d_t, ad, bd, mxf4_idesc<QG>(2 * kk), sfa_t, sfb_t, kk);
                    }
                }
                tc::tc_commit(&S.empty[s]);
                tc::tc_commit(&S.accf[acc]);
                tc::mbar_arrive(&S.accf[acc]);    // releases acc_tile to the epilogue
            }
            __syncwarp();
        }
    } else {
        // ================= epilogue warps: first the queries (B operand), then the scores
        const int et = tid - 64;
        if (et < 128) {
            // thread (h, kb) quantises block kb of head h of each query on its own: 4 x
            // 16-byte loads, a local maximum, 32 codes packed into one 16-byte store
            const int h = et >> 2, kb = et & 3;
#pragma unroll 1
            for (int qi = 0; qi < QG; ++qi)
                if (h < H && t0q + qi < P.n_q)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(P.q + (row0 + qi) * (int64_t)H * kD + h * kD + kb * 32));
            asm volatile("bar.arrive 2, 160;" ::: "memory");     // releases the producer
#pragma unroll 1
            for (int qi = 0; qi < QG; ++qi) {
                const bool live = h < H && t0q + qi < P.n_q;
                uint4 raw[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                                make_uint4(0, 0, 0, 0)};
                if (live) {
                    const uint4 *src = reinterpret_cast<const uint4 *>(P.q + (row0 + qi) * (int64_t)H * kD +
                                                                       h * kD + kb * 32);
#pragma unroll
                    for (int j = 0; j < 4; ++j) raw[j] = src[j];
                }
                float v[32];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t w4[4] = {raw[j].x, raw[j].y, raw[j].z, raw[j].w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        v[8 * j + 2 * k] = __uint_as_float(w4[k] << 16);
                        v[8 * j + 2 * k + 1] = __uint_as_float(w4[k] & 0xffff0000u);
                    }
                }
                uint32_t amax_bits = 0;
#pragma unroll
                for (int e = 0; e < 32; ++e) amax_bits = max(amax_bits, __float_as_uint(v[e]) & 0x7fffffffu);
                const bool finite = amax_bits < 0x7f800000u;
                const int X = mx_block_exponent(__uint_as_float(finite ? amax_bits : 0u));
                const float inv = pow2_neg(X);
                uint32_t packed[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t word = 0;
#pragma unroll
                    for (int e = 0; e < 8; e += 2)
                        word |= e2m1x2_cvt(v[8 * j + e] * inv, v[8 * j + e + 1] * inv) << (4 * e);
                    packed[j] = word;
                }
                // B row n = query x 32 + head, 16-byte chunk kb of the 64-byte row,
                // XOR-swizzled by bits 1-2 of n % 8; its scale byte (n%32)*16 + (n/32)*4 + kb
                const int n = qi * kNPad + h, r8 = n & 7;
                *reinterpret_cast<uint4 *>(S.b + (n >> 3) * 512 + r8 * 64 + ((kb ^ ((r8 >> 1) & 3)) << 4)) =
                    make_uint4(packed[0], packed[1], packed[2], packed[3]);
                reinterpret_cast<uint8_t *>(S.sfb)[h * 16 + qi * 4 + kb] = (uint8_t)(X + 127);
                // per-head exponent range over its non-zero blocks (the 4 blocks sit in 4 lanes)
                int mn = (live && amax_bits != 0) ? X : (1 << 20);
                int mx = (live && amax_bits != 0) ? X : -(1 << 20);
                mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, 1));
                mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, 2));
                mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                if (kb == 0) { S.hmin[qi][h] = mn; S.hmax[qi][h] = mx; }
                if (live && !finite) dev_flag(P.d_status, CSA2_DEV_NONFINITE);
                if (et < kNPad)
                    S.w[qi][et] = et < H && t0q + qi < P.n_q ? P.w[(row0 + qi) * H + et] : 0.0f;
            }
            tc::fence_proxy_async_smem();
            asm volatile("bar.sync 1, 128;" ::: "memory");   // the first four epilogue warps
            if (warp - 2 < QG) {                  // warp 2 + qi: query qi; lane h: head h
                const int qi = warp - 2;
                const int hmn = S.hmin[qi][lane], hmx = S.hmax[qi][lane];
                const bool live = lane < H && hmn <= hmx;     // not an all-zero head
                const int span = __reduce_max_sync(0xffffffffu, live ? hmx - hmn : 0);
                const int mn = __reduce_min_sync(0xffffffffu, live ? hmn : (1 << 20));
                const int mx = __reduce_max_sync(0xffffffffu, live ? hmx : -(1 << 20));
                if (lane == 0) {
                    S.q_span[qi] = span;
                    S.q_min[qi] = mn;
                    S.q_max[qi] = mx;
                }
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (et == 0) tc::mbar_arrive(&S.qready);
        }
        // epilogue warp ew: lane quadrant `quad`, M block mb of each stage, queries
        // [q_lo, q_lo + kQPerWarp)
        const int ew = warp - 2, quad = warp & 3, mb = (ew >> 2) % kMB, q_lo = (ew >> 2) / kMB * kQPerWarp;
        const int m = mb * kTile + quad * 32 + lane;           // position within the stage
        const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
        // this warp's queries' candidates and exponent ranges (read once the first
        // accumulator is full, which is after the queries were quantised)
        int64_t qlen[kQPerWarp];
        int qspan[kQPerWarp], qmin[kQPerWarp], qmax[kQPerWarp];
        bool out_of_range = false;            // a score this warp wrote is not finite
        bool ewaited = !early;
        for (int i = 0;; ++i) {
            const int acc = i % kAcc;
            // the stage itself is not touched here: the MMA's completion frees it
            const bool ok = tc::mbar_wait(&S.accf[acc], (uint32_t)(i / kAcc) & 1u, &S.abort_flag);
            if (!__all_sync(0xffffffffu, ok)) {   // the warp leaves together (aligned ops follow)
                S.abort_flag = 1;
                break;
            }
            const int t = S.acc_tile[acc];
            if (t < 0) break;                     // end marker (the same for the whole warp)
            if (!ewaited && (int64_t)(t + 1) * kSpan > P.fresh_from) {   // newer positions: re-scores read them
                pdl_wait();
                ewaited = true;
            }
            if (i == 0) {
#pragma unroll
                for (int u = 0; u < kQPerWarp; ++u) {
                    qlen[u] = S.qlen[q_lo + u];
                    qspan[u] = S.q_span[q_lo + u];
                    qmin[u] = S.q_min[q_lo + u];
                    qmax[u] = S.q_max[q_lo + u];
                }
            }
            tc::tc_fence_after();
            uint32_t sf4[4] = {0u, 0u, 0u, 0u};
            if constexpr (!C::kDeferred) {
                // the scale atom holds in lane L the words of rows L, L+32, L+64, L+96 (copied
                // to every lane quadrant), so row quad*32+lane is word `quad` of this lane
                asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(sf4[0]), "=r"(sf4[1]), "=r"(sf4[2]), "=r"(sf4[3])
                             : "r"(lane_base + C::kColSfa + 4 * (acc * kMB + mb)));
            }
            uint32_t r[kQPerWarp][32];
#pragma unroll
            for (int u = 0; u < kQPerWarp; ++u)
                tc::tc_ld_32x32b_x32(lane_base + (acc * kMB + mb) * kN + (q_lo + u) * kNPad, r[u]);
            tc::tc_wait_ld();
            const uint32_t sfw = quad == 0 ? sf4[0] : quad == 1 ? sf4[1] : quad == 2 ? sf4[2] : sf4[3];
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&S.acce[acc]);
            const int64_t cand = (int64_t)t * kSpan + m;
            const int64_t g0 = (int64_t)t * kSpan + mb * kTile + quad * 32;   // this warp's 32
            const int e0 = (int)(sfw & 255u), e1 = (int)((sfw >> 8) & 255u);
            const int e2 = (int)((sfw >> 16) & 255u), e3 = (int)(sfw >> 24);
            const int kmin = min(min(e0, e1), min(e2, e3)) - 127;
            const int kmax = max(max(e0, e1), max(e2, e3)) - 127;
            // the score chains of this warp's queries: straight-line over all 32 head slots
            // (a padded head has weight 0 and D = 0 from zero query codes, so its step adds +0
            // to a sum that is never -0)
            // (the chains of a warp's queries advance together: independent FMAs between
            // the dependent steps of each chain)
            float scs[kQPerWarp];
            if constexpr (!C::kDeferred) {
                // decode: one fma chain per query in head order
#pragma unroll
                for (int u = 0; u < kQPerWarp; ++u) scs[u] = 0.0f;
#pragma unroll
                for (int h4 = 0; h4 < kNPad / 4; ++h4) {
                    float wh[kQPerWarp][4];
#pragma unroll
                    for (int u = 0; u < kQPerWarp; ++u) {
                        const float4 wv = reinterpret_cast<const float4 *>(S.w[q_lo + u])[h4];
                        wh[u][0] = wv.x; wh[u][1] = wv.y; wh[u][2] = wv.z; wh[u][3] = wv.w;
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
#pragma unroll
                        for (int u = 0; u < kQPerWarp; ++u) {
                            const float D = __uint_as_float(r[u][4 * h4 + j]);
                            scs[u] = __fmaf_rn(wh[u][j], D > 0.0f ? D : 0.0f, scs[u]);
                        }
                    }
                }
            } else {
                // prefill chunks: eight independent partial sums per query (head h goes to
                // lane h % 2 of packed accumulator (h / 2) % 4), four fused steps deep, then a
                // fixed tree -- the chain's latency no longer paces the epilogue.  Any order
                // keeps the float score within the bound the exact selection uses.
#pragma unroll
                for (int u = 0; u < kQPerWarp; ++u) {
                    unsigned long long acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                    for (int h8 = 0; h8 < kNPad / 8; ++h8) {
                        const float4 wa = reinterpret_cast<const float4 *>(S.w[q_lo + u])[2 * h8];
                        const float4 wb = reinterpret_cast<const float4 *>(S.w[q_lo + u])[2 * h8 + 1];
                        const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const float d0 = fmaxf(__uint_as_float(r[u][8 * h8 + 2 * j]), 0.0f);
                            const float d1 = fmaxf(__uint_as_float(r[u][8 * h8 + 2 * j + 1]), 0.0f);
                            asm("{\n\t.reg .b64 a, b;\n\tmov.b64 a, {%1, %2};\n\tmov.b64 b, {%3, %4};\n\t"
                                "fma.rn.f32x2 %0, a, b, %0;\n\t}"
                                : "+l"(acc[j]) : "f"(wv[2 * j]), "f"(wv[2 * j + 1]), "f"(d0), "f"(d1));
                        }
                    }
                    float lo[4], hi[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        lo[j] = __uint_as_float((uint32_t)acc[j]);
                        hi[j] = __uint_as_float((uint32_t)(acc[j] >> 32));
                    }
                    scs[u] = __fadd_rn(__fadd_rn(__fadd_rn(lo[0], hi[0]), __fadd_rn(lo[1], hi[1])),
                                       __fadd_rn(__fadd_rn(lo[2], hi[2]), __fadd_rn(lo[3], hi[3])));
                }
            }
#pragma unroll
            for (int u = 0; u < kQPerWarp; ++u) {
                const int qi = q_lo + u;
                const bool valid = cand < qlen[u];
                uint32_t key = 0;
                float sc = scs[u];
                if constexpr (!C::kDeferred) {
                    // rare: positions whose tensor-core result cannot be proven exact
                    const bool unsafe = valid && ((kmax - kmin) + qspan[u] > 9 || qmin[u] + kmin - 2 < -126 ||
                                                  qmax[u] + kmax - 2 > 100);
                    const uint32_t todo = __ballot_sync(0xffffffffu, unsafe);
                    if (todo)
                        sc = rescore_flagged<C::kDeferred>(todo, sc, sfw, g0, P.kc + kbase * kRowBytes, pool, P.pool_mode,
                                             P.n_keys, S.b, reinterpret_cast<const uint8_t *>(S.sfb), S.w[qi],
                                             qi, H);
                }
                if (valid) {
                    key = score_key(sc);
                    out_of_range |= !(fabsf(sc) <= 3.4028234663852886e38f);
                    if (fused) S.fkeys[(t - (int)blockIdx.x * R) * kSpan + m] = key;
                    else P.scores[(row0 + qi) * P.n_cand + cand] = sc;
                }
                if (P.gmax && !fused) {  // this warp's 32 candidates are one aligned group
                    const uint32_t gk = __reduce_max_sync(0xffffffffu, key);
                    if (lane == 0 && g0 < qlen[u]) P.gmax[(row0 + qi) * P.G + (g0 >> 5)] = gk;
                }
            }
        }
        // ---- the flagged stages, after every epilogue warp has written its scores: each
        //      position is checked per query and re-scored exactly where the MMA result may
        //      be rounded; the group maxima around re-scored positions are recomputed
        if constexpr (C::kDeferred) {
            if (!ewaited) pdl_wait();             // the re-checks read key rows of any position
            asm volatile("bar.sync 3, %0;" ::"r"((kEpiWarps + 1) * 32) : "memory");
            if (!S.abort_flag) {
                const int nwords = (ntr + 31) >> 5;
                int seen = 0;
#pragma unroll 1
                for (int wi = 0; wi < nwords; ++wi) {
                    uint32_t bits = S.flag_bits[wi];
#pragma unroll 1
                    while (bits) {
                        const int bit = __ffs(bits) - 1;
                        bits &= bits - 1u;
                        if (seen++ % kEpiWarps != ew) continue;
                        recheck_stage<QG, FU>(P, S, wi * 32 + bit, kSpan, row0, t0q, kbase, pool, n_blk_all);
                    }
                }
            }
        }
        if (__any_sync(0xffffffffu, out_of_range) && lane == 0) dev_flag(P.d_status, CSA2_DEV_SCORE_RANGE);
    }

    tc::tc_fence_before();
    __syncthreads();
    if (early) pdl_wait();                         // before the counters and lists are touched
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, C::kTmemCols);
    }
    if constexpr (QG == 1) {
        if (fused && !S.abort_flag) {
            const int64_t pos0 = (int64_t)blockIdx.x * R * kSpan;
            int64_t v = S.qlen[0] - pos0;
            v = v < 0 ? 0 : (v > (int64_t)R * kSpan ? (int64_t)R * kSpan : v);
            fused_list<QG, FU>(P, S, row0, pos0, (int)v);
        }
    }
    if (tid == 0) {
        if (S.abort_flag) dev_flag(P.d_status, CSA2_DEV_TIMEOUT);
        // the group's last CTA to finish sets both counters back to zero for the next call
        __threadfence();
        if (atomicAdd(&P.tile_done[unit], 1u) == gridDim.x - 1u) {
            P.tile_ctr[unit] = 0u;
            P.tile_done[unit] = 0u;
        }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Queries per CTA: 4 for a chunk of queries scored against a shared cache (Full mode,
// at least 8 queries a sequence, and few enough stages for the stage flags), else 1.
int tc_query_group(const csa2_index_args &a)
{
    const int64_t stages = ((int64_t)a.n_keys + kSpanOf<4> - 1) / kSpanOf<4>;
    return a.mode != CSA2_INDEX_POOL && a.n_q >= 8 && stages <= (int64_t)kFlagWords * 32 ? 4 : 1;
}

// CTAs per unit (QG queries): enough units x CTAs to fill the resident CTAs of every SM,
// at most one per stage (span positions) of the unit.
int64_t tc_splits(int64_t units, int64_t n_cand, int ctas_per_sm, int span)
{
    const int64_t tiles = (n_cand + span - 1) / span;
    int64_t s = (int64_t)device_sm_count() * ctas_per_sm / (units > 0 ? units : 1);
    if (s < 1) s = 1;
    if (s > tiles) s = tiles > 0 ? tiles : 1;
    return s;
}

template <int QG, bool FU>
cudaError_t launch_tc(const CUtensorMap &map, const TcParams &P, int64_t units, int64_t splits,
                      cudaStream_t s)
{
    const size_t smem = sizeof(TcSmem<QG, FU>) + 1024;
    cudaError_t e = cudaFuncSetAttribute(index_score_tc_kernel<QG, FU>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // the whole unified L1 as shared memory, so the resident CTAs fit on every SM
    e = cudaFuncSetAttribute(index_score_tc_kernel<QG, FU>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    return launch_pdl(index_score_tc_kernel<QG, FU>, dim3((unsigned)splits, (unsigned)units),
                      dim3(kThreadsOf<QG>), smem, s, 1, map, P);
}

} // namespace

bool index_tc_eligible(const csa2_index_args &a)
{
    if (a.head_dim != kD || a.n_heads > kNPad) return false;
    if (((uintptr_t)a.q & 15) != 0) return false;           // 16-byte query loads
    if (a.mode == CSA2_INDEX_POOL && a.block != 8) return false;
    if ((int64_t)a.batch * a.n_keys >= (int64_t(1) << 31)) return false;
    if (((uintptr_t)a.k_codes & 15) != 0) return false;
    return encode_fn() != nullptr;
}

// CTAs per unit of QG queries (see tc_query_group).
int64_t index_tc_ctas_per_row(const csa2_index_args &a)
{
    const int qg = tc_query_group(a);
    const int64_t units = (int64_t)a.batch * ((a.n_q + qg - 1) / qg);
    const int64_t n_cand = a.mode == CSA2_INDEX_POOL ? (int64_t)a.n_pool_blocks * a.block : a.n_keys;
    return qg == 4 ? tc_splits(units, n_cand, Cfg<4>::kCtasPerSm, kSpanOf<4>)
                   : tc_splits(units, n_cand, Cfg<1>::kCtasPerSm, kSpanOf<1>);
}

// Fused selection (csa2_index_topk): one query per CTA in FULL mode, each CTA a fixed run
// of at most kFuseStages stages, so the row takes at least stages / kFuseStages CTAs.
bool index_tc_fusable(const csa2_index_args &a)
{
    return index_tc_eligible(a) && a.mode != CSA2_INDEX_POOL && tc_query_group(a) == 1;
}

void index_fused_shape(const csa2_index_args &a, int64_t &ctas, int &stages)
{
    const int64_t ntr = ((int64_t)a.n_keys + kSpanOf<1> - 1) / kSpanOf<1>;
    int64_t c = index_tc_ctas_per_row(a);
    const int64_t need = (ntr + kFuseStages - 1) / kFuseStages;
    if (c < need) c = need;
    if (c < 1) c = 1;
    stages = (int)(ntr > 0 ? (ntr + c - 1) / c : 1);
    if (stages < 1) stages = 1;
    ctas = ntr > 0 ? (ntr + stages - 1) / stages : 1;
}

cudaError_t launch_index_tc(const csa2_index_args &a, float *scores, int32_t *row_len,
                            uint32_t *tile_ctr, uint32_t *d_status, cudaStream_t s, const FusedOut *fo)
{
    const int qg = tc_query_group(a);
    int64_t splits = index_tc_ctas_per_row(a);
    const int64_t rows = (int64_t)a.batch * a.n_q;
    const int64_t units = (int64_t)a.batch * ((a.n_q + qg - 1) / qg);
    TcParams P;
    P.n_q = a.n_q;
    P.H = a.n_heads;
    P.ratio_m = a.ratio_m;
    P.block = a.block;
    P.n_pool_blocks = a.n_pool_blocks;
    P.n_keys = a.n_keys;
    P.pool_mode = a.mode == CSA2_INDEX_POOL;
    P.n_cand = P.pool_mode ? (int64_t)a.n_pool_blocks * a.block : a.n_keys;
    P.q = a.q;
    P.w = a.w;
    P.kc = a.k_codes;
    P.ks = a.k_scales;
    P.q_pos = a.q_pos;
    P.pool = a.pool_blocks;
    P.scores = scores;
    P.row_len = row_len;
    P.gmax = a.group_max;
    P.G = (P.n_cand + 31) / 32;
    P.tile_ctr = tile_ctr;
    P.tile_done = tile_ctr + rows;
    P.d_status = d_status;
    P.lst_key = nullptr;
    P.lst_pos = nullptr;
    P.lst_meta = nullptr;
    P.lst_k = 0;
    P.lst_stages = 0;
    P.fresh_from = a.mode == CSA2_INDEX_POOL ? 0 : a.fresh_from;
    if (fo) {                                  // no scores, no group maxima: candidate lists
        if (qg != 1 || P.pool_mode) return cudaErrorInvalidValue;
        int64_t ctas;
        int stages;
        index_fused_shape(a, ctas, stages);
        splits = ctas;
        P.scores = nullptr;
        P.gmax = nullptr;
        P.lst_key = fo->key;
        P.lst_pos = fo->pos;
        P.lst_meta = fo->meta;
        P.lst_k = fo->k;
        P.lst_stages = stages;
    }

    CUtensorMap map;
    cuuint64_t dims[2] = {(cuuint64_t)kRowBytes, (cuuint64_t)((int64_t)a.batch * a.n_keys)};
    cuuint64_t strides[1] = {(cuuint64_t)kRowBytes};
    cuuint32_t box[2] = {(cuuint32_t)kRowBytes,
                         (cuuint32_t)(P.pool_mode ? 8 : (qg == 4 ? kSpanOf<4> : kSpanOf<1>))};
    cuuint32_t estr[2] = {1, 1};
    if (dims[1] == 0) dims[1] = 1;
    CUresult r = encode_fn()(&map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(a.k_codes),
                             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                             CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (qg == 4) return launch_tc<4, false>(map, P, units, splits, s);
    return fo ? launch_tc<1, true>(map, P, units, splits, s) : launch_tc<1, false>(map, P, units, splits, s);
}

} // namespace csa2
