// topk.cu -- Top-K selection (csa2_topk) and the block pool (csa2_block_candidates).
//
// DeepSeek-V4.1-Flash report (aipaper.jasonlin.tech) §2.3: the indexer keeps the Top-K
// entries per query (K = 512, §4.2.1); §2.3.2 and Figure 5: the decoder's first Full
// layer gives each block of 8 positions the maximum index score among its positions and
// keeps the best blocks (at most 2,048).  Ties go to the lower index; output ascending.
//
// Selection is an exact radix select on an order-preserving 32-bit key of each score:
// four 8-bit digit passes (most significant first) find the K-th key tau and how many
// entries equal to tau must be taken; a final pass in index order emits every entry
// above tau and the first `need` entries equal to tau, which yields ascending output.
#include "common.cuh"
#include "exact.cuh"
#include "internal.h"


namespace csa2 {
namespace {

constexpr int kTopkThreads = 1024;

__device__ __forceinline__ int64_t cand_pos(const int32_t *pool_row, int32_t block, int64_t i)
{
    if (!pool_row) return i;
    const uint32_t u = (uint32_t)i, b = (uint32_t)block;    // candidates < 2^31: 32-bit division
    return (int64_t)pool_row[u / b] * block + (int64_t)(u % b);
}

// Block-wide exclusive prefix count of a 1-bit flag (all threads must call).
__device__ __forceinline__ uint32_t block_excl_count(bool f, uint32_t *s_warp, uint32_t &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t bal = __ballot_sync(0xffffffffu, f);
    const uint32_t in_warp = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0) s_warp[warp] = __popc(bal);
    __syncthreads();
    if (warp == 0) {
        uint32_t v = lane < (int)(blockDim.x >> 5) ? s_warp[lane] : 0u;
        uint32_t incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        s_warp[lane] = incl - v;             // exclusive
        if (lane == 31) s_warp[32] = incl;   // total
    }
    __syncthreads();
    const uint32_t r = s_warp[warp] + in_warp;
    total = s_warp[32];
    __syncthreads();
    return r;
}

// Block-wide exclusive prefix sum of one value per thread (all threads must call).
__device__ __forceinline__ uint32_t block_excl_count_sum(uint32_t v, uint32_t *s_warp, uint32_t &total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const uint32_t w = lane < (int)(blockDim.x >> 5) ? s_warp[lane] : 0u;
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

// Whole-row radix select by one CTA of kTopkThreads threads, reading the row from global
// memory in four 8-bit digit passes.  The fallback of the group-max path for rows whose
// candidates do not fit on chip (heavy ties), and the path for more than 2^31 rows.
__device__ __noinline__ void radix_select_row(const float *__restrict__ scores, int64_t n,
                                              const int32_t *__restrict__ row_len,
                                 const int32_t *__restrict__ pool, int32_t block, int32_t k,
                                 int32_t *__restrict__ idx, float *__restrict__ out_scores, int64_t row)
{
    __shared__ uint32_t s_hist[256];
    __shared__ uint32_t s_warp[33];
    __shared__ uint32_t s_prefix, s_mask, s_remaining;

    const int tid = threadIdx.x, lane = tid & 31;
    int64_t len = row_len ? (int64_t)row_len[row] : n;
    len = len < 0 ? 0 : (len > n ? n : len);
    const float *s = scores + row * n;
    const int32_t *pool_row = pool ? pool + row * (n / block) : nullptr;
    int32_t *out = idx + row * (int64_t)k;
    float *out_s = out_scores ? out_scores + row * (int64_t)k : nullptr;

    if (len <= k) {                          // everything competes and wins
        for (int64_t i = tid; i < k; i += kTopkThreads) {
            out[i] = i < len ? (int32_t)cand_pos(pool_row, block, i) : -1;
            if (out_s) out_s[i] = i < len ? s[i] : 0.0f;
        }
        return;
    }

    if (tid == 0) { s_prefix = 0; s_mask = 0; s_remaining = (uint32_t)k; }
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = tid; i < 256; i += kTopkThreads) s_hist[i] = 0;
        __syncthreads();
        const uint32_t prefix = s_prefix, mask = s_mask;
        for (int64_t base = 0; base < len; base += kTopkThreads) {
            const int64_t i = base + tid;
            uint32_t key = 0;
            bool act = false;
            if (i < len) {
                key = score_key(s[i]);
                act = (key & mask) == prefix;
            }
            const uint32_t am = __ballot_sync(0xffffffffu, act);
            if (act) {
                const uint32_t digit = (key >> shift) & 255u;
                const uint32_t peers = __match_any_sync(am, digit);
                if (lane == __ffs(peers) - 1) atomicAdd(&s_hist[digit], (uint32_t)__popc(peers));
            }
        }
        __syncthreads();
        if (tid == 0) {
            uint32_t cum = 0, rem = s_remaining;
            for (int d = 255; d >= 0; --d) {
                const uint32_t h = s_hist[d];
                if (cum + h >= rem) {
                    s_prefix = prefix | ((uint32_t)d << shift);
                    s_mask = mask | (255u << shift);
                    s_remaining = rem - cum;
                    break;
                }
                cum += h;
            }
        }
        __syncthreads();
    }
    const uint32_t tau = s_prefix;
    const uint32_t need = s_remaining;       // entries equal to tau still to take

    uint32_t base_eq = 0, base_sel = 0;
    for (int64_t base = 0; base < len && base_sel < (uint32_t)k; base += kTopkThreads) {
        const int64_t i = base + tid;
        uint32_t key = 0;
        float v = 0.0f;
        if (i < len) { v = s[i]; key = score_key(v); }
        const bool gt = i < len && key > tau;
        const bool eq = i < len && key == tau;
        uint32_t tot_eq, tot_sel;
        const uint32_t eq_rank = base_eq + block_excl_count(eq, s_warp, tot_eq);
        const bool sel = gt || (eq && eq_rank < need);
        const uint32_t sel_rank = base_sel + block_excl_count(sel, s_warp, tot_sel);
        if (sel && sel_rank < (uint32_t)k) {
            out[sel_rank] = (int32_t)cand_pos(pool_row, block, i);
            if (out_s) out_s[sel_rank] = v;
        }
        base_eq += tot_eq;
        base_sel += tot_sel;
    }
}

__global__ void __launch_bounds__(kTopkThreads)
topk_radix_kernel(const float *__restrict__ scores, int64_t n, const int32_t *__restrict__ row_len,
                  const int32_t *__restrict__ pool, int32_t block, int32_t k,
                  int32_t *__restrict__ idx, float *__restrict__ out_scores)
{
    radix_select_row(scores, n, row_len, pool, block, k, idx, out_scores, blockIdx.x);
}

// ------------------------------------------------------------------ group-max select
// Pass 1 (group_max32_kernel / group_max_kernel): the largest key of every group of gs
// consecutive candidates, spread over the whole GPU.  Pass 2 (topk_gmax_kernel, one CTA
// per row): tau0 = the k-th largest group key.  Each of those k groups holds an element
// >= tau0, so at least k elements are >= tau0 and every element of the top-k is >= tau0;
// only groups whose key is >= tau0 can hold one.  Any lower bound of tau0 keeps that
// property, so tau0 is taken to 22 of its 32 bits.  Those groups' elements >= the bound
// are gathered on chip in position order, and an exact radix select among them (key
// desc, position asc) gives the top-k, emitted in order.
constexpr int kGThreads = 1024;
constexpr int kGBins = 2048;
constexpr int kListCap = 8192;          // candidate groups per row listed on chip
constexpr int kMaxGroups = 32768;       // group keys per row (on chip; longer rows: wider groups)
constexpr int kCandCap = 16384;         // candidates per row kept on chip (a whole
                                        // 2,048-block pool of 8 positions fits)

struct GSmem {
    uint32_t coarse[2][kGBins / 32];   // the same counts per 32 consecutive bins
    uint32_t hist[2][kGBins];    // double buffer: the next digit pass clears one while
    uint32_t warp[33];           // the current one counts into the other
    uint32_t pick[2];
};

// One thread per group of 32 whose row starts 16-byte aligned: eight 16-byte loads in
// flight at once, no cross-lane work.
__global__ void __launch_bounds__(256) group_max32_kernel(const float *__restrict__ scores, int64_t n,
                                                          const int32_t *__restrict__ row_len, int64_t rows,
                                                          int64_t G, uint32_t *__restrict__ gkeys)
{
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= rows * G) return;
    const int64_t row = t / G, g = t % G;
    int64_t len = row_len ? (int64_t)row_len[row] : n;
    len = len < 0 ? 0 : (len > n ? n : len);
    const int64_t p0 = g * 32;
    uint32_t m = 0;
    if (p0 + 32 <= len) {
        const float4 *src = reinterpret_cast<const float4 *>(scores + row * n + p0);
        float4 f[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = src[e];
#pragma unroll
        for (int e = 0; e < 8; ++e)
            m = max(max(max(m, score_key(f[e].x)), score_key(f[e].y)), max(score_key(f[e].z), score_key(f[e].w)));
    } else {
        for (int64_t p = p0; p < p0 + 32 && p < len; ++p) m = max(m, score_key(scores[row * n + p]));
    }
    gkeys[t] = m;
}

__global__ void __launch_bounds__(256) group_max_kernel(const float *__restrict__ scores, int64_t n,
                                                        const int32_t *__restrict__ row_len, int64_t rows,
                                                        int32_t gs, int64_t G, uint32_t *__restrict__ gkeys)
{
    const int lane = threadIdx.x & 31;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t w = warp0; w < rows * G; w += nwarps) {
        const int64_t row = w / G, g = w % G;
        int64_t len = row_len ? (int64_t)row_len[row] : n;
        len = len < 0 ? 0 : (len > n ? n : len);
        const float *s = scores + row * n;
        uint32_t m = 0;
        for (int64_t p = g * gs + lane; p < (g + 1) * gs && p < len; p += 32) m = max(m, score_key(s[p]));
        m = __reduce_max_sync(0xffffffffu, m);
        if (lane == 0) gkeys[row * G + g] = m;
    }
}

// k-th largest key of n keys in shared memory by digit passes of 11, 11 and 10 bits.
// With all three passes: the exact key tau, and in need how many keys equal to tau belong
// to the top k.  With the first `passes` only: tau with its unresolved low bits zero, a
// lower bound of the exact key (need is then meaningless).
// Each pass: one histogram of the keys that match the digits found so far, counted per
// bin and per 32 consecutive bins (the other buffers are cleared meanwhile for the next
// pass), then warp 0 alone finds the digit in two warp scans from the top -- over the
// coarse counts, then over the 32 bins of the coarse bin that reaches `remaining` -- so a
// pass costs two block barriers.
__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}
template <class KeyAt>
__device__ __forceinline__ uint32_t g_threshold_at(KeyAt key_at, int n, uint32_t k, GSmem &S, uint32_t &need,
                                                int passes)
{
    const int tid = threadIdx.x, lane = tid & 31;
    uint32_t prefix = 0, mask = 0, remaining = k;
    for (int i = tid; i < kGBins; i += kGThreads) S.hist[0][i] = 0;
    if (tid < kGBins / 32) S.coarse[0][tid] = 0;
    __syncthreads();
#pragma unroll 1
    for (int pass = 0; pass < passes; ++pass) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0), nb = pass < 2 ? 2048 : 1024;
        uint32_t *h = S.hist[pass & 1], *hc = S.coarse[pass & 1];
        if (pass + 1 < passes) {
            for (int i = tid; i < kGBins; i += kGThreads) S.hist[(pass + 1) & 1][i] = 0;
            if (tid < kGBins / 32) S.coarse[(pass + 1) & 1][tid] = 0;
        }
        for (int base = 0; base < n; base += kGThreads) {
            const int i = base + tid;
            uint32_t key = 0;
            bool act = false;
            if (i < n) {
                key = key_at(i);
                act = (key & mask) == prefix;
            }
            const uint32_t am = __ballot_sync(0xffffffffu, act);
            if (act) {
                const uint32_t digit = (key >> shift) & (uint32_t)(nb - 1);
                const uint32_t peers = __match_any_sync(am, digit);
                if (lane == __ffs(peers) - 1) {
                    atomicAdd(&h[digit], (uint32_t)__popc(peers));
                    atomicAdd(&hc[digit >> 5], (uint32_t)__popc(peers));
                }
            }
        }
        __syncthreads();
        if (tid < 32) {
            // coarse bins from the top: lane L holds bin ncb-1-L, and bin 31-L when ncb = 64
            const int ncb = nb >> 5;
            const uint32_t c0 = hc[ncb - 1 - lane], c1 = ncb == 64 ? hc[31 - lane] : 0u;
            const uint32_t i0 = warp_incl_scan(c0, lane);
            const uint32_t i1 = warp_incl_scan(c1, lane) + __shfl_sync(0xffffffffu, i0, 31);
            const uint32_t b0 = __ballot_sync(0xffffffffu, i0 >= remaining);
            const uint32_t b1 = __ballot_sync(0xffffffffu, i1 >= remaining);
            int cb;
            uint32_t above;
            if (b0) {
                const int L = __ffs(b0) - 1;
                cb = ncb - 1 - L;
                above = __shfl_sync(0xffffffffu, i0 - c0, L);
            } else {
                const int L = b1 ? __ffs(b1) - 1 : 31;
                cb = 31 - L;
                above = __shfl_sync(0xffffffffu, i1 - c1, L);
            }
            // the 32 bins of coarse bin cb, from the top
            const uint32_t f = h[cb * 32 + 31 - lane];
            const uint32_t fi = warp_incl_scan(f, lane) + above;
            const uint32_t bf = __ballot_sync(0xffffffffu, fi >= remaining);
            const int Lf = bf ? __ffs(bf) - 1 : 31;
            const uint32_t fabove = __shfl_sync(0xffffffffu, fi - f, Lf);
            if (lane == 0) {
                S.pick[0] = (uint32_t)(cb * 32 + 31 - Lf);
                S.pick[1] = remaining - fabove;
            }
        }
        __syncthreads();
        prefix |= S.pick[0] << shift;
        mask |= (uint32_t)(nb - 1) << shift;
        remaining = S.pick[1];
    }
    need = remaining;
    return prefix;
}
__device__ __forceinline__ uint32_t g_threshold(const uint32_t *keys, int n, uint32_t k, GSmem &S,
                                             uint32_t &need, int passes)
{
    return g_threshold_at([keys](int i) { return keys[i]; }, n, k, S, need, passes);
}

// ------------------------------------------------------------------ exact order (csa2_topk and
// csa2_block_candidates with an exact context)
// The float32 scores s~ the indexer writes are within (H + 2) 2^-24 A + 2^-149 (sum|w| + H)
// of the exact scores s, A = sum_h |w_h| ReLU(d_h) (see csa2_index_score).  The kernel uses
// a bound e(x) >= that error for a candidate whose s~ is x, non-decreasing in x and with
// x - e(x) rising.  With tau~ the k-th largest s~:
//   s~ < lo = tau~ - 2 e(tau~): at least k candidates (those with s~ >= tau~) have
//     s >= tau~ - e(tau~) > s, so the candidate is out;
//   s~ > hi = tau~ + e(tau~) + e(tau~ + 3 e(tau~)): such an s~ has s~ - e(s~) > tau~ + e(tau~);
//     any candidate with s >= this one's s then has s~ > tau~, and fewer than k do, so it
//     is in;
//   the rest (the band) are re-scored exactly and the k - (#in) best of them taken by
//   (exact score desc, candidate asc).
// e: for rows with every w_h >= 0, A_t = s_t <= (s~_t + eta) / (1 - c), so
// e(x) = c (x + eta) / (1 - c) + eta; otherwise one row-wide A through |d_h| <= sum_b 12
// sum_i |2 q_i| 2^(Xq_b + Xk_b - 2), Xk_b the largest key scale exponent of block b in the
// sequence (one pass over its scale bytes).
struct ExactArgs {
    int H, d;                      // indexer heads, head dim (32, 64 or 128)
    int32_t n_q;                   // queries per sequence (row r belongs to sequence r / n_q)
    int64_t n_keys;                // key rows per sequence
    const uint16_t *q;             // [rows, H, d] bf16
    const float *w;                // [rows, H]
    const uint8_t *kc, *ks;        // [B, N, d/2], [B, N, d/32]
    int unit;                      // 1: candidates are positions; > 1: blocks of `unit` positions
    const float *pos_scores;       // unit > 1: position scores [rows, pos_n]
    int64_t pos_n;
    const int32_t *pos_len;        // unit > 1: valid positions per row
    uint32_t *band;                // [gridDim.x][kLimbs][CSA2_EXACT_BAND_CAP] exact keys
    uint32_t *d_status;
};
constexpr int kBandCap = CSA2_EXACT_BAND_CAP;
static_assert(kBandCap <= 2 * kGThreads, "two band entries per thread at most");

// Block-wide min and max of one value per thread (all threads call; ends with a barrier).
__device__ __forceinline__ void block_minmax(uint32_t vmin, uint32_t vmax, uint32_t *s_red, uint32_t &mn, uint32_t &mx)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    vmin = __reduce_min_sync(0xffffffffu, vmin);
    vmax = __reduce_max_sync(0xffffffffu, vmax);
    if (lane == 0) { s_red[warp] = vmin; s_red[32 + warp] = vmax; }
    __syncthreads();
    mn = 0xffffffffu; mx = 0u;
    for (int i = 0; i < nw; ++i) { mn = min(mn, s_red[i]); mx = max(mx, s_red[32 + i]); }
    __syncthreads();
}

// Largest scale byte of each 32-value block over the n_keys key rows of one sequence
// (byte b of the result = block b, nb in {1, 2, 4}); block-wide, ends with a barrier.
__device__ __noinline__ uint32_t key_scale_max(const uint8_t *ks, int64_t n_keys, int nb, uint32_t *s_red)
{
    const int64_t nbytes = n_keys * nb;
    uint32_t r = 0;                           // byte b: largest scale byte of block b
    int64_t i0 = 0;
    if (((uintptr_t)ks & 3u) == 0) {
        // byte j of word v is byte 4v + j, of block (4v + j) % nb = j % nb
        uint32_t m = 0;
        const uint32_t *w4 = reinterpret_cast<const uint32_t *>(ks);
        for (int64_t v = threadIdx.x; v < nbytes / 4; v += blockDim.x) m = __vmaxu4(m, w4[v]);
        for (int j = 0; j < 4; ++j) r = __vmaxu4(r, ((m >> (8 * j)) & 255u) << (8 * (j % nb)));
        i0 = nbytes / 4 * 4;
    }
    for (int64_t i = i0 + threadIdx.x; i < nbytes; i += blockDim.x)
        r = __vmaxu4(r, (uint32_t)ks[i] << (8 * (int)(i % nb)));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) r = __vmaxu4(r, __shfl_xor_sync(0xffffffffu, r, o));
    if (lane == 0) s_red[warp] = r;
    __syncthreads();
    uint32_t t = 0;
    for (int i = 0; i < nw; ++i) t = __vmaxu4(t, s_red[i]);
    __syncthreads();
    return t;
}

__device__ __noinline__ RowBound row_bound(const exact::QuantQuery &Q, const ExactArgs &X, int64_t seq,
                                           uint32_t *s_red)
{
    bool neg;
    RowBound rb = row_bound_nonneg(Q.w, X.H, neg);
    if (!neg) return rb;
    const float c = rb.c1;
    const float eta = rb.c0;
    const int nb = X.d / 32;
    const uint32_t km = key_scale_max(X.ks + seq * X.n_keys * nb, X.n_keys, nb, s_red);
    float A = 0.0f;
    for (int h = 0; h < X.H; ++h) {
        float ah = 0.0f;
        for (int b = 0; b < nb; ++b) {
            const int ex = Q.qx[h * 4 + b] + (int)((km >> (8 * b)) & 255u) - 127 - 2;
            const float p2 = ex < -149 ? 0x1p-149f : ldexpf(1.0f, ex);      // rounded up
            ah = __fmaf_ru(12.0f * (float)Q.q1[h * 4 + b], p2, ah);
        }
        A = __fmaf_ru(fabsf(Q.w[h]), ah, A);
    }
    rb.c0 = __fmaf_ru(c, A, eta);                     // an overflow to +inf puts every candidate in the band
    return rb;
}

// Exact key (limb `lane`) of band candidate i of a row: a position (through the pool), or
// the largest exact score of a block's positions whose float32 score could be its maximum.
template <int D>
__device__ __noinline__ uint32_t unit_key(const exact::QuantQuery &Q, const ExactArgs &X, int64_t row, int64_t seq,
                                          const int32_t *pool_row, int32_t block, int64_t i, uint32_t unit_lo_key)
{
    const int64_t kbase = seq * X.n_keys;
    if (X.unit == 1) {
        int64_t p = cand_pos(pool_row, block, i);
        p = p < 0 ? 0 : (p >= X.n_keys ? X.n_keys - 1 : p);
        return exact::score_key_limb<D>(Q, X.H, X.kc + (kbase + p) * (D / 2), X.ks + (kbase + p) * (D / 32));
    }
    int64_t len = X.pos_len[row];
    len = len < 0 ? 0 : (len > X.pos_n ? X.pos_n : len);
    const float *ps = X.pos_scores + row * X.pos_n;
    uint32_t best = 0;
    bool have = false;
#pragma unroll 1
    for (int j = 0; j < X.unit; ++j) {
        const int64_t p = i * X.unit + j;
        if (p >= len || p >= X.n_keys) break;
        if (score_key(ps[p]) < unit_lo_key) continue;          // cannot be the block's maximum
        const uint32_t l = exact::score_key_limb<D>(Q, X.H, X.kc + (kbase + p) * (D / 2),
                                                    X.ks + (kbase + p) * (D / 32));
        if (!have || exact::compare_keys(l, best) > 0) best = l;
        have = true;
    }
    return best;
}

// Fixed-point exact score (V, E) of band candidate i (see exact::score_fixed); for a block,
// the largest over its positions that could be its maximum.  false: the 128-bit form does
// not hold it (the caller takes the wide path).
template <int D>
__device__ __noinline__ bool unit_fixed(const exact::QuantQuery &Q, const ExactArgs &X, int64_t row, int64_t seq,
                                        const int32_t *pool_row, int32_t block, int64_t i, uint32_t unit_lo_key,
                                        __int128 &V, int &E)
{
    const int64_t kbase = seq * X.n_keys;
    if (X.unit == 1) {
        int64_t p = cand_pos(pool_row, block, i);
        p = p < 0 ? 0 : (p >= X.n_keys ? X.n_keys - 1 : p);
        return exact::score_fixed<D>(Q, X.H, X.kc + (kbase + p) * (D / 2), X.ks + (kbase + p) * (D / 32), V, E);
    }
    int64_t len = X.pos_len[row];
    len = len < 0 ? 0 : (len > X.pos_n ? X.pos_n : len);
    const float *ps = X.pos_scores + row * X.pos_n;
    bool have = false;
    V = 0;
    E = exact::kNoTerms;
#pragma unroll 1
    for (int j = 0; j < X.unit; ++j) {
        const int64_t p = i * X.unit + j;
        if (p >= len || p >= X.n_keys) break;
        if (score_key(ps[p]) < unit_lo_key) continue;          // cannot be the block's maximum
        __int128 v;
        int e;
        if (!exact::score_fixed<D>(Q, X.H, X.kc + (kbase + p) * (D / 2), X.ks + (kbase + p) * (D / 32), v, e))
            return false;
        if (!have) { V = v; E = e; have = true; continue; }
        const int em = min(E, e);
        if (!exact::align_fixed(V, E, em) || !exact::align_fixed(v, e, em)) return false;
        E = em;
        if (v > V) V = v;
    }
    return true;
}

// Among n_band band units whose exact keys are in bk (nwords words each, most significant
// last, word-major with stride kBandCap, compared as unsigned), sets
// state[u] = 1 for the `take` best by (key desc, unit index asc): limb by limb from the top,
// the take-th largest limb value among the units still tied splits them into taken, tied
// and dropped.  Block-wide; act and vals are scratch of n_band entries in shared memory.
__device__ __noinline__ void select_band(const uint32_t *bk, int nwords, int n_band, uint32_t take, uint8_t *state,
                                         uint32_t *act, uint32_t *vals, GSmem &S, uint32_t *s_red)
{
    const int tid = threadIdx.x;
    for (int i = tid; i < n_band; i += kGThreads) { state[i] = 0; act[i] = (uint32_t)i; }
    __syncthreads();
    int n_act = n_band;
    uint32_t remaining = take;
#pragma unroll 1
    for (int j = nwords - 1; j >= 0; --j) {
        if (remaining == 0 || remaining >= (uint32_t)n_act) break;
        uint32_t vmin = 0xffffffffu, vmax = 0u;
        for (int i = tid; i < n_act; i += kGThreads) {
            const uint32_t v = bk[(size_t)j * kBandCap + act[i]];
            vals[i] = v;
            vmin = min(vmin, v);
            vmax = max(vmax, v);
        }
        uint32_t mn, mx;
        block_minmax(vmin, vmax, s_red, mn, mx);           // barrier: vals visible
        if (mn == mx) continue;                             // this limb ties them all
        uint32_t need_eq;
        const uint32_t v = g_threshold(vals, n_act, remaining, S, need_eq, 3);
        const int r0 = min(2 * tid, n_act), r1 = min(r0 + 2, n_act);
        uint32_t keep0 = 0, keep1 = 0;
        int nk = 0;
        for (int i = r0; i < r1; ++i) {
            if (vals[i] > v) state[act[i]] = 1;
            else if (vals[i] == v) { if (nk == 0) keep0 = act[i]; else keep1 = act[i]; ++nk; }
        }
        uint32_t tot;
        const uint32_t at = block_excl_count_sum((uint32_t)nk, S.warp, tot);   // all reads done
        if (nk > 0) act[at] = keep0;
        if (nk > 1) act[at + 1] = keep1;
        __syncthreads();
        n_act = (int)tot;
        remaining = need_eq;
    }
    for (int i = tid; i < n_act && i < (int)remaining; i += kGThreads) state[act[i]] = 1;
    __syncthreads();
}

// Block-wide exclusive max-scan of one value per thread in thread order (identity 0; all
// threads call; ends with a barrier).
__device__ __forceinline__ uint32_t block_excl_max(uint32_t v, uint32_t *s_warp)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl = max(incl, t);
    }
    uint32_t excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = 0u;
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const uint32_t wv = lane < nw ? s_warp[lane] : 0u;
        uint32_t wi = wv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t t = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi = max(wi, t);
        }
        uint32_t we = __shfl_up_sync(0xffffffffu, wi, 1);
        if (lane == 0) we = 0u;
        s_warp[lane] = we;
    }
    __syncthreads();
    const uint32_t r = max(s_warp[warp], excl);
    __syncthreads();
    return r;
}

// Key rows p and q of one sequence hold the same bytes (codes and scales).
template <int D>
__device__ __forceinline__ bool same_key_row(const ExactArgs &X, int64_t kbase, int64_t p, int64_t q)
{
    const uint4 *a = reinterpret_cast<const uint4 *>(X.kc + (kbase + p) * (D / 2));
    const uint4 *b = reinterpret_cast<const uint4 *>(X.kc + (kbase + q) * (D / 2));
    bool eq = true;
#pragma unroll
    for (int i = 0; i < D / 32; ++i) {
        const uint4 x = a[i], y = b[i];
        eq = eq && x.x == y.x && x.y == y.y && x.z == y.z && x.w == y.w;
    }
#pragma unroll
    for (int i = 0; i < D / 32; ++i) eq = eq && X.ks[(kbase + p) * (D / 32) + i] == X.ks[(kbase + q) * (D / 32) + i];
    return eq;
}

// Exact pass over a row's band (n_band candidates s_band[u] into the candidate arrays, in
// position order; take = how many of them are selected): sets s_state[u].  Runs of band
// candidates with equal float keys and byte-identical key rows have equal exact scores, so
// only the first of each run is scored.  Scores go first to 128-bit fixed point at one row
// exponent (4-word keys); where that form does not hold them, every candidate is scored as
// 26 limbs.  Either way the keys are selected word by word (select_band).  Block-wide.
template <int D>
__device__ __noinline__ void band_exact(const exact::QuantQuery &Q, const ExactArgs &X, const RowBound &rb,
                                        int64_t row, int64_t seq, const int32_t *pool_row, int32_t block,
                                        const uint32_t *s_band, const uint32_t *s_ck, const int32_t *s_cp,
                                        uint32_t n_band, uint32_t take, uint8_t *s_state, uint32_t *s_act,
                                        uint32_t *s_val, GSmem &S, uint32_t *s_red)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t *bk = X.band + (size_t)blockIdx.x * exact::kLimbs * kBandCap;   // [word][kBandCap]
    uint32_t *g_head = bk + 4 * kBandCap, *g_v = bk + 5 * kBandCap;          // rows 4 and 5..9
    const int64_t kbase = seq * X.n_keys;
    int32_t *s_pos = reinterpret_cast<int32_t *>(s_val);   // free until select_band
    // the single position that can hold each candidate's score (-1: several)
    for (uint32_t u = tid; u < n_band; u += kGThreads) {
        const uint32_t i = s_band[u];
        int64_t p = -1;
        if (X.unit == 1) {
            p = cand_pos(pool_row, block, s_cp[i]);
            p = p < 0 ? 0 : (p >= X.n_keys ? X.n_keys - 1 : p);
        } else {
            int64_t len = X.pos_len[row];
            len = len < 0 ? 0 : (len > X.pos_n ? X.pos_n : len);
            const float *ps = X.pos_scores + row * X.pos_n;
            const uint32_t ulo = score_key(rb.lo(key_value(s_ck[i])));
            int cnt = 0;
            for (int j = 0; j < X.unit; ++j) {
                const int64_t q = (int64_t)s_cp[i] * X.unit + j;
                if (q >= len || q >= X.n_keys) break;
                if (score_key(ps[q]) >= ulo) { p = q; ++cnt; }
            }
            if (cnt != 1) p = -1;
        }
        s_pos[u] = (int32_t)p;
    }
    __syncthreads();
    // run heads: thread t takes candidates 2t and 2t + 1
    uint32_t a[2] = {0u, 0u};
    for (int k = 0; k < 2; ++k) {
        const uint32_t u = 2 * tid + k;
        if (u >= n_band) continue;
        bool same = false;
        if (u > 0 && s_pos[u] >= 0 && s_pos[u - 1] >= 0 && s_ck[s_band[u]] == s_ck[s_band[u - 1]])
            same = same_key_row<D>(X, kbase, s_pos[u], s_pos[u - 1]);
        a[k] = same ? 0u : u;
    }
    const uint32_t pre = block_excl_max(max(a[0], a[1]), S.warp);
    const uint32_t h0 = max(pre, a[0]), h1 = max(h0, a[1]);
    uint32_t n_heads;
    const int nh = (2 * tid < n_band && h0 == 2 * tid) + (2 * tid + 1 < n_band && h1 == 2 * tid + 1);
    const uint32_t at = block_excl_count_sum((uint32_t)nh, S.warp, n_heads);
    {
        uint32_t o = at;
        if (2 * tid < n_band) {
            g_head[2 * tid] = h0;
            if (h0 == 2 * tid) s_act[o++] = 2 * tid;
        }
        if (2 * tid + 1 < n_band) {
            g_head[2 * tid + 1] = h1;
            if (h1 == 2 * tid + 1) s_act[o++] = 2 * tid + 1;
        }
    }
    __syncthreads();
    if (n_heads == 1) {
        // one run: every band candidate has the same exact score, so the lowest positions
        // (the band is in position order) are the ones taken
        for (uint32_t u = tid; u < n_band; u += kGThreads) s_state[u] = u < take ? 1 : 0;
        __syncthreads();
        return;
    }
    // fixed point for the run heads
    bool ok = true;
#pragma unroll 1
    for (uint32_t hi_ = warp; hi_ < n_heads; hi_ += kGThreads / 32) {
        const uint32_t u = s_act[hi_], i = s_band[u];
        const uint32_t ulo = X.unit > 1 ? score_key(rb.lo(key_value(s_ck[i]))) : 0u;
        __int128 V;
        int E;
        ok = unit_fixed<D>(Q, X, row, seq, pool_row, block, s_cp[i], ulo, V, E) && ok;
        if (lane < 4) g_v[(size_t)lane * kBandCap + u] = (uint32_t)(V >> (32 * lane));
        if (lane == 4) g_v[(size_t)4 * kBandCap + u] = (uint32_t)E;
    }
    ok = __syncthreads_and(ok) != 0;
    if (ok) {
        int e_row = exact::kNoTerms;
        for (uint32_t k = tid; k < n_heads; k += kGThreads) e_row = min(e_row, (int)g_v[(size_t)4 * kBandCap + s_act[k]]);
        e_row = __reduce_min_sync(0xffffffffu, e_row);
        if (lane == 0) s_red[warp] = (uint32_t)e_row;
        __syncthreads();
        e_row = exact::kNoTerms;
        for (int k = 0; k < kGThreads / 32; ++k) e_row = min(e_row, (int)s_red[k]);
        __syncthreads();
        for (uint32_t u = tid; u < n_band; u += kGThreads) {
            const uint32_t h = g_head[u];
            unsigned __int128 w = 0;
            for (int k = 3; k >= 0; --k) w = (w << 32) | g_v[(size_t)k * kBandCap + h];
            __int128 V = (__int128)w;
            ok = exact::align_fixed(V, (int)g_v[(size_t)4 * kBandCap + h], e_row) && ok;
            for (int k = 0; k < 4; ++k) {
                uint32_t word = (uint32_t)((unsigned __int128)V >> (32 * k));
                if (k == 3) word ^= 0x80000000u;
                bk[(size_t)k * kBandCap + u] = word;
            }
        }
        ok = __syncthreads_and(ok) != 0;
    }
    if (ok) {
        select_band(bk, 4, (int)n_band, take, s_state, s_act, s_val, S, s_red);
        return;
    }
    // wide form: every band candidate as 26 limbs
#pragma unroll 1
    for (uint32_t u = warp; u < n_band; u += kGThreads / 32) {
        const uint32_t i = s_band[u];
        const uint32_t ulo = X.unit > 1 ? score_key(rb.lo(key_value(s_ck[i]))) : 0u;
        const uint32_t limb = unit_key<D>(Q, X, row, seq, pool_row, block, s_cp[i], ulo);
        if (lane < exact::kLimbs) bk[(size_t)lane * kBandCap + u] = limb;
    }
    __syncthreads();
    select_band(bk, exact::kLimbs, (int)n_band, take, s_state, s_act, s_val, S, s_red);
}

// Candidate lists (csa2_index_topk): the scoring kernel's CTAs of a row each wrote a list
// of (key, position) in position order, with the list's K-th key (0 when it holds K or
// fewer: then it holds them all) and whether it met a non-finite score.  Each list holds
// every entry at or above lo(its K-th key), so the row's exact top K and its band are in
// their union; the row's K-th score is at least the largest list K-th key.
struct TopkLists {
    int n_lists;                   // lists per row (in position order)
    int64_t cap;                   // entries per list
    const uint32_t *key;           // [rows, n_lists, cap]
    const int32_t *pos;            // [rows, n_lists, cap]
    const uint32_t *meta;          // [rows, n_lists, 4]: count, K-th key, non-finite, 0
};
constexpr int kMaxLists = 1024;

template <bool EXACT, int D, bool LISTS, bool SHORT>
__global__ void __launch_bounds__(kGThreads, 1)
topk_gmax_kernel(const float *__restrict__ scores, int64_t n, int64_t rows, const int32_t *__restrict__ row_len,
                 const int32_t *__restrict__ pool, int32_t block, int32_t k, int32_t *__restrict__ idx,
                 float *__restrict__ out_scores, const uint32_t *__restrict__ gkeys, int32_t gs, int64_t G,
                 const ExactArgs X, const TopkLists Ls)
{
    // shared memory: the candidate-group list (later the exact band), then the group keys,
    // whose space the candidates' keys and positions take once the list is made
    extern __shared__ uint32_t g_sm[];
    uint32_t *s_g = g_sm;                                  // candidate-group list / exact band
    uint32_t *s_gk = g_sm + kListCap;                      // group keys
    uint32_t *s_ck = g_sm + kListCap;                      // candidate keys
    int32_t *s_cp = reinterpret_cast<int32_t *>(s_ck + kCandCap);   // candidate positions (index)
    static_assert(2 * kCandCap >= kMaxGroups, "group keys and candidates share their space");
    static_assert(16 * kGThreads <= kCandCap && 2 * kGThreads <= 2 * kCandCap, "short rows fit on chip");
    __shared__ GSmem S;
    __shared__ uint32_t s_red[64];
    __shared__ exact::QuantQuery QQ;                       // exact order: the row's query
    __shared__ uint32_t s_lpre[LISTS ? kMaxLists + 1 : 1];   // lists: offsets of the row's lists
    __shared__ uint32_t s_tmax;                           // lists: the largest list K-th key
    const int tid = threadIdx.x;
    // exact order: the first row's query and error bound come from inputs the kernel before
    // does not write (csa2_topk), so they are prepared before the dependency wait
    RowBound rb_first{0.0f, -1.0f};
    if constexpr (EXACT) {
        if ((int64_t)blockIdx.x < rows) {
            const int64_t r = blockIdx.x;
            exact::quantise_query(QQ, X.q + r * (int64_t)X.H * D, X.w + r * (int64_t)X.H, X.H, D);
            rb_first = row_bound(QQ, X, r / X.n_q, s_red);
        }
    }
    pdl_wait();                                            // scores / lists come from the kernel before
    pdl_allow_dependents();
#pragma unroll 1
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
    __syncthreads();                                       // the previous row is done with shared memory
    int64_t len = row_len ? (int64_t)row_len[row] : n;
    len = len < 0 ? 0 : (len > n ? n : len);
    const float *s = scores + row * n;
    const int32_t *pool_row = pool ? pool + row * (n / block) : nullptr;
    int32_t *out = idx + row * (int64_t)k;
    float *out_s = out_scores ? out_scores + row * (int64_t)k : nullptr;

    if (!LISTS && len <= k) {                              // everything competes and wins
        for (int64_t i = tid; i < k; i += kGThreads) {
            out[i] = i < len ? (int32_t)cand_pos(pool_row, block, i) : -1;
            if (out_s) out_s[i] = i < len ? s[i] : 0.0f;
        }
        continue;
    }
    uint32_t n_c = 0;
    bool overflow = false;
    RowBound rb{0.0f, -1.0f};
    int64_t seq = 0;
    bool nonfinite = false;
    if constexpr (LISTS) {
        // ---- the row's lists: counts, the largest list K-th key, non-finite flags
        const uint32_t *meta = Ls.meta + row * Ls.n_lists * 4;
        uint32_t cnt = 0, tk = 0;
        if (tid < Ls.n_lists) {
            cnt = meta[tid * 4];
            tk = meta[tid * 4 + 1];
            nonfinite = meta[tid * 4 + 2] != 0u;
        }
        if (tid == 0) s_tmax = 0u;
        nonfinite = __syncthreads_or(nonfinite) != 0;
        if (tid < Ls.n_lists && tk) atomicMax(&s_tmax, tk);
        uint32_t total;
        const uint32_t pre = block_excl_count_sum(cnt, S.warp, total);
        if (tid < Ls.n_lists) s_lpre[tid] = pre;
        if (tid == 0) s_lpre[Ls.n_lists] = total;
        __syncthreads();
        if constexpr (EXACT) {
            seq = row / X.n_q;
            if (row == (int64_t)blockIdx.x) {
                rb = rb_first;
            } else {
                exact::quantise_query(QQ, X.q + row * (int64_t)X.H * D, X.w + row * (int64_t)X.H, X.H, D);
                rb = row_bound(QQ, X, seq, s_red);
            }
            if (nonfinite) rb.c0 = -1.0f;
        }
        const bool ex_row = EXACT && rb.c0 >= 0.0f;
        const uint32_t *lk = Ls.key + row * Ls.n_lists * Ls.cap;
        const int32_t *lp = Ls.pos + row * Ls.n_lists * Ls.cap;
        const int nls = Ls.n_lists;
        const int64_t cap = Ls.cap;
        const uint32_t *lpre = s_lpre;
        // entry i of the row's lists, in list order (= position order)
        auto list_at = [lpre, nls, cap](uint32_t i) -> int64_t {
            int lo = 0, hi = nls;                           // the list c with lpre[c] <= i < lpre[c+1]
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (lpre[mid] <= i) lo = mid; else hi = mid;
            }
            return (int64_t)lo * cap + (i - lpre[lo]);
        };
        // entries at or above lo_key into shared memory, in list order; false: they do not
        // fit.  Thread t reads entries 4t .. 4t + 3 of each round of 4,096.
        auto load_lists = [&](uint32_t lo_key) -> bool {
            n_c = 0;
#pragma unroll 1
            for (uint32_t base = 0; base < total; base += 4 * kGThreads) {
                const uint32_t i0 = base + 4u * tid;
                uint32_t key[4];
                int32_t cd[4];
                uint32_t keep = 0;
                if (i0 < total) {
                    int64_t at = list_at(i0);
                    int c = (int)(at / cap);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint32_t i = i0 + u;
                        key[u] = 0u;
                        cd[u] = 0;
                        if (i < total) {
                            while (i >= lpre[c + 1]) ++c;      // the next non-empty list
                            at = (int64_t)c * cap + (i - lpre[c]);
                            key[u] = lk[at];
                            cd[u] = lp[at];
                            keep |= (uint32_t)(key[u] >= lo_key) << u;
                        }
                    }
                }
                uint32_t tot;
                uint32_t o = n_c + block_excl_count_sum((uint32_t)__popc(keep), S.warp, tot);
                if (n_c + tot > (uint32_t)kCandCap) return false;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if ((keep >> u) & 1u) {
                        s_ck[o] = key[u];
                        s_cp[o] = cd[u];
                        ++o;
                    }
                }
                n_c += tot;
            }
            return true;
        };
        // The row's K-th score is at least s_tmax, so the entries at or above lo(s_tmax) hold
        // the row's candidates and band.  When those do not fit on chip (a list's own K-th
        // key was a weak bound), the row's K-th float key is found over the lists where they
        // are and the load repeated at lo() of it; if even that does not fit (more than
        // kCandCap candidates tie with it), the row is selected in float order from the
        // lists directly and CSA2_DEV_BAND_LIMIT is set.
        const uint32_t tfl = s_tmax;
        uint32_t lo_t = tfl == 0u ? 0u : (ex_row ? score_key(rb.lo(key_value(tfl))) : tfl);
        if (!load_lists(lo_t)) {
            uint32_t need_g;
            const uint32_t tau_g = g_threshold_at([&](int i) { return lk[list_at((uint32_t)i)]; }, (int)total,
                                                  (uint32_t)k, S, need_g, 3);
            lo_t = ex_row ? score_key(rb.lo(key_value(tau_g))) : tau_g;
            if (!load_lists(lo_t)) {
                // float order straight from the lists: above tau_g, then the first need_g at it
                uint32_t n_gt = 0, n_eq = 0;
#pragma unroll 1
                for (uint32_t base = 0; base < total; base += kGThreads) {
                    const uint32_t i = base + tid;
                    uint32_t key = 0u;
                    int32_t ps = 0;
                    if (i < total) {
                        const int64_t at = list_at(i);
                        key = lk[at];
                        ps = lp[at];
                    }
                    uint32_t tg, te;
                    const uint32_t og = block_excl_count(i < total && key > tau_g, S.warp, tg);
                    const uint32_t oe = block_excl_count(i < total && key == tau_g, S.warp, te);
                    bool sel = i < total && key > tau_g;
                    if (i < total && key == tau_g) sel = n_eq + oe < need_g;
                    if (sel) {
                        const uint32_t o = n_gt + og + min(n_eq + oe, need_g);
                        if (o < (uint32_t)k) {
                            out[o] = (int32_t)cand_pos(pool_row, block, ps);
                            if (out_s) out_s[o] = key_value(key);
                        }
                    }
                    n_gt += tg;
                    n_eq += te;
                }
                if (tid == 0) dev_flag(X.d_status, CSA2_DEV_BAND_LIMIT);
                continue;
            }
        }
        __syncthreads();
        if (n_c <= (uint32_t)k) {                          // everything listed wins
            for (uint32_t i = tid; i < (uint32_t)k; i += kGThreads) {
                out[i] = i < n_c ? (int32_t)cand_pos(pool_row, block, s_cp[i]) : -1;
                if (out_s) out_s[i] = i < n_c ? key_value(s_ck[i]) : 0.0f;
            }
            continue;
        }
    } else if constexpr (SHORT) {
        // ---- short rows (a Reindex pool, a short context): thread t holds the keys of
        //      candidates [16 t, 16 t + 16) in registers.  Each of the k blocks of 8 with the
        //      largest maxima holds an element >= the k-th largest block maximum, so a lower
        //      bound of that maximum keeps every top-k element; only the elements at or above
        //      it are listed.  (Groups of 32 cannot prune a row of 16,384 at k = 512.)
        const int64_t b0 = 16 * (int64_t)tid;
        uint32_t kv[16];
        if (b0 >= len) {
    #pragma unroll
            for (int i = 0; i < 16; ++i) kv[i] = 0u;
        } else if (b0 + 16 <= n && (reinterpret_cast<uintptr_t>(s) & 15u) == 0) {
            const float4 *src = reinterpret_cast<const float4 *>(s + b0);
            float4 f[4];
    #pragma unroll
            for (int e = 0; e < 4; ++e) f[e] = src[e];
    #pragma unroll
            for (int e = 0; e < 4; ++e) {
                kv[4 * e] = score_key(f[e].x);
                kv[4 * e + 1] = score_key(f[e].y);
                kv[4 * e + 2] = score_key(f[e].z);
                kv[4 * e + 3] = score_key(f[e].w);
            }
        } else {
    #pragma unroll
            for (int i = 0; i < 16; ++i) kv[i] = b0 + i < len ? score_key(s[b0 + i]) : 0u;
        }
    #pragma unroll
        for (int i = 0; i < 16; ++i)
            if (b0 + i >= len) kv[i] = 0u;
        uint32_t bm0 = 0, bm1 = 0;                             // maxima of the thread's two blocks
    #pragma unroll
        for (int i = 0; i < 8; ++i) {
            bm0 = max(bm0, kv[i]);
            bm1 = max(bm1, kv[8 + i]);
        }
        s_gk[2 * tid] = bm0;
        s_gk[2 * tid + 1] = bm1;
        // a group of 32 (two threads) whose maximum is not finite: as in the grouped path
        uint32_t g32 = max(bm0, bm1);
        g32 = max(g32, __shfl_xor_sync(0xffffffffu, g32, 1));
        nonfinite = (tid & 1) == 0 && b0 < len && (g32 >= 0xff800000u || g32 <= 0x007fffffu);
        nonfinite = __syncthreads_or(nonfinite) != 0;
        if constexpr (EXACT) {
            seq = row / X.n_q;
            if (row == (int64_t)blockIdx.x) {
                rb = rb_first;
            } else {
                exact::quantise_query(QQ, X.q + row * (int64_t)X.H * D, X.w + row * (int64_t)X.H, X.H, D);
                rb = row_bound(QQ, X, seq, s_red);
            }
            if (nonfinite) rb.c0 = -1.0f;
        }
        const bool ex_row = EXACT && rb.c0 >= 0.0f;
        const int nb = (int)((len + 7) / 8);
        uint32_t need0;
        uint32_t tau0 = nb > k ? g_threshold(s_gk, nb, (uint32_t)k, S, need0, 2) : 0u;
        if (ex_row && tau0 != 0u) tau0 = score_key(rb.lo(key_value(tau0)));
        uint32_t sel = 0;
    #pragma unroll
        for (int i = 0; i < 16; ++i) sel |= (uint32_t)(b0 + i < len && kv[i] >= tau0) << i;
        uint32_t tot;
        uint32_t o = block_excl_count_sum((uint32_t)__popc(sel), S.warp, tot);   // block maxima read
    #pragma unroll
        for (int i = 0; i < 16; ++i) {
            if ((sel >> i) & 1u) {
                s_ck[o] = kv[i];
                s_cp[o] = (int32_t)(b0 + i);
                ++o;
            }
        }
        n_c = tot;                                         // <= 16 kGThreads = kCandCap
        __syncthreads();
    } else {
        const int ng = (int)((len + gs - 1) / gs);             // <= kMaxGroups
        const uint32_t *gk = s_gk;
        for (int g = tid; g < ng; g += kGThreads) {
            const uint32_t v = gkeys[row * G + g];
            s_gk[g] = v;
            nonfinite |= v >= 0xff800000u || v <= 0x007fffffu;
        }
        nonfinite = __syncthreads_or(nonfinite) != 0;
        // exact order: the row's error bound of the float32 scores (c0 < 0: none made)
        if constexpr (EXACT) {
            seq = row / X.n_q;
            if (row == (int64_t)blockIdx.x) {
                rb = rb_first;
            } else {
                exact::quantise_query(QQ, X.q + row * (int64_t)X.H * D, X.w + row * (int64_t)X.H, X.H, D);
                rb = row_bound(QQ, X, seq, s_red);
            }
            if (nonfinite) rb.c0 = -1.0f;
        }
        const bool ex_row = EXACT && rb.c0 >= 0.0f;
        // a lower bound of the k-th largest group key is enough to keep every top-k element
        // (the groups above the bound are a superset of those above the exact key); in exact
        // order the bound is lowered to lo() of it, so the whole band is gathered
        uint32_t need0;
        uint32_t tau0 = ng > k ? g_threshold(gk, ng, (uint32_t)k, S, need0, 2) : 0u;
        if (ex_row && tau0 != 0u) tau0 = score_key(rb.lo(key_value(tau0)));

        // candidate groups (key >= tau0), listed in s_g in ascending order: thread t owns the
        // run [t*run, (t+1)*run)
        const int run = (ng + kGThreads - 1) / kGThreads;        // <= 32
        const int r0 = min(tid * run, ng), r1 = min(r0 + run, ng);
        uint32_t mine = 0;                                      // bit j: group r0+j is a candidate
        for (int i = r0; i < r1; ++i) mine |= (gk[i] >= tau0 ? 1u : 0u) << (i - r0);
        uint32_t n_cg;
        const uint32_t at = block_excl_count_sum((uint32_t)__popc(mine), S.warp, n_cg);
        if (n_cg > (uint32_t)kListCap) {                        // too many to list on chip
            radix_select_row(scores, n, row_len, pool, block, k, idx, out_scores, row);
            if (EXACT && tid == 0) dev_flag(X.d_status, CSA2_DEV_BAND_LIMIT);
            continue;
        }
        {
            uint32_t o = at;
            for (int i = r0; i < r1; ++i)
                if ((mine >> (i - r0)) & 1u) s_g[o++] = (uint32_t)i;
        }
        __syncthreads();
        // gather candidates, in position order: one thread per candidate group reads its
        // scores (groups of 32 as eight 16-byte loads, all in flight at once) and keeps a bit
        // mask of its elements >= tau0; after a scan of the counts it walks the mask in a
        // rolled loop, reading each selected score again (the lines are in L1 by then).  This
        // code runs once per row, so it is kept small.
        const bool vec = gs == 32 && ((reinterpret_cast<uintptr_t>(s) & 15u) == 0);   // 16-byte rows
    #pragma unroll 1
        for (uint32_t base = 0; base < n_cg; base += kGThreads) {
            const uint32_t j = base + tid;
            uint32_t sel = 0;                                  // groups of 32: bit e = element e
            uint32_t cnt = 0;
            int64_t g0 = 0;
            if (j < n_cg) {
                g0 = (int64_t)s_g[j] * gs;
                if (vec && g0 + 32 <= n) {
                    float4 f[8];
                    const float4 *src = reinterpret_cast<const float4 *>(s + g0);
    #pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = src[e];
    #pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        sel |= (uint32_t)(score_key(f[e].x) >= tau0) << (4 * e);
                        sel |= (uint32_t)(score_key(f[e].y) >= tau0) << (4 * e + 1);
                        sel |= (uint32_t)(score_key(f[e].z) >= tau0) << (4 * e + 2);
                        sel |= (uint32_t)(score_key(f[e].w) >= tau0) << (4 * e + 3);
                    }
                    if (g0 + 32 > len) sel &= len > g0 ? (1u << (len - g0)) - 1u : 0u;
                    cnt = __popc(sel);
                } else {
    #pragma unroll 1
                    for (int e = 0; e < gs && g0 + e < len; ++e) cnt += score_key(s[g0 + e]) >= tau0;
                }
            }
            uint32_t tot;
            uint32_t o = n_c + block_excl_count_sum(cnt, S.warp, tot);
            if (n_c + tot > kCandCap) {                        // does not fit on chip: fall back
                overflow = true;
                break;
            }
            if (j < n_cg) {
                if (vec && g0 + 32 <= n) {
    #pragma unroll 1
                    while (sel) {
                        const int e = __ffs(sel) - 1;
                        sel &= sel - 1u;
                        s_ck[o] = score_key(s[g0 + e]);
                        s_cp[o] = (int32_t)(g0 + e);
                        ++o;
                    }
                } else {
    #pragma unroll 1
                    for (int e = 0; e < gs && g0 + e < len; ++e) {
                        const uint32_t key = score_key(s[g0 + e]);
                        if (key >= tau0) { s_ck[o] = key; s_cp[o] = (int32_t)(g0 + e); ++o; }
                    }
                }
            }
            n_c += tot;
        }
        __syncthreads();
        if (overflow) {                                        // does not fit on chip: fall back
            radix_select_row(scores, n, row_len, pool, block, k, idx, out_scores, row);
            if (EXACT && tid == 0) dev_flag(X.d_status, CSA2_DEV_BAND_LIMIT);
            continue;
        }
    }
    const bool exact_row = EXACT && rb.c0 >= 0.0f;
    // selection among the candidates (n_c >= k) in float order: the k-th key tau and how
    // many candidates equal to it are taken
    uint32_t need;
    uint32_t tau = g_threshold(s_ck, (int)n_c, (uint32_t)k, S, need, 3);
    const int crun = ((int)n_c + kGThreads - 1) / kGThreads;
    const int c0 = min(tid * crun, (int)n_c), c1 = min(c0 + crun, (int)n_c);
    uint32_t band_n = 0;                                   // lists: band entries re-scored exactly
    if constexpr (EXACT) {
        if (exact_row && tau != 0u) {
            // the band [lo(tau~), hi(tau~)] in key terms; above it: selected
            const float tv = key_value(tau);
            const uint32_t lo_key = score_key(rb.lo(tv));
            const uint32_t hi_key = score_key(rb.hi(tv));
            uint32_t n_hi = 0, n_bd = 0;
            for (int i = c0; i < c1; ++i) {
                n_hi += s_ck[i] > hi_key;
                n_bd += s_ck[i] >= lo_key && s_ck[i] <= hi_key;
            }
            uint32_t tot;
            const uint32_t before = block_excl_count_sum((n_hi << 16) | n_bd, S.warp, tot);
            const uint32_t n_in = tot >> 16, n_band = tot & 0xffffu;
            const uint32_t take = (uint32_t)k > n_in ? (uint32_t)k - n_in : 0u;
            uint32_t *s_band = s_g;                        // band candidates, in position order
            uint32_t *s_act = s_g + kBandCap;
            uint32_t *s_val = s_g + 2 * kBandCap;
            uint8_t *s_state = reinterpret_cast<uint8_t *>(s_g + 3 * kBandCap);
            if (n_band <= (uint32_t)kBandCap) {
                uint32_t o = before & 0xffffu;
                for (int i = c0; i < c1; ++i)
                    if (s_ck[i] >= lo_key && s_ck[i] <= hi_key) s_band[o++] = (uint32_t)i;
            }
            __syncthreads();
            if (n_band < take) {
                // cannot happen (every candidate >= tau~ is above or in the band): float order
            } else if (n_band > take && n_band > (uint32_t)kBandCap) {
                if (tid == 0) dev_flag(X.d_status, CSA2_DEV_BAND_LIMIT);    // float order stays
            } else {
                if (n_band > take) {
                    band_exact<D>(QQ, X, rb, row, seq, pool_row, block, s_band, s_ck, s_cp, n_band, take, s_state,
                                  s_act, s_val, S, s_red);
                    // band candidates taken rank above hi, the others below every
                    // candidate: the float-order emission below then takes exactly these
                    // (lists: the band's own keys are kept by band index for the scores out)
                    for (uint32_t u = tid; u < n_band; u += kGThreads) {
                        if (LISTS) s_act[u] = s_ck[s_band[u]];
                        s_ck[s_band[u]] = s_state[u] ? 0xffffffffu : 0u;
                    }
                    __syncthreads();
                    tau = hi_key;
                    need = 0;
                    band_n = n_band;
                } else {
                    // the whole band is taken: every candidate >= lo is selected
                    tau = lo_key;
                    need = 0xffffffffu;
                }
            }
        }
    }
    uint32_t n_gt = 0, n_eq = 0;
    for (int i = c0; i < c1; ++i) {
        n_gt += s_ck[i] > tau;
        n_eq += s_ck[i] == tau;
    }
    // one scan of (above, equal) counts packed in 16-bit halves (n_c <= kCandCap < 2^16):
    // the candidates equal to tau taken are the first `need` in position order
    uint32_t t_both;
    const uint32_t before = block_excl_count_sum((n_gt << 16) | n_eq, S.warp, t_both);
    const uint32_t eq_before = before & 0xffffu;
    uint32_t o = (before >> 16) + min(eq_before, need);
    uint32_t ties = eq_before;
    for (int i = c0; i < c1; ++i) {
        const uint32_t key = s_ck[i];
        bool sel = key > tau;
        if (key == tau) sel = ties++ < need;
        if (sel && o < (uint32_t)k) {
            out[o] = (int32_t)cand_pos(pool_row, block, s_cp[i]);
            if (out_s) {
                if constexpr (LISTS) {
                    uint32_t kk = key;
                    if (key == 0xffffffffu) {          // a band candidate taken: its own key
                        uint32_t lo = 0, hi = band_n;
                        while (lo < hi) {
                            const uint32_t mid = (lo + hi) >> 1;
                            if (s_g[mid] < (uint32_t)i) lo = mid + 1; else hi = mid;
                        }
                        kk = s_g[kBandCap + lo];               // s_act (band index order)
                    }
                    out_s[o] = key_value(kk);
                } else {
                    out_s[o] = s[s_cp[i]];
                }
            }
            ++o;
        }
    }
    }   // rows
}

int32_t group_size_for(int64_t n)
{
    int32_t gs = 32;
    while ((n + gs - 1) / gs > kMaxGroups && gs < (1 << 20)) gs *= 2;
    return gs;
}

// Block score = max over the block's valid positions (NaN ignored; all-NaN -> NaN).
__global__ void block_max_kernel(const float *__restrict__ scores, int64_t n,
                                 const int32_t *__restrict__ row_len, int32_t block, int64_t nbmax,
                                 float *__restrict__ bscores, int32_t *__restrict__ brow_len)
{
    const int64_t row = blockIdx.y;
    int64_t len = row_len ? (int64_t)row_len[row] : n;
    len = len < 0 ? 0 : (len > n ? n : len);
    const int64_t nblk = (len + block - 1) / block;
    if (blockIdx.x == 0 && threadIdx.x == 0) brow_len[row] = (int32_t)nblk;
    const float *s = scores + row * n;
    for (int64_t bi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; bi < nblk;
         bi += (int64_t)gridDim.x * blockDim.x) {
        float m = __uint_as_float(0x7fc00000u);
        const int64_t p0 = bi * block;
        for (int j = 0; j < block && p0 + j < len; ++j) m = fmaxf(m, s[p0 + j]);
        bscores[row * nbmax + bi] = m;
    }
}

} // namespace

namespace {

constexpr int64_t kExactSlots = 160;      // per-CTA band slots of the exact pass

size_t align256(size_t a) { return (a + 255) & ~(size_t)255; }

int64_t exact_slots(int64_t rows) { return rows < kExactSlots ? rows : kExactSlots; }

size_t group_keys_bytes(int64_t rows, int64_t n)
{
    const int64_t G = (n + group_size_for(n) - 1) / group_size_for(n);
    return (size_t)rows * (size_t)(G > 0 ? G : 1) * sizeof(uint32_t);
}

// The selection kernel for float order, or exact order at the indexer head dim.
template <bool EXACT, int D, bool LISTS = false, bool SHORT = false>
cudaError_t launch_gmax(unsigned grid, size_t smem, cudaStream_t s, const float *scores, int64_t n, int64_t rows,
                        const int32_t *row_len, const int32_t *pool, int32_t block, int32_t k, int32_t *idx,
                        float *out_scores, const uint32_t *gkeys, int32_t gs, int64_t G, const ExactArgs &X,
                        const TopkLists &L = TopkLists{})
{
    cudaError_t e = cudaFuncSetAttribute(topk_gmax_kernel<EXACT, D, LISTS, SHORT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(topk_gmax_kernel<EXACT, D, LISTS, SHORT>, dim3(grid), dim3(kGThreads), smem, s, 1, scores, n, rows,
                      row_len, pool, block, k, idx, out_scores, gkeys, gs, G, X, L);
}

} // namespace

size_t topk_ws_bytes(int64_t rows, int64_t n, int32_t, bool exact)
{
    size_t a = group_keys_bytes(rows, n);
    if (exact) a = align256(a) + (size_t)exact_slots(rows) * exact::kLimbs * kBandCap * sizeof(uint32_t);
    return a;
}

cudaError_t launch_topk(const float *scores, int64_t rows, int64_t n, const int32_t *row_len,
                        const uint32_t *group_max, const int32_t *pool, int32_t block, int32_t k,
                        int32_t *idx, float *out_scores, void *ws, uint32_t *d_status, cudaStream_t s,
                        const csa2_index_args *ex, int32_t unit, const float *pos_scores, int64_t pos_n,
                        const int32_t *pos_len)
{
    if (rows == 0 || k == 0) return cudaSuccess;
    if (!ex && (rows > 0x7fffffffLL || !ws)) {
        topk_radix_kernel<<<(unsigned)rows, kTopkThreads, 0, s>>>(scores, n, row_len, pool, block, k,
                                                                 idx, out_scores);
        return cudaGetLastError();
    }
    const int32_t gs = group_size_for(n);
    const int64_t G = (n + gs - 1) / gs;
    const uint32_t *gkeys = static_cast<const uint32_t *>(ws);
    // rows of at most 16 candidates a thread: the short-row instance (its bound comes from
    // maxima of blocks of 8 it takes itself, no group keys)
    const bool short_rows = n <= 16 * kGThreads;
    if (short_rows || (group_max && gs == 32)) {
        if (!short_rows) gkeys = group_max;                // written by the indexer
    } else if (G > 0) {
        uint32_t *gk = static_cast<uint32_t *>(ws);
        if (gs == 32 && ((uintptr_t)scores % 16) == 0 && n % 4 == 0) {
            const int64_t blocks = (rows * G + 255) / 256;
            group_max32_kernel<<<(unsigned)blocks, 256, 0, s>>>(scores, n, row_len, rows, G, gk);
        } else {
            int64_t blocks = (rows * G * 32 + 255) / 256;
            const int64_t cap = (int64_t)device_sm_count() * 16;
            if (blocks > cap) blocks = cap;
            group_max_kernel<<<(unsigned)blocks, 256, 0, s>>>(scores, n, row_len, rows, gs, G, gk);
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const size_t smem = (size_t)(kListCap + 2 * kCandCap) * sizeof(uint32_t);
    ExactArgs X = {};
    if (!ex)
        return short_rows ? launch_gmax<false, 0, false, true>((unsigned)rows, smem, s, scores, n, rows, row_len, pool,
                                                               block, k, idx, out_scores, gkeys, gs, G, X)
                          : launch_gmax<false, 0>((unsigned)rows, smem, s, scores, n, rows, row_len, pool, block, k,
                                                  idx, out_scores, gkeys, gs, G, X);
    // exact order: persistent CTAs (at most one per SM and per band slot), rows strided
    X.H = ex->n_heads;
    X.d = ex->head_dim;
    X.n_q = ex->n_q;
    X.n_keys = ex->n_keys;
    X.q = ex->q;
    X.w = ex->w;
    X.kc = ex->k_codes;
    X.ks = ex->k_scales;
    X.unit = unit;
    X.pos_scores = pos_scores;
    X.pos_n = pos_n;
    X.pos_len = pos_len;
    X.band = reinterpret_cast<uint32_t *>(static_cast<char *>(ws) + align256(group_keys_bytes(rows, n)));
    X.d_status = d_status;
    int64_t grid = exact_slots(rows);
    if (grid > device_sm_count()) grid = device_sm_count();
#define CSA2_TOPK_CASE(DIM)                                                                                  \
    case DIM:                                                                                                \
        return short_rows ? launch_gmax<true, DIM, false, true>((unsigned)grid, smem, s, scores, n, rows, row_len, \
                                                                pool, block, k, idx, out_scores, gkeys, gs, G, X)    \
                          : launch_gmax<true, DIM>((unsigned)grid, smem, s, scores, n, rows, row_len, pool, block,  \
                                                   k, idx, out_scores, gkeys, gs, G, X);
    switch (ex->head_dim) {
    CSA2_TOPK_CASE(32)
    CSA2_TOPK_CASE(64)
    CSA2_TOPK_CASE(128)
#undef CSA2_TOPK_CASE
    default: return cudaErrorInvalidValue;
    }
}

size_t topk_lists_ws_bytes(int64_t rows)
{
    return (size_t)exact_slots(rows) * exact::kLimbs * kBandCap * sizeof(uint32_t);
}

cudaError_t launch_topk_lists(const csa2_index_args &ex, int32_t k, const uint32_t *key, const int32_t *pos,
                              const uint32_t *meta, int n_lists, int64_t cap, int32_t *idx, float *out_scores,
                              void *ws, uint32_t *d_status, cudaStream_t s)
{
    const int64_t rows = (int64_t)ex.batch * ex.n_q;
    if (rows == 0 || k == 0) return cudaSuccess;
    if (n_lists < 1 || n_lists > kMaxLists) return cudaErrorInvalidValue;
    TopkLists L;
    L.n_lists = n_lists;
    L.cap = cap;
    L.key = key;
    L.pos = pos;
    L.meta = meta;
    ExactArgs X = {};
    X.H = ex.n_heads;
    X.d = ex.head_dim;
    X.n_q = ex.n_q;
    X.n_keys = ex.n_keys;
    X.q = ex.q;
    X.w = ex.w;
    X.kc = ex.k_codes;
    X.ks = ex.k_scales;
    X.unit = 1;
    X.band = static_cast<uint32_t *>(ws);
    X.d_status = d_status;
    int64_t grid = exact_slots(rows);
    if (grid > device_sm_count()) grid = device_sm_count();
    const size_t smem = (size_t)(kListCap + 2 * kCandCap) * sizeof(uint32_t);
    const int64_t n = ex.n_keys;
    switch (ex.head_dim) {
    case 32: return launch_gmax<true, 32, true>((unsigned)grid, smem, s, nullptr, n, rows, nullptr, nullptr, 1, k,
                                                idx, out_scores, nullptr, 32, 0, X, L);
    case 64: return launch_gmax<true, 64, true>((unsigned)grid, smem, s, nullptr, n, rows, nullptr, nullptr, 1, k,
                                                idx, out_scores, nullptr, 32, 0, X, L);
    case 128: return launch_gmax<true, 128, true>((unsigned)grid, smem, s, nullptr, n, rows, nullptr, nullptr, 1,
                                                  k, idx, out_scores, nullptr, 32, 0, X, L);
    default: return cudaErrorInvalidValue;
    }
}

size_t block_candidates_ws_bytes(int64_t rows, int64_t n, int32_t block, int32_t nb, bool exact)
{
    const int64_t nbmax = (n + block - 1) / block;
    size_t a = align256((size_t)rows * (size_t)nbmax * sizeof(float));
    a = align256(a + (size_t)rows * sizeof(int32_t));
    return a + topk_ws_bytes(rows, nbmax, nb, exact);
}

cudaError_t launch_block_candidates(const float *scores, int64_t rows, int64_t n,
                                    const int32_t *row_len, int32_t block, int32_t nb,
                                    int32_t *block_ids, void *ws, uint32_t *d_status,
                                    cudaStream_t s, const csa2_index_args *ex)
{
    if (rows == 0 || nb == 0) return cudaSuccess;
    const int64_t nbmax = (n + block - 1) / block;
    float *bscores = static_cast<float *>(ws);
    const size_t off = align256((size_t)rows * (size_t)nbmax * sizeof(float));
    int32_t *brow_len = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + off);
    int64_t gx = (nbmax + 255) / 256;
    if (gx > 64) gx = 64;
    if (gx < 1) gx = 1;
    block_max_kernel<<<dim3((unsigned)gx, (unsigned)rows), 256, 0, s>>>(scores, n, row_len, block,
                                                                        nbmax, bscores, brow_len);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t off2 = align256(off + (size_t)rows * sizeof(int32_t));
    return launch_topk(bscores, rows, nbmax, brow_len, nullptr, nullptr, 1, nb, block_ids, nullptr,
                       static_cast<char *>(ws) + off2, d_status, s, ex, block, scores, n, row_len);
}

} // namespace csa2
