// index_score.cu -- CSA2 indexer scoring (csa2_index_score).
//
// DeepSeek-V4.1-Flash report (aipaper.jasonlin.tech) §2.3: the lightweight indexer scores
// main-KV entries with indexer Q and indexer K (both MXFP4, §2.4.4) and the query keeps
// its Top-K; §2.3.2: the first Full layer scores every causally visible position, later
// Reindex layers score only the positions of the block pool.
//
// Score of position t: s_t = sum_h w_h * max(0, q_hat_h . k_hat_t), written out as its float32
// approximation D_h = RN32(q_hat_h . k_hat_t), s = fma32 chain of w_h * max(D_h, 0), within a
// proven bound of the exact value (csa2_topk ranks by the exact value, re-scoring the
// candidates the bound leaves undecided); a score that is not finite sets
// CSA2_DEV_SCORE_RANGE.
//
// This file holds the exact CUDA-core kernel: each thread owns one candidate position,
// expands its FP4 codes to int8 (twice the E2M1 value), takes exact per-block integer
// dots with dp4a against the query (quantised once per CTA into shared memory), and
// rounds each head's dyadic sum once to float32.
#include "common.cuh"
#include "internal.h"

namespace csa2 {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxHeads = 64;

struct IndexParams {
    int32_t n_q, H, ratio_m, block, n_pool_blocks;
    int64_t n_keys, n_cand, chunk;
    const uint16_t *q;
    const float *w;
    const uint8_t *kc, *ks;
    const int32_t *q_pos, *pool;
    bool pool_mode;
    float *scores;
    int32_t *row_len;
    uint32_t *gmax;              // optional [rows, G]: largest selection key of each 32-group
    int64_t G;
    uint32_t *d_status;
};

// Visible entries of a query at token position p: (j+1)*m - 1 <= p (report §2.3: an entry
// covers m tokens with no overlap; only complete entries are visible).
__device__ __forceinline__ int64_t visible_entries(const IndexParams &P, int64_t row)
{
    if (!P.q_pos) return P.n_keys;
    int64_t p = P.q_pos[row];
    int64_t v = (p + 1) / P.ratio_m;
    if (p + 1 < 0) v = 0;
    return v < 0 ? 0 : (v > P.n_keys ? P.n_keys : v);
}

// Exact score of one candidate: the key row's codes as int8x4 words of twice the E2M1
// values, per-block integer dots with dp4a against the quantised query, each head's
// dyadic sum rounded once to float32, then the fma chain over heads.
template <int D>
__device__ __forceinline__ float score_candidate(const IndexParams &P, const int32_t *pool, int64_t kbase,
                                                 int64_t cand, const int32_t *s_qw, const int32_t *s_qx,
                                                 const float *s_w, const uint16_t *s_lut)
{
    constexpr int NB = D / 32, NW = D / 4;
    int64_t pos = cand;
    if (P.pool_mode) {
        const int32_t id = pool[cand / P.block];
        pos = (int64_t)(id < 0 ? 0 : id) * P.block + cand % P.block;
        if (pos >= P.n_keys) pos = P.n_keys - 1;           // only for a flagged bad pool
    }
    int32_t kw[NW];
    const uint8_t *kc = P.kc + (kbase + pos) * (D / 2);
#pragma unroll
    for (int v = 0; v < D / 32; ++v) {
        const uint4 raw = *reinterpret_cast<const uint4 *>(kc + 16 * v);
        const uint32_t r4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            kw[v * 8 + 2 * j] = (int32_t)((uint32_t)s_lut[r4[j] & 0xff] |
                                          ((uint32_t)s_lut[(r4[j] >> 8) & 0xff] << 16));
            kw[v * 8 + 2 * j + 1] = (int32_t)((uint32_t)s_lut[(r4[j] >> 16) & 0xff] |
                                              ((uint32_t)s_lut[r4[j] >> 24] << 16));
        }
    }
    int kx[NB];
    const uint8_t *ks = P.ks + (kbase + pos) * NB;
#pragma unroll
    for (int k = 0; k < NB; ++k) kx[k] = (int)ks[k] - 127;

    float s = 0.0f;
    for (int h = 0; h < P.H; ++h) {
        int I[NB], E[NB];
#pragma unroll
        for (int k = 0; k < NB; ++k) {
            int acc = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) acc = __dp4a(s_qw[h * NW + k * 8 + j], kw[k * 8 + j], acc);
            I[k] = acc;
            E[k] = s_qx[h * NB + k] + kx[k] - 2;
        }
        const float Dh = dyadic_sum_f32<NB>(I, E);
        s = __fmaf_rn(s_w[h], Dh > 0.0f ? Dh : 0.0f, s);
    }
    return s;
}

template <int D>
__global__ void __launch_bounds__(kThreads) index_score_exact_kernel(IndexParams P)
{
    constexpr int NB = D / 32;   // 32-value blocks per head
    constexpr int NW = D / 4;    // int8x4 words per head
    __shared__ int32_t s_qw[kMaxHeads * NW];
    __shared__ int32_t s_qx[kMaxHeads * NB];
    __shared__ float s_w[kMaxHeads];
    __shared__ uint16_t s_lut[256];
    __shared__ int64_t s_len;
    __shared__ uint32_t s_bad;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t row = blockIdx.y;
    const int64_t b = row / P.n_q;
    const int H = P.H;
    for (int i = tid; i < 256; i += kThreads)
        s_lut[i] = (uint16_t)((e2m1_twice(i & 15u) & 0xff) | ((e2m1_twice(i >> 4) & 0xff) << 8));
    if (tid == 0) { s_len = 0; s_bad = 0; }
    for (int h = tid; h < H; h += kThreads) s_w[h] = P.w[row * H + h];

    // quantise this query's indexer heads to MXFP4, one warp per 32-value block
    const uint16_t *q = P.q + row * (int64_t)H * D;
    for (int blk = warp; blk < H * NB; blk += kThreads / 32) {
        const float v = __uint_as_float((uint32_t)q[blk * 32 + lane] << 16);
        const uint32_t amax_bits = __reduce_max_sync(0xffffffffu, __float_as_uint(v) & 0x7fffffffu);
        const int X = mx_block_exponent(__uint_as_float(amax_bits >= 0x7f800000u ? 0u : amax_bits));
        const uint32_t c = e2m1_encode(v, pow2_neg(X));
        const uint32_t t = (uint32_t)e2m1_twice(c) & 0xffu;
        uint32_t word = t;
        word |= __shfl_down_sync(0xffffffffu, t, 1) << 8;
        word |= __shfl_down_sync(0xffffffffu, t, 2) << 16;
        word |= __shfl_down_sync(0xffffffffu, t, 3) << 24;
        if ((lane & 3) == 0) s_qw[blk * 8 + (lane >> 2)] = (int32_t)word;
        if (lane == 0) s_qx[blk] = X;
        if (amax_bits >= 0x7f800000u && lane == 0) dev_flag(P.d_status, CSA2_DEV_NONFINITE);
    }
    __syncthreads();

    // valid candidates of this row
    const int64_t n_vis = visible_entries(P, row);
    const int32_t *pool = P.pool_mode ? P.pool + row * (int64_t)P.n_pool_blocks : nullptr;
    if (!P.pool_mode) {
        if (tid == 0) s_len = n_vis;
    } else {
        const int64_t n_blk_all = (P.n_keys + P.block - 1) / P.block;
        int64_t part = 0;
        uint32_t bad = 0;
        for (int i = tid; i < P.n_pool_blocks; i += kThreads) {
            const int32_t id = pool[i];
            const int32_t prev = i > 0 ? pool[i - 1] : -1;
            if (id >= 0) {
                if (id >= n_blk_all || (i > 0 && (prev < 0 || prev >= id))) bad = 1;
                int64_t c = n_vis - (int64_t)id * P.block;
                part += c <= 0 ? 0 : (c > P.block ? P.block : c);
            }
        }
        if (bad) atomicOr(&s_bad, 1u);
        atomicAdd((unsigned long long *)&s_len, (unsigned long long)part);
    }
    __syncthreads();
    const int64_t len = s_len;
    if (blockIdx.x == 0 && tid == 0) {
        if (P.row_len) P.row_len[row] = (int32_t)len;
        if (s_bad) dev_flag(P.d_status, CSA2_DEV_BAD_POOL);
    }

    const int64_t kbase = b * P.n_keys;
    {
        const int64_t c0 = (int64_t)blockIdx.x * P.chunk;
        const int64_t c1 = min(c0 + P.chunk, len);
        // uniform trip count: every warp meets the group reduction below; c0 is a multiple
        // of 32, so each warp's 32 candidates form one group
        for (int64_t base = c0; base < c1; base += kThreads) {
            const int64_t cand = base + tid;
            uint32_t gkey = 0;
            if (cand < c1) {
                const float s = score_candidate<D>(P, pool, kbase, cand, s_qw, s_qx, s_w, s_lut);
                P.scores[row * P.n_cand + cand] = s;
                gkey = score_key(s);
                if (!(fabsf(s) <= 3.4028234663852886e38f)) dev_flag(P.d_status, CSA2_DEV_SCORE_RANGE);
            }
            if (P.gmax) {
                const uint32_t gk = __reduce_max_sync(0xffffffffu, gkey);
                const int64_t g0 = base + (tid & ~31);
                if (lane == 0 && g0 < c1) P.gmax[row * P.G + (g0 >> 5)] = gk;
            }
        }
    }
}

} // namespace

// Exact CUDA-core scoring: one CTA per (segment of `chunk` candidates, query row).
cudaError_t launch_index_exact(const csa2_index_args &a, float *scores, int32_t *row_len,
                               uint32_t *d_status, cudaStream_t s)
{
    IndexParams P;
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
    P.d_status = d_status;
    const int64_t rows = (int64_t)a.batch * a.n_q;
    if (rows == 0) return cudaSuccess;
    int64_t chunk = 2048;          // so that the grid covers the GPU a few times over
    while (chunk > 256 && rows * ((P.n_cand + chunk - 1) / chunk) < (int64_t)device_sm_count() * 8) chunk /= 2;
    P.chunk = chunk;
    const int64_t gx = (P.n_cand + chunk - 1) / chunk;
    dim3 grid((unsigned)(gx > 0 ? gx : 1), (unsigned)rows);
    switch (a.head_dim) {
    case 32: index_score_exact_kernel<32><<<grid, kThreads, 0, s>>>(P); break;
    case 64: index_score_exact_kernel<64><<<grid, kThreads, 0, s>>>(P); break;
    case 128: index_score_exact_kernel<128><<<grid, kThreads, 0, s>>>(P); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

// Workspace of the tensor-core path: two counters per query row (tiles claimed, CTAs done),
// zero between calls: the row's last CTA clears them.
size_t index_score_ws_bytes(const csa2_index_args &a)
{
    if (!index_tc_eligible(a)) return 0;
    const size_t rows = (size_t)a.batch * a.n_q;
    return (2 * rows * sizeof(uint32_t) + 15) & ~(size_t)15;
}

cudaError_t launch_index_score(const csa2_index_args &a, float *scores, int32_t *row_len, void *ws,
                               uint32_t *d_status, cudaStream_t s)
{
    const int64_t rows = (int64_t)a.batch * a.n_q;
    if (rows == 0) return cudaSuccess;
    if (!index_tc_eligible(a) || !ws) return launch_index_exact(a, scores, row_len, d_status, s);
    return launch_index_tc(a, scores, row_len, static_cast<uint32_t *>(ws), d_status, s);
}

} // namespace csa2
