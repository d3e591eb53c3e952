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
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace csa2 {
namespace {

constexpr int kTopkThreads = 1024;

__device__ __forceinline__ int64_t cand_pos(const int32_t *pool_row, int32_t block, int64_t i)
{
    if (!pool_row) return i;
    return (int64_t)pool_row[i / block] * block + i % block;
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

__global__ void __launch_bounds__(kTopkThreads)
topk_radix_kernel(const float *__restrict__ scores, int64_t n, const int32_t *__restrict__ row_len,
                  const int32_t *__restrict__ pool, int32_t block, int32_t k,
                  int32_t *__restrict__ idx, float *__restrict__ out_scores)
{
    __shared__ uint32_t s_hist[256];
    __shared__ uint32_t s_warp[33];
    __shared__ uint32_t s_prefix, s_mask, s_remaining;

    const int tid = threadIdx.x, lane = tid & 31;
    const int64_t row = blockIdx.x;
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

// ------------------------------------------------------------------ cluster radix select
// One thread-block cluster per row.  CTA r of the cluster owns the contiguous slice r of
// the row (kept as keys in shared memory when it fits).  Three digit passes of 11, 11 and
// 10 bits: each CTA histograms its slice, the cluster sums the histograms through
// distributed shared memory, and every CTA derives the same digit.  The final pass emits
// the selected entries in position order: CTA r starts after everything earlier CTAs
// selected, and takes ties in order until the cluster-wide quota is used up.
constexpr int kClThreads = 512;
constexpr int kClBins = 2048;
constexpr int kClKeyCap = 24576;            // keys per CTA kept in shared memory (96 KB)

struct ClusterTopkArgs {
    const float *scores;
    int64_t n;
    const int32_t *row_len;
    const int32_t *pool;
    int32_t block, k;
    int32_t *idx;
    float *out_scores;
    int64_t key_cap;     // keys of a slice that fit the launch's dynamic shared memory
};

// Block-wide exclusive prefix sum of one value per thread (kClThreads threads).
__device__ __forceinline__ uint32_t cl_block_excl_sum(uint32_t v, uint32_t *s_warp, uint32_t &total)
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
        const uint32_t w = lane < kClThreads / 32 ? s_warp[lane] : 0u;
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

__global__ void __launch_bounds__(kClThreads) topk_cluster_kernel(const ClusterTopkArgs A)
{
    extern __shared__ uint32_t s_keys[];
    __shared__ __align__(16) uint32_t s_hist[kClBins];
    __shared__ uint32_t s_warp[33];
    __shared__ uint32_t s_cnt[2];
    __shared__ uint32_t s_pick[2];
    cg::cluster_group cl = cg::this_cluster();
    const int rank = (int)cl.block_rank(), CS = (int)cl.num_blocks();
    const int tid = threadIdx.x, lane = tid & 31;
    const int64_t row = blockIdx.y;
    int64_t len = A.row_len ? (int64_t)A.row_len[row] : A.n;
    len = len < 0 ? 0 : (len > A.n ? A.n : len);
    const float *s = A.scores + row * A.n;
    const int32_t *pool_row = A.pool ? A.pool + row * (A.n / A.block) : nullptr;
    int32_t *out = A.idx + row * (int64_t)A.k;
    float *out_s = A.out_scores ? A.out_scores + row * (int64_t)A.k : nullptr;
    const int64_t per = (len + CS - 1) / CS;
    const int64_t lo = min((int64_t)rank * per, len), hi = min(lo + per, len);
    const int m = (int)(hi - lo);

    if (len <= A.k) {                          // everything competes and wins
        for (int i = tid; i < m; i += kClThreads) {
            out[lo + i] = (int32_t)cand_pos(pool_row, A.block, lo + i);
            if (out_s) out_s[lo + i] = s[lo + i];
        }
        if (rank == CS - 1)
            for (int64_t i = len + tid; i < A.k; i += kClThreads) {
                out[i] = -1;
                if (out_s) out_s[i] = 0.0f;
            }
        return;
    }
    const bool in_smem = per <= A.key_cap;
    if (in_smem)
        for (int i = tid; i < m; i += kClThreads) s_keys[i] = score_key(s[lo + i]);

    uint32_t prefix = 0, mask = 0, remaining = (uint32_t)A.k;
    const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = shifts[pass], nb = 1 << widths[pass];
        for (int i = tid; i < kClBins; i += kClThreads) s_hist[i] = 0;
        __syncthreads();
        for (int base = 0; base < m; base += kClThreads) {
            const int i = base + tid;
            uint32_t key = 0;
            bool act = false;
            if (i < m) {
                key = in_smem ? s_keys[i] : score_key(s[lo + i]);
                act = (key & mask) == prefix;
            }
            const uint32_t am = __ballot_sync(0xffffffffu, act);
            if (act) {
                const uint32_t digit = (key >> shift) & (uint32_t)(nb - 1);
                const uint32_t peers = __match_any_sync(am, digit);
                if (lane == __ffs(peers) - 1) atomicAdd(&s_hist[digit], (uint32_t)__popc(peers));
            }
        }
        cl.sync();
        // thread t owns bins nb-1-4t .. nb-4-4t (descending); cluster-wide totals
        uint32_t tot[4], sum = 0;
        {
            // all remote loads of this thread's four bins issued before any is consumed
            const int bin0 = nb - 4 - 4 * tid;               // bins bin0 .. bin0+3
            uint4 part[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                part[r] = make_uint4(0, 0, 0, 0);
                if (r < CS && bin0 >= 0)
                    part[r] = *reinterpret_cast<const uint4 *>(cl.map_shared_rank(s_hist, r) + bin0);
            }
            uint4 t4 = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                t4.x += part[r].x; t4.y += part[r].y; t4.z += part[r].z; t4.w += part[r].w;
            }
            tot[0] = t4.w; tot[1] = t4.z; tot[2] = t4.y; tot[3] = t4.x;  // descending bins
            sum = t4.x + t4.y + t4.z + t4.w;
        }
        uint32_t all;
        uint32_t c = cl_block_excl_sum(sum, s_warp, all);   // elements with a larger digit
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int bin = nb - 1 - (4 * tid + j);
            if (bin >= 0 && c < remaining && c + tot[j] >= remaining) {
                s_pick[0] = (uint32_t)bin;
                s_pick[1] = remaining - c;
            }
            c += tot[j];
        }
        cl.sync();                             // histograms read everywhere before reuse
        prefix |= s_pick[0] << shift;
        mask |= (uint32_t)(nb - 1) << shift;
        remaining = s_pick[1];
    }
    const uint32_t tau = prefix, need = remaining;   // take `need` entries equal to tau

    // counts of this slice, then what earlier CTAs of the cluster select.  Thread t owns the
    // contiguous run [t*run, (t+1)*run) of the slice, so two block scans order everything.
    const int run = (m + kClThreads - 1) / kClThreads;
    const int r0 = min(tid * run, m), r1 = min(r0 + run, m);
    uint32_t n_gt = 0, n_eq = 0;
    for (int i = r0; i < r1; ++i) {
        const uint32_t key = in_smem ? s_keys[i] : score_key(s[lo + i]);
        n_gt += key > tau;
        n_eq += key == tau;
    }
    uint32_t t_gt, t_eq;
    const uint32_t gt_mine_before = cl_block_excl_sum(n_gt, s_warp, t_gt);
    const uint32_t eq_mine_before = cl_block_excl_sum(n_eq, s_warp, t_eq);
    if (tid == 0) { s_cnt[0] = t_gt; s_cnt[1] = t_eq; }
    cl.sync();
    uint32_t gt_before = 0, eq_before = 0;
    for (int r = 0; r < rank; ++r) {
        const uint32_t *rc = cl.map_shared_rank(s_cnt, r);
        gt_before += rc[0];
        eq_before += rc[1];
    }
    cl.sync();                                 // remote counts read: CTAs may now finish alone
    // ties taken by this thread: the ones whose cluster-wide tie rank is below `need`
    const uint32_t tie0 = eq_before + eq_mine_before;
    const uint32_t take_eq = tie0 >= need ? 0u : min(n_eq, need - tie0);
    uint32_t t_sel;
    const uint32_t sel_before = cl_block_excl_sum(n_gt + take_eq, s_warp, t_sel);
    uint32_t out_pos = gt_before + min(eq_before, need) + sel_before;
    uint32_t ties = 0;
    for (int i = r0; i < r1; ++i) {
        const uint32_t key = in_smem ? s_keys[i] : score_key(s[lo + i]);
        bool sel = key > tau;
        if (key == tau) sel = ties++ < take_eq;
        if (sel) {
            if (out_pos < (uint32_t)A.k) {
                out[out_pos] = (int32_t)cand_pos(pool_row, A.block, lo + i);
                if (out_s) out_s[out_pos] = s[lo + i];
            }
            ++out_pos;
        }
    }
    (void)gt_mine_before;
}

int cluster_size_for(int64_t rows, int64_t n)
{
    int64_t want = (152 + rows - 1) / (rows > 0 ? rows : 1);          // about one CTA per SM
    int64_t need = (n + kClKeyCap - 1) / kClKeyCap;                   // keep keys on chip
    int64_t c = want > need ? want : need;
    int64_t per_min = 2048;                                           // no tiny slices
    int64_t cap = (n + per_min - 1) / per_min;
    if (c > cap) c = cap;
    int cs = 1;
    while (cs < c && cs < 16) cs <<= 1;
    return cs;
}

cudaError_t launch_topk_cluster(ClusterTopkArgs A, int64_t rows, cudaStream_t s)
{
    const int cs = cluster_size_for(rows, A.n);
    const int64_t per = (A.n + cs - 1) / cs;          // slice of the longest possible row
    const size_t smem = per <= kClKeyCap ? (size_t)(per > 0 ? per : 1) * sizeof(uint32_t) : 0;
    A.key_cap = (int64_t)(smem / sizeof(uint32_t));
    cudaError_t e = cudaFuncSetAttribute(topk_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(kClKeyCap * sizeof(uint32_t)));
    if (e != cudaSuccess) return e;
    if (cs > 8) {
        e = cudaFuncSetAttribute(topk_cluster_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cs, (unsigned)rows, 1);
    cfg.blockDim = dim3(kClThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, topk_cluster_kernel, A);
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

size_t topk_ws_bytes(int64_t, int64_t, int32_t) { return 0; }

cudaError_t launch_topk(const float *scores, int64_t rows, int64_t n, const int32_t *row_len,
                        const int32_t *pool, int32_t block, int32_t k, int32_t *idx,
                        float *out_scores, void *, uint32_t *, cudaStream_t s)
{
    if (rows == 0 || k == 0) return cudaSuccess;
    if (rows > 65535) {
        topk_radix_kernel<<<(unsigned)rows, kTopkThreads, 0, s>>>(scores, n, row_len, pool, block, k,
                                                                 idx, out_scores);
        return cudaGetLastError();
    }
    ClusterTopkArgs A{scores, n, row_len, pool, block, k, idx, out_scores, 0};
    return launch_topk_cluster(A, rows, s);
}

size_t block_candidates_ws_bytes(int64_t rows, int64_t n, int32_t block, int32_t)
{
    const int64_t nbmax = (n + block - 1) / block;
    size_t a = (size_t)rows * (size_t)nbmax * sizeof(float);
    a = (a + 255) & ~(size_t)255;
    return a + (size_t)rows * sizeof(int32_t);
}

cudaError_t launch_block_candidates(const float *scores, int64_t rows, int64_t n,
                                    const int32_t *row_len, int32_t block, int32_t nb,
                                    int32_t *block_ids, void *ws, uint32_t *d_status,
                                    cudaStream_t s)
{
    if (rows == 0 || nb == 0) return cudaSuccess;
    const int64_t nbmax = (n + block - 1) / block;
    float *bscores = static_cast<float *>(ws);
    size_t off = ((size_t)rows * (size_t)nbmax * sizeof(float) + 255) & ~(size_t)255;
    int32_t *brow_len = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + off);
    int64_t gx = (nbmax + 255) / 256;
    if (gx > 64) gx = 64;
    if (gx < 1) gx = 1;
    block_max_kernel<<<dim3((unsigned)gx, (unsigned)rows), 256, 0, s>>>(scores, n, row_len, block,
                                                                        nbmax, bscores, brow_len);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_topk(bscores, rows, nbmax, brow_len, nullptr, 1, nb, block_ids, nullptr, nullptr,
                       d_status, s);
}

} // namespace csa2
