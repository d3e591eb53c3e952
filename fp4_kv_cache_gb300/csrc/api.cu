// api.cu -- extern "C" entry points of libcsa2.so (declared in include/csa2.h).
//
// Host-side validation happens here, before any launch; the kernels live in quant.cu (cache
// codec, RoPE + quantise), index_tc.cu and index_score.cu (indexer), topk.cu (Top-K, block
// pool), attn_tc.cu and attn.cu (attention) and selftest.cu (bounded-wait check);
// noalloc.cu holds the indexer entry point that needs no workspace.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/csa2.h"
#include "internal.h"

using namespace csa2;

namespace csa2 {

// Streaming multiprocessors of the current device, queried once per device ordinal (grid
// sizes are multiples of it); 1 if the query fails.
int device_sm_count()
{
    constexpr int kMaxDevices = 64;
    static std::atomic<int> cached[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
    if (dev < kMaxDevices) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
    if (dev < kMaxDevices) cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

} // namespace csa2

namespace {

inline bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

inline csa2_status from_cuda(cudaError_t e) { return e == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA; }

inline cudaStream_t as_stream(csa2_stream s) { return reinterpret_cast<cudaStream_t>(s); }

// values per scale of a 4-bit format (0: not a format)
inline int fmt_block(csa2_fp4_format f)
{
    return f == CSA2_FMT_MXFP4 ? 32 : f == CSA2_FMT_NVFP4_E4M3_16 ? 16 : 0;
}

bool index_args_ok(const csa2_index_args *a)
{
    if (!a) return false;
    if (a->batch < 0 || a->n_q < 0 || a->n_keys < 0 || a->n_keys >= (int64_t(1) << 31)) return false;
    if ((int64_t)a->batch * a->n_q > 65535) return false;
    if (a->n_heads < 1 || a->n_heads > 64) return false;
    if (a->head_dim != 32 && a->head_dim != 64 && a->head_dim != 128) return false;
    if (a->ratio_m < 1) return false;
    if (a->mode != CSA2_INDEX_FULL && a->mode != CSA2_INDEX_POOL) return false;
    if (a->block < 1 || a->block > 32) return false;
    if (a->fresh_from < 0) return false;
    const bool empty = (int64_t)a->batch * a->n_q == 0;
    if (!empty && (!a->q || !a->w || (a->n_keys > 0 && (!a->k_codes || !a->k_scales)))) return false;
    if (a->k_codes && !aligned(a->k_codes, 16)) return false;
    if (a->mode == CSA2_INDEX_POOL) {
        if (a->n_pool_blocks < 0) return false;
        if (!empty && a->n_pool_blocks > 0 && !a->pool_blocks) return false;
        if ((int64_t)a->n_pool_blocks * a->block >= (int64_t(1) << 31)) return false;
    }
    return true;
}

int64_t index_candidates(const csa2_index_args *a)
{
    return a->mode == CSA2_INDEX_POOL ? (int64_t)a->n_pool_blocks * a->block : a->n_keys;
}

bool attn_args_ok(const csa2_attn_args *a)
{
    if (!a) return false;
    if (a->batch < 0 || a->n_q < 0 || a->n_kv < 0) return false;
    if ((int64_t)a->batch * a->n_q > 65535) return false;
    if (a->n_heads < 1 || a->n_heads > 128) return false;
    if (a->d_qk < 32 || a->d_qk > 1024 || a->d_qk % 32) return false;
    if (a->d_v < 8 || a->d_v > a->d_qk || a->d_v % 8) return false;
    if (a->topk < 0 || a->topk > 2048 || a->window < 0) return false;
    if (a->kv_fmt != CSA2_FMT_MXFP4 && a->kv_fmt != CSA2_FMT_NVFP4_E4M3_16) return false;
    const bool empty = (int64_t)a->batch * a->n_q == 0;
    if (empty) return true;
    if (!a->q) return false;
    if (a->topk > 0 && (!a->idx || (a->n_kv > 0 && (!a->kv_codes || !a->kv_scales)))) return false;
    if (a->swa_fmt != CSA2_SWA_BF16 && a->swa_fmt != CSA2_SWA_MXFP8) return false;
    if (a->swa) {
        if (a->n_swa < 0 || !a->swa_pos0 || !a->q_pos) return false;
        if (a->swa_fmt == CSA2_SWA_MXFP8 && !a->swa_scales) return false;
    }
    return true;
}

} // namespace

extern "C" {

const char *csa2_status_string(csa2_status s)
{
    switch (s) {
    case CSA2_OK: return "ok";
    case CSA2_ERR_INVALID_ARG: return "invalid argument";
    case CSA2_ERR_UNSUPPORTED: return "unsupported request";
    case CSA2_ERR_CUDA: return "CUDA launch error";
    case CSA2_ERR_WORKSPACE: return "workspace too small";
    }
    return "unknown status";
}

int csa2_version(void) { return 100; }

size_t csa2_cache_bytes_per_position(csa2_fp4_format main_fmt, int32_t d_main, int32_t d_idx)
{
    if (d_main <= 0 || d_idx <= 0 || d_idx % 32) return 0;
    size_t main_bytes;
    if (main_fmt == CSA2_FMT_MXFP4) {
        if (d_main % 32) return 0;
        main_bytes = (size_t)d_main / 2 + (size_t)d_main / 32;     // E2M1 codes + E8M0 / 32
    } else if (main_fmt == CSA2_FMT_NVFP4_E4M3_16) {
        if (d_main % 16) return 0;
        main_bytes = (size_t)d_main / 2 + (size_t)d_main / 16;     // E2M1 codes + E4M3 / 16
    } else {
        return 0;
    }
    return main_bytes + (size_t)d_idx / 2 + (size_t)d_idx / 32;    // MXFP4 indexer key
}

csa2_status csa2_quant_fp4(const void *x, csa2_dtype xt, int64_t rows, int64_t cols, int64_t ldx,
                           uint8_t *codes, int64_t ldc, uint8_t *scales, int64_t lds,
                           csa2_fp4_format fmt, uint32_t *d_status, csa2_stream stream)
{
    const int G = fmt_block(fmt);
    if (!G || (xt != CSA2_BF16 && xt != CSA2_F32)) return CSA2_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || cols % G) return CSA2_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return CSA2_OK;
    if (!x || !codes || !scales) return CSA2_ERR_INVALID_ARG;
    if (ldx < cols || ldc < cols / 2 || lds < cols / G) return CSA2_ERR_INVALID_ARG;
    if (fmt == CSA2_FMT_NVFP4_E4M3_16)
        return from_cuda(launch_quant_nvfp4(x, xt == CSA2_BF16, rows, cols, ldx, codes, ldc, scales,
                                            lds, d_status, as_stream(stream)));
    return from_cuda(launch_quant_mxfp4(x, xt == CSA2_BF16, rows, cols, ldx, codes, ldc, scales,
                                        lds, d_status, as_stream(stream)));
}

csa2_status csa2_quant_fp4_batch(const csa2_quant_job *jobs, int32_t n_jobs, csa2_fp4_format fmt,
                                 uint32_t *d_status, csa2_stream stream)
{
    const int G = fmt_block(fmt);
    if (!G || n_jobs < 0 || n_jobs > CSA2_QUANT_MAX_JOBS) return CSA2_ERR_INVALID_ARG;
    if (n_jobs == 0) return CSA2_OK;
    if (!jobs) return CSA2_ERR_INVALID_ARG;
    QuantJobDesc d[CSA2_QUANT_MAX_JOBS];
    bool vec = fmt == CSA2_FMT_MXFP4;
    for (int k = 0; k < n_jobs; ++k) {
        const csa2_quant_job &j = jobs[k];
        if (j.xt != CSA2_BF16 && j.xt != CSA2_F32) return CSA2_ERR_INVALID_ARG;
        if (j.rows < 0 || j.cols < 0 || j.cols % G) return CSA2_ERR_INVALID_ARG;
        if (j.rows && j.cols) {
            if (!j.x || !j.codes || !j.scales) return CSA2_ERR_INVALID_ARG;
            if (j.ldx < j.cols || j.ldc < j.cols / 2 || j.lds < j.cols / G) return CSA2_ERR_INVALID_ARG;
        }
        d[k] = {j.x, j.xt == CSA2_BF16, j.rows, j.cols, j.ldx, j.codes, j.ldc, j.scales, j.lds};
        vec = vec && quant_job_vec_ok(d[k]);
    }
    if (vec) return from_cuda(launch_quant_mxfp4_batch(d, n_jobs, d_status, as_stream(stream)));
    for (int k = 0; k < n_jobs; ++k) {           // NVFP4 or misaligned rows: one launch per job
        const cudaError_t e =
            fmt == CSA2_FMT_NVFP4_E4M3_16
                ? launch_quant_nvfp4(d[k].x, d[k].x_bf16, d[k].rows, d[k].cols, d[k].ldx, d[k].codes, d[k].ldc,
                                     d[k].scales, d[k].lds, d_status, as_stream(stream))
                : launch_quant_mxfp4(d[k].x, d[k].x_bf16, d[k].rows, d[k].cols, d[k].ldx, d[k].codes, d[k].ldc,
                                     d[k].scales, d[k].lds, d_status, as_stream(stream));
        if (e != cudaSuccess) return from_cuda(e);
    }
    return CSA2_OK;
}

csa2_status csa2_rope_quant_fp4(const csa2_rope_quant_job *jobs, int32_t n_jobs, uint32_t *d_status,
                                csa2_stream stream)
{
    if (n_jobs < 0 || n_jobs > CSA2_QUANT_MAX_JOBS) return CSA2_ERR_INVALID_ARG;
    if (n_jobs == 0) return CSA2_OK;
    if (!jobs) return CSA2_ERR_INVALID_ARG;
    RopeQuantJobDesc d[CSA2_QUANT_MAX_JOBS];
    for (int k = 0; k < n_jobs; ++k) {
        const csa2_rope_quant_job &j = jobs[k];
        const int G = fmt_block(j.fmt);
        if (!G || j.rows < 0 || j.cols < 0 || j.cols % G) return CSA2_ERR_INVALID_ARG;
        if (j.rope_dim < 0 || j.rope_dim % 2 || j.rope_dim > j.cols) return CSA2_ERR_INVALID_ARG;
        if (j.rows && j.cols) {
            if (!j.x || !j.codes || !j.scales) return CSA2_ERR_INVALID_ARG;
            if (j.ldx < j.cols || j.ldc < j.cols / 2 || j.lds < j.cols / G) return CSA2_ERR_INVALID_ARG;
            if (!aligned(j.x, 16) || j.ldx % 8 || !aligned(j.codes, 4) || j.ldc % 4) return CSA2_ERR_INVALID_ARG;
            if (j.rope_dim > 0 && (!j.pos || !j.cos_sin || j.n_pos < 1 || !aligned(j.cos_sin, 4)))
                return CSA2_ERR_INVALID_ARG;
        }
        d[k] = {j.x, j.rows, j.cols, j.ldx, j.rope_dim, j.pos, j.cos_sin, j.n_pos, j.codes, j.ldc, j.scales, j.lds,
                j.fmt == CSA2_FMT_NVFP4_E4M3_16};
    }
    return from_cuda(launch_rope_quant(d, n_jobs, d_status, as_stream(stream)));
}

csa2_status csa2_quant_fp8(const void *x, csa2_dtype xt, int64_t rows, int64_t cols, int64_t ldx,
                           uint8_t *codes, int64_t ldc, uint8_t *scales, int64_t lds,
                           uint32_t *d_status, csa2_stream stream)
{
    if (xt != CSA2_BF16 && xt != CSA2_F32) return CSA2_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || cols % 32) return CSA2_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return CSA2_OK;
    if (!x || !codes || !scales) return CSA2_ERR_INVALID_ARG;
    if (ldx < cols || ldc < cols || lds < cols / 32) return CSA2_ERR_INVALID_ARG;
    return from_cuda(launch_quant_mxfp8(x, xt == CSA2_BF16, rows, cols, ldx, codes, ldc, scales, lds, d_status,
                                        as_stream(stream)));
}

csa2_status csa2_dequant_fp8(const uint8_t *codes, int64_t ldc, const uint8_t *scales, int64_t lds,
                             int64_t rows, int64_t cols, void *y, csa2_dtype yt, int64_t ldy,
                             csa2_stream stream)
{
    if (yt != CSA2_BF16 && yt != CSA2_F32) return CSA2_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || cols % 32) return CSA2_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return CSA2_OK;
    if (!y || !codes || !scales) return CSA2_ERR_INVALID_ARG;
    if (ldy < cols || ldc < cols || lds < cols / 32) return CSA2_ERR_INVALID_ARG;
    return from_cuda(launch_dequant_mxfp8(codes, ldc, scales, lds, rows, cols, y, yt == CSA2_BF16, ldy,
                                          as_stream(stream)));
}

csa2_status csa2_dequant_fp4(const uint8_t *codes, int64_t ldc, const uint8_t *scales,
                             int64_t lds, int64_t rows, int64_t cols, csa2_fp4_format fmt,
                             void *y, csa2_dtype yt, int64_t ldy, csa2_stream stream)
{
    const int G = fmt_block(fmt);
    if (!G || (yt != CSA2_BF16 && yt != CSA2_F32)) return CSA2_ERR_INVALID_ARG;
    if (rows < 0 || cols < 0 || cols % G) return CSA2_ERR_INVALID_ARG;
    if (rows == 0 || cols == 0) return CSA2_OK;
    if (!y || !codes || !scales) return CSA2_ERR_INVALID_ARG;
    if (ldy < cols || ldc < cols / 2 || lds < cols / G) return CSA2_ERR_INVALID_ARG;
    return from_cuda(launch_dequant_fp4(codes, ldc, scales, lds, rows, cols, fmt == CSA2_FMT_NVFP4_E4M3_16, y,
                                        yt == CSA2_BF16, ldy, as_stream(stream)));
}

size_t csa2_index_score_workspace_size(const csa2_index_args *a)
{
    if (!index_args_ok(a)) return 0;
    return index_score_ws_bytes(*a);
}

csa2_status csa2_index_score(const csa2_index_args *a, float *scores, int32_t *row_len, void *ws,
                             size_t ws_bytes, uint32_t *d_status, csa2_stream stream)
{
    if (!index_args_ok(a)) return CSA2_ERR_INVALID_ARG;
    if ((int64_t)a->batch * a->n_q == 0) return CSA2_OK;
    if (!scores && index_candidates(a) > 0) return CSA2_ERR_INVALID_ARG;
    const size_t need = csa2_index_score_workspace_size(a);
    if (ws_bytes < need) return CSA2_ERR_WORKSPACE;
    if (need && (!ws || !aligned(ws, 16))) return CSA2_ERR_INVALID_ARG;
    return from_cuda(launch_index_score(*a, scores, row_len, need ? ws : nullptr, d_status,
                                        as_stream(stream)));
}

// An exact context fits scores of `rows` rows of n candidates: rows = batch * n_q and n its
// candidate count; in POOL mode the pool is given again and matches, in FULL mode none is.
bool exact_ctx_ok(const csa2_index_args *ex, int64_t rows, int64_t n, const int32_t *pool_blocks,
                  int32_t block, const int32_t *row_len, bool blocks)
{
    if (!index_args_ok(ex) || !aligned(ex->q, 16)) return false;
    if ((int64_t)ex->batch * ex->n_q != rows || index_candidates(ex) != n || !row_len) return false;
    if (ex->mode == CSA2_INDEX_POOL) {
        if (blocks || pool_blocks != ex->pool_blocks || block != ex->block) return false;
    } else if (pool_blocks) {
        return false;
    }
    return true;
}

size_t csa2_topk_workspace_size(int64_t rows, int64_t n, int32_t k, const csa2_index_args *exact)
{
    return topk_ws_bytes(rows, n, k, exact != nullptr);
}

csa2_status csa2_topk(const float *scores, int64_t rows, int64_t n, const int32_t *row_len,
                      const uint32_t *group_max, const int32_t *pool_blocks, int32_t block,
                      const csa2_index_args *exact, int32_t k, int32_t *idx, float *out_scores, void *ws,
                      size_t ws_bytes, uint32_t *d_status, csa2_stream stream)
{
    if (rows < 0 || n < 0 || n >= (int64_t(1) << 31) || k < 0 || rows > (int64_t(1) << 31))
        return CSA2_ERR_INVALID_ARG;
    if (pool_blocks && (block < 1 || n % block)) return CSA2_ERR_INVALID_ARG;
    if (exact && !exact_ctx_ok(exact, rows, n, pool_blocks, block, row_len, false)) return CSA2_ERR_INVALID_ARG;
    if (rows == 0 || k == 0) return CSA2_OK;
    if (!idx || (n > 0 && !scores)) return CSA2_ERR_INVALID_ARG;
    const size_t need = csa2_topk_workspace_size(rows, n, k, exact);
    if (ws_bytes < need) return CSA2_ERR_WORKSPACE;
    if (exact && (!ws || !aligned(ws, 16))) return CSA2_ERR_INVALID_ARG;
    if (group_max && !aligned(group_max, 4)) return CSA2_ERR_INVALID_ARG;
    return from_cuda(launch_topk(scores, rows, n, row_len, group_max, pool_blocks, block, k, idx,
                                 out_scores, ws, d_status, as_stream(stream), exact));
}

// csa2_index_topk workspace.  Tensor-core FULL mode with one query per CTA (the decode
// shape): the indexer's tile counters | candidate keys | positions | list meta | band slots.
// Otherwise: the indexer's workspace | scores | row lengths | csa2_topk's workspace.
namespace {
struct FusedLayout {
    bool fused;
    int64_t ctas, cap;            // fused: lists per row, entries per list
    size_t idx_ws, a, b, c, d, total;
};
FusedLayout fused_layout(const csa2_index_args &a, int32_t k)
{
    FusedLayout L = {};
    const int64_t rows = (int64_t)a.batch * a.n_q;
    L.idx_ws = index_score_ws_bytes(a);
    L.fused = index_tc_fusable(a);
    size_t off = (L.idx_ws + 255) & ~(size_t)255;
    if (L.fused) {
        int stages;
        index_fused_shape(a, L.ctas, stages);
        L.cap = (int64_t)stages * 256;
        const size_t lst = (size_t)rows * L.ctas * L.cap * sizeof(uint32_t);
        L.a = off;
        L.b = L.a + ((lst + 255) & ~(size_t)255);
        L.c = L.b + ((lst + 255) & ~(size_t)255);
        L.d = L.c + (((size_t)rows * L.ctas * 4 * sizeof(uint32_t) + 255) & ~(size_t)255);
        L.total = L.d + topk_lists_ws_bytes(rows);
    } else {
        const int64_t n = index_candidates(&a);
        L.a = off;                                          // scores
        L.b = L.a + (((size_t)rows * n * sizeof(float) + 255) & ~(size_t)255);   // row lengths
        L.c = L.b + (((size_t)rows * sizeof(int32_t) + 255) & ~(size_t)255);     // Top-K workspace
        L.total = L.c + topk_ws_bytes(rows, n, k, true);
    }
    return L;
}
} // namespace

size_t csa2_index_topk_workspace_size(const csa2_index_args *a, int32_t k)
{
    if (!index_args_ok(a) || k < 0) return 0;
    return fused_layout(*a, k).total;
}

csa2_status csa2_index_topk(const csa2_index_args *a, int32_t k, int32_t *idx, float *out_scores,
                            int32_t *row_len, void *ws, size_t ws_bytes, uint32_t *d_status,
                            csa2_stream stream)
{
    if (!index_args_ok(a) || k < 0 || !aligned(a->q, 16)) return CSA2_ERR_INVALID_ARG;
    const int64_t rows = (int64_t)a->batch * a->n_q;
    if (rows == 0) return CSA2_OK;
    if (k > 0 && !idx) return CSA2_ERR_INVALID_ARG;
    const FusedLayout L = fused_layout(*a, k);
    if (ws_bytes < L.total) return CSA2_ERR_WORKSPACE;
    if (!ws || !aligned(ws, 16)) return CSA2_ERR_INVALID_ARG;
    char *w = static_cast<char *>(ws);
    const cudaStream_t s = as_stream(stream);
    uint32_t *tile_ctr = L.idx_ws ? reinterpret_cast<uint32_t *>(w) : nullptr;
    if (L.fused) {
        FusedOut fo;
        fo.key = reinterpret_cast<uint32_t *>(w + L.a);
        fo.pos = reinterpret_cast<int32_t *>(w + L.b);
        fo.meta = reinterpret_cast<uint32_t *>(w + L.c);
        fo.k = k > 0 ? k : 1;
        cudaError_t e = launch_index_tc(*a, nullptr, row_len, tile_ctr, d_status, s, &fo);
        if (e != cudaSuccess || k == 0) return from_cuda(e);
        return from_cuda(launch_topk_lists(*a, k, fo.key, fo.pos, fo.meta, (int)L.ctas, L.cap, idx, out_scores,
                                           w + L.d, d_status, s));
    }
    float *scores = reinterpret_cast<float *>(w + L.a);
    int32_t *rl = row_len ? row_len : reinterpret_cast<int32_t *>(w + L.b);
    cudaError_t e = launch_index_score(*a, scores, rl, tile_ctr, d_status, s);
    if (e != cudaSuccess || k == 0) return from_cuda(e);
    const int64_t n = index_candidates(a);
    const bool pool = a->mode == CSA2_INDEX_POOL;
    return from_cuda(launch_topk(scores, rows, n, rl, nullptr, pool ? a->pool_blocks : nullptr, a->block, k, idx,
                                 out_scores, w + L.c, d_status, s, a));
}

size_t csa2_block_candidates_workspace_size(int64_t rows, int64_t n, int32_t block, int32_t nb,
                                            const csa2_index_args *exact)
{
    if (rows <= 0 || n < 0 || block < 1 || nb <= 0) return 0;
    return block_candidates_ws_bytes(rows, n, block, nb, exact != nullptr);
}

csa2_status csa2_block_candidates(const float *scores, int64_t rows, int64_t n,
                                  const int32_t *row_len, int32_t block, int32_t nb,
                                  const csa2_index_args *exact, int32_t *block_ids, void *ws,
                                  size_t ws_bytes, uint32_t *d_status, csa2_stream stream)
{
    if (rows < 0 || n < 0 || n >= (int64_t(1) << 31) || block < 1 || nb < 0 ||
        rows > (int64_t(1) << 31))
        return CSA2_ERR_INVALID_ARG;
    if (exact && !exact_ctx_ok(exact, rows, n, nullptr, block, row_len, true)) return CSA2_ERR_INVALID_ARG;
    if (rows == 0 || nb == 0) return CSA2_OK;
    if (!block_ids || (n > 0 && !scores)) return CSA2_ERR_INVALID_ARG;
    const size_t need = csa2_block_candidates_workspace_size(rows, n, block, nb, exact);
    if (ws_bytes < need) return CSA2_ERR_WORKSPACE;
    if (need && (!ws || !aligned(ws, 16))) return CSA2_ERR_INVALID_ARG;
    return from_cuda(launch_block_candidates(scores, rows, n, row_len, block, nb, block_ids, ws,
                                             d_status, as_stream(stream), exact));
}

size_t csa2_sparse_attn_workspace_size(const csa2_attn_args *a)
{
    return a ? sparse_attn_ws_bytes(*a) : 0;
}

csa2_status csa2_sparse_attn(const csa2_attn_args *a, uint16_t *out, float *lse, void *ws,
                             size_t ws_bytes, uint32_t *d_status, csa2_stream stream)
{
    if (!attn_args_ok(a)) return CSA2_ERR_INVALID_ARG;
    if ((int64_t)a->batch * a->n_q == 0) return CSA2_OK;
    if (!out) return CSA2_ERR_INVALID_ARG;
    const size_t need = csa2_sparse_attn_workspace_size(a);
    if (ws_bytes < need) return CSA2_ERR_WORKSPACE;
    if (need && (!ws || !aligned(ws, 16))) return CSA2_ERR_INVALID_ARG;
    return from_cuda(launch_sparse_attn(*a, out, lse, ws, d_status, as_stream(stream)));
}

csa2_status csa2_selftest_bounded_wait(uint32_t polls, uint32_t *d_status, csa2_stream stream)
{
    if (polls < 1 || polls > (1u << 20) || !d_status) return CSA2_ERR_INVALID_ARG;
    return from_cuda(launch_bounded_wait_selftest(polls, d_status, as_stream(stream)));
}

} // extern "C"
