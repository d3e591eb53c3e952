// internal.h -- launchers shared between the kernel files and the C-ABI layer.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>
#include <utility>
#include "../../include/csa2.h"

namespace csa2 {

cudaError_t launch_quant_mxfp4(const void *x, bool x_bf16, int64_t rows, int64_t cols, int64_t ldx,
                               uint8_t *codes, int64_t ldc, uint8_t *scales, int64_t lds,
                               uint32_t *d_status, cudaStream_t s);
// One launch for up to four quantisation jobs whose rows meet the vector kernel's alignment
// (returns cudaErrorInvalidValue, launching nothing, when one does not).
struct QuantJobDesc {
    const void *x;
    bool x_bf16;
    int64_t rows, cols, ldx;
    uint8_t *codes;
    int64_t ldc;
    uint8_t *scales;
    int64_t lds;
};
bool quant_job_vec_ok(const QuantJobDesc &j);
cudaError_t launch_quant_mxfp4_batch(const QuantJobDesc *jobs, int n_jobs, uint32_t *d_status, cudaStream_t s);
cudaError_t launch_quant_nvfp4(const void *x, bool x_bf16, int64_t rows, int64_t cols, int64_t ldx,
                               uint8_t *codes, int64_t ldc, uint8_t *scales, int64_t lds,
                               uint32_t *d_status, cudaStream_t s);
// The cache write with the rotary embedding fused in (csa2_rope_quant_fp4): up to four jobs,
// rows already validated (16-byte aligned bf16 x, 4-byte aligned codes).
struct RopeQuantJobDesc {
    const uint16_t *x;
    int64_t rows, cols, ldx;
    int32_t rope_dim;
    const int32_t *pos;
    const float *cos_sin;
    int64_t n_pos;
    uint8_t *codes;
    int64_t ldc;
    uint8_t *scales;
    int64_t lds;
    bool nvfp4;
};
cudaError_t launch_rope_quant(const RopeQuantJobDesc *jobs, int n_jobs, uint32_t *d_status, cudaStream_t s);
cudaError_t launch_quant_mxfp8(const void *x, bool x_bf16, int64_t rows, int64_t cols, int64_t ldx,
                               uint8_t *codes, int64_t ldc, uint8_t *scales, int64_t lds,
                               uint32_t *d_status, cudaStream_t s);
cudaError_t launch_dequant_mxfp8(const uint8_t *codes, int64_t ldc, const uint8_t *scales, int64_t lds,
                                 int64_t rows, int64_t cols, void *y, bool y_bf16, int64_t ldy, cudaStream_t s);
cudaError_t launch_dequant_fp4(const uint8_t *codes, int64_t ldc, const uint8_t *scales,
                               int64_t lds, int64_t rows, int64_t cols, bool nvfp4, void *y,
                               bool y_bf16, int64_t ldy, cudaStream_t s);

// Indexer scoring: tensor-core path where it applies (index_tc.cu; it re-scores the rare
// positions it cannot prove exact on CUDA cores), else the exact CUDA-core kernel
// (index_score.cu).
size_t index_score_ws_bytes(const csa2_index_args &a);
cudaError_t launch_index_score(const csa2_index_args &a, float *scores, int32_t *row_len, void *ws,
                               uint32_t *d_status, cudaStream_t s);
cudaError_t launch_index_exact(const csa2_index_args &a, float *scores, int32_t *row_len,
                               uint32_t *d_status, cudaStream_t s);
bool index_tc_eligible(const csa2_index_args &a);
int64_t index_tc_ctas_per_row(const csa2_index_args &a);
// Candidate lists of the fused selection (csa2_index_topk): per row, `ctas` lists of
// stages x 256 entries (key, position) in position order, and per list (count, K-th key,
// non-finite flag, 0).
struct FusedOut {
    uint32_t *key;
    int32_t *pos;
    uint32_t *meta;
    int32_t k;
};
bool index_tc_fusable(const csa2_index_args &a);
void index_fused_shape(const csa2_index_args &a, int64_t &ctas, int &stages);
cudaError_t launch_index_tc(const csa2_index_args &a, float *scores, int32_t *row_len,
                            uint32_t *tile_ctr, uint32_t *d_status, cudaStream_t s,
                            const FusedOut *fo = nullptr);
// The exact Top-K of every row from its candidate lists (see TopkLists in topk.cu);
// ws: topk_lists_ws_bytes(rows).
size_t topk_lists_ws_bytes(int64_t rows);
cudaError_t launch_topk_lists(const csa2_index_args &ex, int32_t k, const uint32_t *key, const int32_t *pos,
                              const uint32_t *meta, int n_lists, int64_t cap, int32_t *idx, float *out_scores,
                              void *ws, uint32_t *d_status, cudaStream_t s);

// Top-K over rows of float scores (see csa2_topk).  ws: topk_ws_bytes(rows, n, k, ex != 0).
// ex != NULL: exact order for the scores of csa2_index_score(*ex); candidates are positions
// (unit 1) or blocks of `unit` positions whose position scores are pos_scores [rows, pos_n]
// with valid lengths pos_len.
size_t topk_ws_bytes(int64_t rows, int64_t n, int32_t k, bool exact);
cudaError_t launch_topk(const float *scores, int64_t rows, int64_t n, const int32_t *row_len,
                        const uint32_t *group_max, const int32_t *pool, int32_t block, int32_t k,
                        int32_t *idx, float *out_scores, void *ws, uint32_t *d_status,
                        cudaStream_t s, const csa2_index_args *ex = nullptr, int32_t unit = 1,
                        const float *pos_scores = nullptr, int64_t pos_n = 0,
                        const int32_t *pos_len = nullptr);
size_t block_candidates_ws_bytes(int64_t rows, int64_t n, int32_t block, int32_t nb, bool exact);
cudaError_t launch_block_candidates(const float *scores, int64_t rows, int64_t n,
                                    const int32_t *row_len, int32_t block, int32_t nb,
                                    int32_t *block_ids, void *ws, uint32_t *d_status,
                                    cudaStream_t s, const csa2_index_args *ex);

// Streaming multiprocessors of the current device (queried once per device).
int device_sm_count();

size_t sparse_attn_ws_bytes(const csa2_attn_args &a);
bool attn_tc_eligible(const csa2_attn_args &a);
size_t attn_tc_ws_bytes(const csa2_attn_args &a);
cudaError_t launch_attn_tc(const csa2_attn_args &a, uint16_t *out, float *lse, void *ws,
                           uint32_t *d_status, cudaStream_t s);
cudaError_t launch_sparse_attn(const csa2_attn_args &a, uint16_t *out, float *lse, void *ws,
                               uint32_t *d_status, cudaStream_t s);

// Self-test of the bounded device waits (csa2_selftest_bounded_wait).
cudaError_t launch_bounded_wait_selftest(uint32_t polls, uint32_t *d_status, cudaStream_t s);

// Launch with programmatic dependent launch: the kernel may start while the previous kernel
// in the stream is still running, and must execute griddepcontrol.wait (pdl_wait) before it
// reads anything that kernel writes.  cluster_x > 1 also groups consecutive CTAs along x
// into clusters of that size.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, unsigned cluster_x, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

} // namespace csa2
