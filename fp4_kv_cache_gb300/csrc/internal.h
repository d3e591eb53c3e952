// internal.h -- launchers shared between the kernel files and the C-ABI layer.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>
#include "../../include/csa2.h"

namespace csa2 {

cudaError_t launch_quant_mxfp4(const void *x, bool x_bf16, int64_t rows, int64_t cols, int64_t ldx,
                               uint8_t *codes, int64_t ldc, uint8_t *scales, int64_t lds,
                               uint32_t *d_status, cudaStream_t s);
cudaError_t launch_dequant_mxfp4(const uint8_t *codes, int64_t ldc, const uint8_t *scales,
                                 int64_t lds, int64_t rows, int64_t cols, void *y, bool y_bf16,
                                 int64_t ldy, cudaStream_t s);

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
cudaError_t launch_index_tc(const csa2_index_args &a, float *scores, int32_t *row_len,
                            uint32_t *tile_ctr, uint32_t *d_status, cudaStream_t s);

// Top-K over rows of float scores (see csa2_topk).  ws: topk_ws_bytes(rows, n, k).
size_t topk_ws_bytes(int64_t rows, int64_t n, int32_t k);
cudaError_t launch_topk(const float *scores, int64_t rows, int64_t n, const int32_t *row_len,
                        const uint32_t *group_max, const int32_t *pool, int32_t block, int32_t k,
                        int32_t *idx, float *out_scores, void *ws, uint32_t *d_status,
                        cudaStream_t s);
size_t block_candidates_ws_bytes(int64_t rows, int64_t n, int32_t block, int32_t nb);
cudaError_t launch_block_candidates(const float *scores, int64_t rows, int64_t n,
                                    const int32_t *row_len, int32_t block, int32_t nb,
                                    int32_t *block_ids, void *ws, uint32_t *d_status,
                                    cudaStream_t s);

size_t sparse_attn_ws_bytes(const csa2_attn_args &a);
bool attn_tc_eligible(const csa2_attn_args &a);
size_t attn_tc_ws_bytes(const csa2_attn_args &a);
cudaError_t launch_attn_tc(const csa2_attn_args &a, uint16_t *out, float *lse, void *ws,
                           uint32_t *d_status, cudaStream_t s);
cudaError_t launch_sparse_attn(const csa2_attn_args &a, uint16_t *out, float *lse, void *ws,
                               uint32_t *d_status, cudaStream_t s);

} // namespace csa2
