/*
 * csa2.h -- C ABI of libcsa2.so, the GB300 (sm_103a) CSA2 decode/prefill hot path.
 *
 * CSA2 = Compressed Sparse Attention 2 of "DeepSeek-V4.1-Flash: Pushing the Limits of
 * KV Cache Compression".  Citations name the page and its section:
 *   [report]  aipaper.jasonlin.tech  (the report's own text, its § numbers)
 *   [review]  papers.chlience.com    (analytical review; byte ledger, layer schedule)
 *
 * The path (report §2.3, §2.3.1, §2.3.2; review, "CSA2" section and Figure 4 reading):
 *   indexer Q + FP4 indexer K  -> scores -> Top-512 (+ block pool in the decoder's
 *   first Full layer) -> gather + dequantise the selected FP4 main-KV entries ->
 *   join with the layer's SWA window -> core latent attention over all query heads.
 * Modes (report §2.3.1): Full = score all visible entries; Reindex = score only the
 * block pool with the layer's own indexer query; Reuse = attention over given indices.
 *
 * Conventions for every entry point
 *   - Pointers are DEVICE pointers owned by the caller unless a comment says "host".
 *     The library never allocates device memory and never frees caller memory.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream)
 *     and is asynchronous: no call synchronises and none copies between host and device.
 *   - Scratch memory is a caller buffer `ws` of at least *_workspace_size() bytes
 *     (16-byte aligned); ws may be NULL when that size is 0.
 *   - Return value: CSA2_OK, or an error found on the host BEFORE anything is launched
 *     (bad shapes, NULL pointers, misalignment, too-small workspace, launch failure).
 *   - Errors found on the device are ORed as CSA2_DEV_* bits into *d_status (a caller
 *     uint32_t in device memory; may be NULL to ignore them).  Read it after the stream
 *     synchronises.  The affected outputs are then unspecified but every access stays
 *     in bounds.
 *   - bf16 tensors are passed as uint16_t bit patterns.  Layouts are dense row-major
 *     (C order) with the shapes given; "B" = batch, "T" = query tokens per sequence.
 *   - Calls on different streams with disjoint outputs may run concurrently; the
 *     library keeps no mutable global state.
 *   - Kernels are launched with programmatic dependent launch: a kernel may start its
 *     set-up while the kernel before it on the stream drains, and waits for that kernel
 *     to complete before it reads what that kernel may write.  The indexer, Top-K,
 *     attention and csa2_rope_quant_fp4 kernels let their dependents start right after
 *     that wait; the other conversion calls (csa2_quant_*, csa2_dequant_*) only when they
 *     finish.  Three read inputs before the wait: csa2_sparse_attn reads q, q_pos,
 *     swa_pos0, swa_start, swa and swa_scales (and works through the SWA window) before
 *     it (only idx may come from the kernel just before it); csa2_topk /
 *     csa2_block_candidates with an exact context read its q, w and k_scales before
 *     theirs (only the scores, row lengths and group maxima may come from the kernel just
 *     before them); and csa2_index_score / csa2_index_topk with fresh_from > 0 read q, w,
 *     q_pos and the cache positions below fresh_from before theirs.  Those inputs must not
 *     be written by a kernel that lets its dependents start early and runs just before
 *     the call: a plain kernel, a csa2_quant_* / csa2_dequant_* call, or a call of this
 *     library whose outputs they are not is fine (so a csa2_rope_quant_fp4 that writes
 *     the decoded token's cache rows may come just before the indexer with fresh_from set
 *     to that token's position, not just before an exact csa2_topk on the same cache).
 *     With fresh_from > 0 the kernel just before must not use this call's outputs or
 *     workspace either.
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CSA2_API __attribute__((visibility("default")))
#else
#define CSA2_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef void *csa2_stream; /* a cudaStream_t */

typedef enum {
    CSA2_OK = 0,
    CSA2_ERR_INVALID_ARG = 1, /* shape, pointer, alignment or enum out of range */
    CSA2_ERR_UNSUPPORTED = 2, /* valid request the library does not implement    */
    CSA2_ERR_CUDA = 3,        /* a CUDA launch or attribute call failed          */
    CSA2_ERR_WORKSPACE = 4    /* ws_bytes below the *_workspace_size() value     */
} csa2_status;

/* Device-side status bits (ORed into *d_status). */
#define CSA2_DEV_BAD_INDEX 0x1u  /* an attention index outside [-1, n_kv) was ignored      */
#define CSA2_DEV_BAD_POOL 0x2u   /* pool block ids not ascending-unique, -1 padded, in range */
#define CSA2_DEV_NONFINITE 0x4u  /* a quantiser block held Inf/NaN (its output unspecified) */
#define CSA2_DEV_TIMEOUT 0x8u    /* a bounded device wait gave up; outputs unspecified      */
#define CSA2_DEV_SCORE_RANGE 0x10u /* an indexer score left the float32 range (Inf/NaN): the */
                                   /* exact-order guarantee of the selections made on these */
                                   /* scores does not hold                                  */
#define CSA2_DEV_BAND_LIMIT 0x20u  /* a selection row had more candidates within the float32 */
                                   /* scores' error bound of its K-th score than the exact   */
                                   /* pass holds (CSA2_EXACT_BAND_CAP); that row follows the */
                                   /* float32 order                                          */

typedef enum { CSA2_BF16 = 0, CSA2_F32 = 1 } csa2_dtype;

/* 4-bit cache formats.
 * MXFP4: E2M1 codes + one E8M0 (power-of-two) scale per 32 values -- the OCP MX format
 *   the report gives for indexer queries and keys (report §2.4.4), used here for both
 *   caches.  Codes are packed two per byte, element 2i in the low nibble; scale byte
 *   e means 2^(e-127).  Quantisation: X = floor(log2(max|x|)) - 2 clamped to
 *   [-127, 127] (X = 0 for an all-zero block), element code = round-half-even of
 *   |x|/2^X onto {0, .5, 1, 1.5, 2, 3, 4, 6}, saturating at 6, sign bit = sign bit of x.
 * NVFP4_E4M3_16: E2M1 + one E4M3 scale per 16, no global scale -- the report's main-KV
 *   format (report §2.4.4; the review's byte ledger counts 256 B of codes and 32 B of
 *   scales for 512 channels).  Codes are packed as for MXFP4; scale byte = an E4M3 value
 *   (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; 0x7F/0xFF are NaN).  The pages
 *   do not say how a scale is chosen; here the block maximum is mapped onto 6: scale =
 *   amax/6 rounded to the nearest E4M3 value (ties to the even code, values above 448
 *   clamped to 448), element code = round-half-even of |x|/scale onto the E2M1 grid,
 *   saturating at 6, sign bit = sign bit of x; a scale that rounds to 0 encodes its block
 *   as signed zeros.  Every element value (code x scale) is exact in bf16.  Accepted by
 *   the codec calls and as the main-KV format of csa2_sparse_attn; the indexer keys are
 *   always MXFP4 (report §2.4.4). */
typedef enum { CSA2_FMT_MXFP4 = 0, CSA2_FMT_NVFP4_E4M3_16 = 1 } csa2_fp4_format;

/* SWA KV formats.  The report keeps the SWA cache in FP8 (§2.4.4: it is sensitive to
 * quantisation) without saying which; MXFP8 is the OCP MX format with E4M3 elements: one
 * E8M0 scale per 32 values, X = floor(log2(max|x|)) - 8 clamped to [-127, 127] (X = 0 for
 * an all-zero block), element = round-half-even of x / 2^X onto the E4M3 grid (1 sign, 4
 * exponent bits with bias 7, 3 mantissa bits, subnormals m x 2^-9), saturating at +-448,
 * sign bit = sign bit of x.  Element x 2^X is exact in bf16 while it stays normal. */
typedef enum { CSA2_SWA_BF16 = 0, CSA2_SWA_MXFP8 = 1 } csa2_swa_format;

typedef enum {
    CSA2_INDEX_FULL = 0, /* every causally visible entry is a candidate (Full mode)     */
    CSA2_INDEX_POOL = 1  /* only the positions of the given block pool (Reindex mode)    */
} csa2_index_mode;

CSA2_API const char *csa2_status_string(csa2_status s);
CSA2_API int csa2_version(void); /* major*10000 + minor*100 + patch */

/* Bytes one global position takes in the cache of one source layer: main-KV latent of
 * d_main channels in `main_fmt` plus an MXFP4 indexer key of d_idx channels.
 * Review page, "四位缓存：890 字节究竟由什么组成": 512-channel E2M1 + E4M3/16 main KV and
 * a 128-channel MXFP4 indexer key give 256 + 32 + 64 + 4 = 356 bytes.  Returns 0 for an
 * invalid request (d not a multiple of the format's block). */
CSA2_API size_t csa2_cache_bytes_per_position(csa2_fp4_format main_fmt, int32_t d_main, int32_t d_idx);

/* ---------------------------------------------------------------------------------- */
/* csa2_quant_fp4 / csa2_dequant_fp4 -- the 4-bit cache codec (report §2.4.4).         */
/* x: rows x cols values of type xt (BF16 or F32), row stride ldx elements.  cols is a  */
/* multiple of the format's block G (32 for MXFP4, 16 for NVFP4_E4M3_16).  codes: rows  */
/* x cols/2 bytes, row stride ldc bytes; scales: rows x cols/G bytes, row stride lds    */
/* bytes.  Non-finite input sets CSA2_DEV_NONFINITE.  dequant writes y (BF16 or F32,    */
/* row stride ldy); every MXFP4 value with scale byte <= 252 and every finite           */
/* NVFP4_E4M3_16 value is exact in both types.                                          */
/* ---------------------------------------------------------------------------------- */
CSA2_API csa2_status csa2_quant_fp4(const void *x, csa2_dtype xt, int64_t rows, int64_t cols, int64_t ldx,
                           uint8_t *codes, int64_t ldc, uint8_t *scales, int64_t lds,
                           csa2_fp4_format fmt, uint32_t *d_status, csa2_stream stream);
CSA2_API csa2_status csa2_dequant_fp4(const uint8_t *codes, int64_t ldc, const uint8_t *scales,
                             int64_t lds, int64_t rows, int64_t cols, csa2_fp4_format fmt,
                             void *y, csa2_dtype yt, int64_t ldy, csa2_stream stream);

/* ---------------------------------------------------------------------------------- */
/* csa2_quant_fp8 / csa2_dequant_fp8 -- the MXFP8 (E4M3 + E8M0 per 32) SWA cache codec  */
/* (report §2.4.4: FP8 SWA KV; the format is the reading stated at csa2_swa_format).    */
/* x: rows x cols values of type xt (BF16 or F32), row stride ldx elements, cols % 32  */
/* == 0.  codes: rows x cols bytes, row stride ldc; scales: rows x cols/32 bytes, row  */
/* stride lds.  Non-finite input sets CSA2_DEV_NONFINITE.  dequant writes y (BF16 or   */
/* F32, row stride ldy): code value x 2^(scale byte - 127), exact in float32.          */
/* ---------------------------------------------------------------------------------- */
CSA2_API csa2_status csa2_quant_fp8(const void *x, csa2_dtype xt, int64_t rows, int64_t cols, int64_t ldx,
                                    uint8_t *codes, int64_t ldc, uint8_t *scales, int64_t lds,
                                    uint32_t *d_status, csa2_stream stream);
CSA2_API csa2_status csa2_dequant_fp8(const uint8_t *codes, int64_t ldc, const uint8_t *scales, int64_t lds,
                                      int64_t rows, int64_t cols, void *y, csa2_dtype yt, int64_t ldy,
                                      csa2_stream stream);

/* ---------------------------------------------------------------------------------- */
/* csa2_quant_fp4_batch -- up to CSA2_QUANT_MAX_JOBS independent csa2_quant_fp4 calls  */
/* in one launch (a decode step writes its token's main-KV row and indexer-K row).      */
/* jobs: HOST array of n_jobs (0..CSA2_QUANT_MAX_JOBS) descriptions, each with the      */
/* meaning and rules of the csa2_quant_fp4 arguments of the same names; every job uses  */
/* format fmt.  The outputs of different jobs must not overlap.  Results are those of   */
/* n_jobs separate csa2_quant_fp4 calls (one kernel when fmt is MXFP4 and every job has */
/* 16-byte aligned rows of x and 4-byte aligned rows of codes, else one launch per job).*/
/* ---------------------------------------------------------------------------------- */
#define CSA2_QUANT_MAX_JOBS 4
typedef struct {
    const void *x;        /* rows x cols values of type xt, row stride ldx elements        */
    csa2_dtype xt;        /* CSA2_BF16 or CSA2_F32                                         */
    int64_t rows, cols, ldx;
    uint8_t *codes;       /* rows x cols/2 bytes, row stride ldc                           */
    int64_t ldc;
    uint8_t *scales;      /* rows x cols/32 bytes, row stride lds                          */
    int64_t lds;
} csa2_quant_job;
CSA2_API csa2_status csa2_quant_fp4_batch(const csa2_quant_job *jobs, int32_t n_jobs, csa2_fp4_format fmt,
                                          uint32_t *d_status, csa2_stream stream);

/* ---------------------------------------------------------------------------------- */
/* csa2_rope_quant_fp4 -- the decode step's cache write with the rotary embedding fused */
/* in: report §2.4.4 quantises the main-KV cache AFTER RoPE, with the RoPE and non-RoPE */
/* channels in the same 4-bit format.  Up to CSA2_QUANT_MAX_JOBS jobs in one launch,    */
/* each with its own format and rotated width.  For job j, row r of x (bf16):           */
/*   the last rope_dim channels c0 = cols - rope_dim ... cols-1 are rotated in pairs     */
/*   (c0 + 2i, c0 + 2i + 1), i < rope_dim/2, by the caller's table row p = pos[r]:       */
/*     c = cos_sin[p * rope_dim + i], s = cos_sin[p * rope_dim + rope_dim/2 + i]         */
/*     y[c0+2i]   = RN32(RN32(a*c) - RN32(b*s)),  y[c0+2i+1] = RN32(RN32(a*s) + RN32(b*c)) */
/*   (a, b = the pair's input values; float32, one rounding per product and per sum,  */
/*   no fused multiply-add), the other channels y = x; then y (float32, not rounded to  */
/*   bf16) is quantised in format fmt exactly as csa2_quant_fp4 quantises its input.    */
/* The pages give no RoPE formula; the pairing, the table and its frequencies are the   */
/* caller's (rope_dim = 0: no rotation, pos and cos_sin unused).                        */
/* Requirements per job: x rows 16-byte aligned (x and ldx*2), codes rows 4-byte        */
/* aligned (codes and ldc), cols % G == 0 (G = 32 MXFP4, 16 NVFP4_E4M3_16), rope_dim    */
/* even and <= cols; with rope_dim > 0: pos [rows] (device) and cos_sin [n_pos,        */
/* rope_dim] float32 (device), n_pos >= 1.  A row whose pos is outside [0, n_pos) sets  */
/* CSA2_DEV_BAD_INDEX and is quantised unrotated.  Outputs of different jobs must not   */
/* overlap.                                                                            */
/* ---------------------------------------------------------------------------------- */
typedef struct {
    const uint16_t *x;       /* bf16 rows x cols, row stride ldx elements                 */
    int64_t rows, cols, ldx;
    int32_t rope_dim;        /* rotated trailing channels (0: none)                       */
    const int32_t *pos;      /* [rows] token position of each row (rope_dim > 0)          */
    const float *cos_sin;    /* [n_pos, rope_dim]: rope_dim/2 cosines, then the sines      */
    int64_t n_pos;
    uint8_t *codes;          /* rows x cols/2 bytes, row stride ldc                        */
    int64_t ldc;
    uint8_t *scales;         /* rows x cols/G bytes, row stride lds                        */
    int64_t lds;
    csa2_fp4_format fmt;
} csa2_rope_quant_job;
CSA2_API csa2_status csa2_rope_quant_fp4(const csa2_rope_quant_job *jobs, int32_t n_jobs,
                                         uint32_t *d_status, csa2_stream stream);

/* ---------------------------------------------------------------------------------- */
/* csa2_index_score -- indexer scores (report §2.3: the indexer scores main-KV entries  */
/* with indexer Q and indexer K; §2.3.2: Reindex layers score only the pool).           */
/*                                                                                    */
/* Score of a candidate position t for a query with heads h = 0..H-1 (the pages give   */
/* no formula; the head-weighted ReLU sum is the workload's definition):               */
/*   s_t = sum_h w_h * max(0, q_hat_h . k_hat_t),  q_hat = MXFP4(q_h) (quantised inside */
/*   the call, 32-value blocks, same rule as csa2_quant_fp4), w_h the exact value of    */
/*   the float32 weight.  Selections (csa2_topk / csa2_block_candidates with `exact`)   */
/*   rank positions by this exact value.  The float32 scores written out here are its  */
/*   approximation from D_h = float32 round-to-nearest-even of the exact dot and        */
/*   R_h = max(D_h, 0): a float32 fma chain s <- fma(w_h, R_h, s) over h = 0..H-1 from  */
/*   s = +0; except for a chunk of queries (FULL mode, n_q >= 8, head_dim 128,          */
/*   n_heads <= 32, n_keys <= 2^21, batch * n_keys < 2^31, q 16-byte aligned), where    */
/*   eight chains p_j run over the heads h = j mod 8 and                                */
/*   s = ((p0 + p1) + (p2 + p3)) + ((p4 + p5) + (p6 + p7)).  Either is within           */
/*   (H + 2) 2^-24 A_t + 2^-149 (sum_h |w_h| + H) of s_t, A_t = sum_h |w_h| *           */
/*   max(0, q_hat_h . k_hat_t), whenever it is finite.  A score that is not finite sets */
/*   CSA2_DEV_SCORE_RANGE.                                                              */
/* Visibility: entry j covers tokens [j*m, j*m+m-1] (no overlap, report §2.3) and a     */
/* query at token position p sees entries with (j+1)*m - 1 <= p:                       */
/*   n_vis = min(n_keys, (p + 1) / m).                                                  */
/* ---------------------------------------------------------------------------------- */
typedef struct {
    int32_t batch, n_q;        /* B, T                                                    */
    int32_t n_heads, head_dim; /* H_i (1..64), d_i (32, 64 or 128)                         */
    int32_t ratio_m;           /* compression ratio m >= 1                                 */
    int64_t n_keys;            /* N entries per sequence (< 2^31)                          */
    const uint16_t *q;         /* bf16 [B, T, H_i, d_i]                                    */
    const float *w;            /* [B, T, H_i] head weights (finite)                        */
    const uint8_t *k_codes;    /* [B, N, d_i/2]   MXFP4 indexer-K codes                    */
    const uint8_t *k_scales;   /* [B, N, d_i/32]  MXFP4 indexer-K scales                   */
    const int32_t *q_pos;      /* [B, T] absolute token positions; NULL: all N visible     */
    csa2_index_mode mode;
    const int32_t *pool_blocks; /* POOL: [B, T, n_pool_blocks] block ids, ascending and     */
    int32_t n_pool_blocks;      /* unique, padded with -1 at the end; block b covers        */
    int32_t block;              /* positions [b*block, b*block+block-1].  block: 1..32.     */
    uint32_t *group_max;        /* optional output (NULL: none), [B, T, ceil(n_cand/32)]:   */
                                /* per row, for every group of 32 consecutive candidates   */
                                /* that holds a valid one, the largest selection key of    */
                                /* its valid candidates; entries past the valid groups are */
                                /* left unwritten.  Handing it to csa2_topk spares that    */
                                /* call its first pass.  Selection key of a score s (the   */
                                /* order csa2_topk uses): 0 for NaN; with u = the bits of  */
                                /* s and -0 read as +0, u | 0x80000000 for s >= 0 and ~u   */
                                /* for s < 0 (so keys rise with the score).                */
    int64_t fresh_from;         /* 0: the scoring kernel waits for the kernel just before  */
                                /* it on the stream before it reads any input.  > 0 (FULL  */
                                /* mode): only the positions >= fresh_from of each         */
                                /* sequence may be written by that kernel (e.g. it is the  */
                                /* cache write of the decoded token): the kernel streams   */
                                /* the positions below it, and reads q, w and q_pos,       */
                                /* before its wait, which it takes only before the first   */
                                /* stage that holds a position >= fresh_from.              */
} csa2_index_args;

/* Outputs: scores [B, T, n_cand] float32, n_cand = N (FULL) or n_pool_blocks*block (POOL);
 * candidate i is position i (FULL) or pool_blocks[i/block]*block + i%block (POOL).
 * row_len [B, T] int32: the candidates 0..row_len-1 of each row are the valid ones
 * (FULL: n_vis; POOL: the pool positions that exist and are visible -- a prefix because
 * the pool is ascending).  Entries at or beyond row_len are left unwritten.  row_len is
 * required (not NULL) when the scores are to be selected with `exact`. */
/* Workspace: per-row tile counters.  Zero-fill it before its first use; every call     */
/* leaves it zero-filled again (a call that raised CSA2_DEV_TIMEOUT may not: zero it     */
/* again before reusing it).                                                            */
CSA2_API size_t csa2_index_score_workspace_size(const csa2_index_args *a);
CSA2_API csa2_status csa2_index_score(const csa2_index_args *a, float *scores, int32_t *row_len,
                             void *ws, size_t ws_bytes, uint32_t *d_status, csa2_stream stream);

/* ---------------------------------------------------------------------------------- */
/* csa2_topk -- Top-K selection (report §2.3: Top-K entries per query; §4.2.1: K=512).  */
/* For each of `rows` rows of n candidates: the k candidates with the largest scores,   */
/* ties broken by the lower candidate index.  Only candidates 0..row_len[r]-1 compete   */
/* (row_len NULL: all n).                                                              */
/*   exact == NULL: the scores are the given floats, in float order (-0 == +0, NaN     */
/*     below every number).                                                            */
/*   exact != NULL: scores, row_len and group_max are the outputs of csa2_index_score  */
/*     called with *exact (rows = batch * n_q, n = its n_cand, row_len required), and   */
/*     the candidates are ranked by their EXACT indexer scores (see csa2_index_score).  */
/*     The float32 scores decide every candidate farther than their error bound from   */
/*     the k-th score; the candidates within it are re-scored exactly on the GPU (wide  */
/*     integers) and ordered by the exact values.  pool_blocks / block must be those of */
/*     *exact (POOL) or NULL / any (FULL); exact->q must be 16-byte aligned.  A row     */
/*     with more than CSA2_EXACT_BAND_CAP such candidates sets CSA2_DEV_BAND_LIMIT and  */
/*     follows the float32 order.                                                      */
/* idx [rows, k] int32: the selected POSITIONS in ascending order, padded with -1 when  */
/* fewer than k compete.  Position of candidate i: i, or with pool_blocks != NULL        */
/* ([rows, n/block]) pool_blocks[i/block]*block + i%block -- ascending candidates map to */
/* ascending positions, so the tie rule is the lower position.                         */
/* out_scores (nullable) [rows, k]: the float32 score of each selected entry (0 for     */
/* padding).                                                                           */
/* group_max (nullable) [rows, ceil(n/32)]: the group_max output of the csa2_index_score */
/* call that wrote these scores and row_len; when given, the call skips computing it.  */
/* (Used only while n <= 2^20; longer rows use wider groups and compute their own.)     */
/* Workspace: csa2_topk_workspace_size(rows, n, k, exact) bytes.                        */
/* ---------------------------------------------------------------------------------- */
#define CSA2_EXACT_BAND_CAP 2048
CSA2_API size_t csa2_topk_workspace_size(int64_t rows, int64_t n, int32_t k, const csa2_index_args *exact);
CSA2_API csa2_status csa2_topk(const float *scores, int64_t rows, int64_t n, const int32_t *row_len,
                      const uint32_t *group_max, const int32_t *pool_blocks, int32_t block,
                      const csa2_index_args *exact, int32_t k, int32_t *idx, float *out_scores,
                      void *ws, size_t ws_bytes, uint32_t *d_status, csa2_stream stream);

/* ---------------------------------------------------------------------------------- */
/* csa2_block_candidates -- the hierarchical sparse indexer's block pool (report §2.3.2 */
/* and Figure 5; review: block selection uses the global position scores directly).     */
/* For each row of FULL-mode scores (candidate i = position i, valid i < row_len): block */
/* b covers positions [b*block, b*block+block-1]; its score is the max of its valid     */
/* positions' scores.  block_ids [rows, nb]: the nb best blocks by (score desc, block   */
/* id asc), ascending, -1 padded (at most 2,048 blocks of 8 = 16,384 positions in the   */
/* report's configuration, §4.2.1).                                                     */
/*   exact == NULL: scores are the given floats (NaN ignored; all-NaN -> NaN).          */
/*   exact != NULL: scores and row_len are the outputs of csa2_index_score with *exact  */
/*     (FULL mode; row_len required) and a block's score is the largest EXACT score of  */
/*     its valid positions, resolved as in csa2_topk (CSA2_DEV_BAND_LIMIT likewise).    */
/* ---------------------------------------------------------------------------------- */
CSA2_API size_t csa2_block_candidates_workspace_size(int64_t rows, int64_t n, int32_t block, int32_t nb,
                                                     const csa2_index_args *exact);
CSA2_API csa2_status csa2_block_candidates(const float *scores, int64_t rows, int64_t n,
                                  const int32_t *row_len, int32_t block, int32_t nb,
                                  const csa2_index_args *exact, int32_t *block_ids, void *ws,
                                  size_t ws_bytes, uint32_t *d_status, csa2_stream stream);

/* ---------------------------------------------------------------------------------- */
/* csa2_index_topk -- the indexer and the exact Top-K in one call, with no score matrix  */
/* (report §2.3: each query keeps the Top-K of its indexer scores; report §1 / §3.2 run   */
/* the selection fused with the scoring).  Computes exactly what csa2_index_score(a)    */
/* followed by csa2_topk(scores, ..., exact = a, k) computes: idx [B, T, k] the exact    */
/* top-k positions of each query (ascending, -1 padded; in POOL mode positions through  */
/* the pool), out_scores (nullable) [B, T, k] their float32 scores (-0 is returned as   */
/* +0), row_len (nullable) [B, T] the candidates of each row.                           */
/* Where the tensor-core indexer takes the call with one query per CTA (FULL mode, head  */
/* dim 128, at most 32 heads: the decode shape), each of its CTAs keeps its scores in    */
/* shared memory and writes only a candidate list -- every score at least lo(its own    */
/* k-th), lo the exact selection's band bound -- and a second kernel selects each row    */
/* from its lists.  Other shapes run csa2_index_score into the workspace, then          */
/* csa2_topk.  a->q must be 16-byte aligned.                                            */
/* Workspace: csa2_index_topk_workspace_size(a, k) bytes, 16-byte aligned, zero-filled   */
/* before its first use (its first part holds the indexer's counters, which every call  */
/* leaves zero).  The size depends on the current device's SM count.                    */
/* ---------------------------------------------------------------------------------- */
CSA2_API size_t csa2_index_topk_workspace_size(const csa2_index_args *a, int32_t k);
CSA2_API csa2_status csa2_index_topk(const csa2_index_args *a, int32_t k, int32_t *idx, float *out_scores,
                                     int32_t *row_len, void *ws, size_t ws_bytes, uint32_t *d_status,
                                     csa2_stream stream);

/* ---------------------------------------------------------------------------------- */
/* csa2_sparse_attn -- core attention (report §2.3 and §2.3.1: every mode attends the   */
/* selected main-KV entries together with the layer's SWA KV; review: the main KV is a  */
/* latent shared by all query heads; report §3.2.2: SWA keys of a query at token i are   */
/* [max(s, i-W+1), i] for a replay starting at s).                                      */
/* SWA keys are bf16, or MXFP8 dequantised exactly (swa_fmt).                          */
/* Key set of query (b, t): the main-KV rows idx[b,t,j] for j < topk with idx >= 0      */
/* (dequantised exactly; duplicates kept; idx >= n_kv or < -1 sets CSA2_DEV_BAD_INDEX   */
/* and is ignored), then the SWA slots j whose token swa_pos0[b] + j lies in            */
/* [max(s, p-W+1, 0), p], p = q_pos[b,t], s = swa_start ? swa_start[b] : 0.            */
/* Per head h: l_j = sm_scale * q_h . k_j over d_qk dims; o_h = sum_j softmax(l)_j *     */
/* k_j[0:d_v] (V = the latent's leading d_v dims); lse_h = log sum_j exp(l_j) (natural  */
/* log).  A query with no keys gets o = 0 and lse = -inf.  fp32 accumulation.           */
/* ---------------------------------------------------------------------------------- */
typedef struct {
    int32_t batch, n_q;      /* B, T                                                      */
    int32_t n_heads;         /* H (1..128)                                                */
    int32_t d_qk, d_v;       /* d_qk % 32 == 0, d_qk <= 1024; d_v <= d_qk, d_v % 8 == 0     */
    int32_t topk;            /* entries per idx row (0..2048)                             */
    int32_t window;          /* SWA window W (>= 0)                                       */
    float sm_scale;          /* logit scale, e.g. 1/sqrt(d_qk)                            */
    int64_t n_kv;            /* main-KV entries per sequence                              */
    const uint16_t *q;       /* bf16 [B, T, H, d_qk]                                      */
    const uint8_t *kv_codes; /* [B, n_kv, d_qk/2]  main-KV codes (format kv_fmt)          */
    const uint8_t *kv_scales;/* [B, n_kv, d_qk/G]  main-KV scales, G = 32 (MXFP4) or 16   */
    const int32_t *idx;      /* [B, T, topk]                                              */
    const uint16_t *swa;     /* [B, n_swa, d_qk] bf16 (or E4M3 bytes, swa_fmt); NULL = no */
                             /* SWA keys                                                  */
    int32_t n_swa;           /* SWA slots per sequence                                    */
    const int32_t *swa_pos0; /* [B] token position of slot 0 (required with swa)          */
    const int32_t *swa_start;/* [B] replay start s, or NULL for s = 0                     */
    const int32_t *q_pos;    /* [B, T] token position of each query (required with swa)   */
    csa2_fp4_format kv_fmt;  /* main-KV format: CSA2_FMT_MXFP4 (0) or NVFP4_E4M3_16 (1)   */
    csa2_swa_format swa_fmt; /* SWA format: CSA2_SWA_BF16 (0): swa holds bf16 values;    */
                             /* CSA2_SWA_MXFP8 (1): swa holds [B, n_swa, d_qk] E4M3 codes */
                             /* (one byte each) and swa_scales their E8M0 scales          */
    const uint8_t *swa_scales; /* MXFP8: [B, n_swa, d_qk/32] scale bytes, else unused      */
} csa2_attn_args;

/* Workspace: split rows keep their partial outputs there.  Its size depends on the    */
/* arguments and on the current device (its SM count sets how finely rows are split),  */
/* so query it with that device current; 0 means ws may be NULL.                       */
CSA2_API size_t csa2_sparse_attn_workspace_size(const csa2_attn_args *a);
CSA2_API csa2_status csa2_sparse_attn(const csa2_attn_args *a, uint16_t *out, float *lse, void *ws,
                             size_t ws_bytes, uint32_t *d_status, csa2_stream stream);

/* ---------------------------------------------------------------------------------- */
/* csa2_index_score_noalloc -- csa2_index_score for callers that cannot allocate device */
/* memory.  The paper has no counterpart; this is a deployment convenience.             */
/*                                                                                    */
/* Who needs it: an inference server that splits all device memory into fixed pools at */
/* start-up and forbids later allocations, a plug-in inside a framework that owns the    */
/* allocator, or a decode loop that must not block on the allocator or risk running out */
/* of memory mid-step.  Such callers cannot provide the workspace csa2_index_score asks  */
/* for.  This call takes the same arguments minus the workspace and computes exactly    */
/* what csa2_index_score computes.                                                      */
/*                                                                                    */
/* Scratch: a file-scope __device__ array of 65,536 32-bit words (256 KB), which every  */
/* GPU that loads the library holds until the process exits.  A request whose workspace */
/* (csa2_index_score_workspace_size) exceeds 256 KB is rejected with CSA2_ERR_WORKSPACE */
/* before anything is launched (it needs two words per query row, so up to 32,768 rows  */
/* fit).  The call makes no cudaMalloc, cudaFree or other allocating call; it clears    */
/* the scratch it uses with cudaMemsetAsync on `stream`.                                */
/*                                                                                    */
/* The first call on a device (with that device current) looks up the array's device   */
/* address with cudaGetSymbolAddress and caches it for the life of the process, keyed   */
/* by device ordinal; make that first call before any stream capture on that device.   */
/* The cached address belongs to the device's primary context: it does not survive a   */
/* cudaDeviceReset, and a call with another context current must not be made.  All     */
/* calls on a device share the one array and it keeps the last call's contents: calls  */
/* whose GPU work overlaps (concurrent streams) race on it, so serialise them.          */
/* ---------------------------------------------------------------------------------- */
CSA2_API csa2_status csa2_index_score_noalloc(const csa2_index_args *a, float *scores,
                                              int32_t *row_len, uint32_t *d_status,
                                              csa2_stream stream);

/* ---------------------------------------------------------------------------------- */
/* csa2_selftest_bounded_wait -- failure-detection self-test.  The pages have no        */
/* counterpart; it checks a property of this library.                                 */
/*                                                                                    */
/* Every device wait of the library's kernels (an mbarrier phase completed by a copy, */
/* an MMA commit or another warp) is bounded: after its poll limit it gives up, the     */
/* kernel ORs CSA2_DEV_TIMEOUT into *d_status and returns, so a lost arrival ends the   */
/* kernel instead of hanging the GPU, and the context stays usable.  This call launches */
/* one CTA whose threads wait, through the same routine with a limit of `polls` polls   */
/* (1 .. 2^20; each poll may suspend the thread for a short, hardware-defined time),    */
/* on an mbarrier that nothing ever arrives on; it must leave CSA2_DEV_TIMEOUT in       */
/* *d_status (device memory, required).  Nothing else is read or written.              */
/* ---------------------------------------------------------------------------------- */
CSA2_API csa2_status csa2_selftest_bounded_wait(uint32_t polls, uint32_t *d_status, csa2_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* CSA2_H */
