// attn.cu -- CSA2 core sparse latent attention (csa2_sparse_attn), CUDA-core kernel.
//
// DeepSeek-V4.1-Flash report (aipaper.jasonlin.tech) §2.3 / §2.3.1: in every mode a query
// attends the selected main-KV entries together with the layer's SWA KV; §2.4.4: the FP4
// main-KV entries are dequantised before attention; §3.2.2: a query at token i attends
// SWA keys in [max(s, i-W+1), i].  Review page (papers.chlience.com, CSA2 section): the
// main KV is a latent shared by every query head, so V is its leading d_v dims.
//
// One CTA = one query row x 8 heads x one span of its key slots.  Keys stream through
// shared memory in tiles of 32 (gathered FP4 rows -- MXFP4 or E2M1 + E4M3/16 --
// dequantised exactly to float, then the SWA slots, bf16 or MXFP8 (report §2.4.4 keeps
// the SWA KV in FP8)), with an online softmax per head and fp32 accumulation.  When the
// rows and head groups alone would leave most SMs idle, a row's slots are split over
// several CTAs (flash-decoding style): each writes its (m, l, unnormalised output) to the
// workspace and a second small kernel merges them.
#include "common.cuh"
#include "internal.h"
#include <math.h>

namespace csa2 {
namespace {

constexpr int kThreads = 256;
constexpr int kHG = 8;    // heads per CTA (one warp each for the logits)
constexpr int kKT = 32;   // keys per tile (one lane each for the logits)

struct AttnParams {
    int32_t T, H, d_qk, d_v, topk, window, n_swa;
    int32_t splits, tiles_per_split;   // spans of key tiles per row (splits > 1: partials to ws)
    float *part;             // splits > 1: [rows, head groups, splits, kHG, d_v + 2] (m, l, acc)
    int32_t nv;              // main KV: 0 = MXFP4 (E8M0 / 32), 1 = E2M1 + E4M3 / 16
    float sm_scale;
    int64_t n_kv;
    const uint16_t *q;
    const uint8_t *kvc, *kvs;
    const int32_t *idx;
    const uint16_t *swa;     // bf16 rows, or E4M3 bytes when swa8
    const uint8_t *swa_scales;
    int32_t swa8;            // SWA in MXFP8
    const int32_t *swa_pos0, *swa_start, *q_pos;
    uint16_t *out;
    float *lse;
    uint32_t *d_status;
};

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// One 16-value chunk of a tile's key row (values 16 q .. 16 q + 15): its raw bytes are
// loaded first (every load of a thread's chunks in flight together), then widened to float.
struct KvChunk {
    uint4 a, b;              // main KV: a.x, a.y = the 8 code bytes; SWA: the 16 values' bytes
    uint32_t scale;          // the chunk's scale byte (main KV, MXFP8 SWA)
    int kind;                // 0: none (zeros), 1: main KV, 2: bf16 SWA, 3: MXFP8 SWA
};

__device__ __forceinline__ KvChunk load_chunk(const AttnParams &P, int64_t b, int64_t src, int q)
{
    KvChunk k;
    k.a = make_uint4(0u, 0u, 0u, 0u);
    k.b = k.a;
    k.scale = 0u;
    k.kind = 0;
    if (src >= 0) {
        const int64_t r = b * P.n_kv + src;
        const uint8_t *cp = P.kvc + r * (P.d_qk / 2) + q * 8;
        if ((reinterpret_cast<uintptr_t>(cp) & 7u) == 0) {
            const uint2 v = *reinterpret_cast<const uint2 *>(cp);
            k.a.x = v.x;
            k.a.y = v.y;
        } else {
            uint32_t w[2] = {0u, 0u};
#pragma unroll
            for (int i = 0; i < 8; ++i) w[i >> 2] |= (uint32_t)cp[i] << (8 * (i & 3));
            k.a.x = w[0];
            k.a.y = w[1];
        }
        k.scale = P.nv ? P.kvs[r * (P.d_qk / 16) + q] : P.kvs[r * (P.d_qk / 32) + q / 2];
        k.kind = 1;
    } else if (src <= -2) {
        const int64_t r = b * P.n_swa + (-src - 2);
        if (P.swa8) {        // 16 E4M3 bytes and the block's E8M0 scale
            const uint8_t *vp = reinterpret_cast<const uint8_t *>(P.swa) + r * P.d_qk + q * 16;
            if ((reinterpret_cast<uintptr_t>(vp) & 15u) == 0) {
                k.a = *reinterpret_cast<const uint4 *>(vp);
            } else {
                uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int i = 0; i < 16; ++i) w[i >> 2] |= (uint32_t)vp[i] << (8 * (i & 3));
                k.a = make_uint4(w[0], w[1], w[2], w[3]);
            }
            k.scale = P.swa_scales[r * (P.d_qk / 32) + q / 2];
            k.kind = 3;
        } else {             // 16 bf16
            const uint16_t *vp = P.swa + r * (int64_t)P.d_qk + q * 16;
            if ((reinterpret_cast<uintptr_t>(vp) & 15u) == 0) {
                k.a = reinterpret_cast<const uint4 *>(vp)[0];
                k.b = reinterpret_cast<const uint4 *>(vp)[1];
            } else {
                uint32_t w[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) w[i] = (uint32_t)vp[2 * i] | ((uint32_t)vp[2 * i + 1] << 16);
                k.a = make_uint4(w[0], w[1], w[2], w[3]);
                k.b = make_uint4(w[4], w[5], w[6], w[7]);
            }
            k.kind = 2;
        }
    }
    return k;
}

__device__ __forceinline__ void store_chunk(const AttnParams &P, const KvChunk &k, float *dst)
{
    if (k.kind == 1) {                   // E2M1 codes (low nibble first) times the block scale
        const float sc = P.nv ? e4m3_value(k.scale) : e8m0_value(k.scale);
        const uint32_t w[2] = {k.a.x, k.a.y};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t code = (w[i >> 3] >> (4 * (i & 7))) & 15u;
            const float v = e2m1_mag(code & 7u) * sc;
            dst[i] = (code & 8u) ? -v : v;
        }
    } else if (k.kind == 2) {
        const uint32_t w[8] = {k.a.x, k.a.y, k.a.z, k.a.w, k.b.x, k.b.y, k.b.z, k.b.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            dst[2 * i] = __uint_as_float(w[i] << 16);
            dst[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    } else if (k.kind == 3) {            // MXFP8: E4M3 value x 2^(e - 127), exact in float32
        const float sc = e8m0_value(k.scale);
        const uint32_t w[4] = {k.a.x, k.a.y, k.a.z, k.a.w};
#pragma unroll
        for (int i = 0; i < 16; ++i) dst[i] = e4m3_value((w[i >> 2] >> (8 * (i & 3))) & 255u) * sc;
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) dst[i] = 0.0f;
    }
}

template <int CPT>
__global__ void __launch_bounds__(kThreads) sparse_attn_cc_kernel(AttnParams P)
{
    extern __shared__ float smem[];
    const int ldk = P.d_qk + 1;
    float *s_k = smem;                       // [kKT][ldk]
    float *s_q = s_k + kKT * ldk;            // [kHG][d_qk]
    float *s_p = s_q + kHG * P.d_qk;         // [kHG][kKT]
    __shared__ int64_t s_src[kKT];           // >= 0: main-KV row; <= -2: SWA slot -(src+2); -1: none
    __shared__ float s_corr[kHG], s_m[kHG], s_l[kHG];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t row = blockIdx.y;
    const int64_t b = row / P.T;
    const int h0 = blockIdx.x * kHG;

    // the head group's query rows, 8 bf16 a load where the rows are 16-byte aligned
    if ((reinterpret_cast<uintptr_t>(P.q) & 15u) == 0) {
        const int n8 = P.d_qk / 8;
        for (int e = tid; e < kHG * n8; e += kThreads) {
            const int hh = e / n8, c8 = e - hh * n8;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (h0 + hh < P.H)
                v = *reinterpret_cast<const uint4 *>(P.q + (row * P.H + h0 + hh) * (int64_t)P.d_qk + c8 * 8);
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
            float *dst = s_q + hh * P.d_qk + c8 * 8;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                dst[2 * i] = __uint_as_float(w4[i] << 16);
                dst[2 * i + 1] = __uint_as_float(w4[i] & 0xffff0000u);
            }
        }
    } else {
        for (int e = tid; e < kHG * P.d_qk; e += kThreads) {
            const int hh = e / P.d_qk, c = e % P.d_qk;
            s_q[e] = (h0 + hh < P.H)
                         ? __uint_as_float((uint32_t)P.q[(row * P.H + h0 + hh) * (int64_t)P.d_qk + c] << 16)
                         : 0.0f;
        }
    }

    // SWA slots of this query: tokens [max(s, p - W + 1, 0), p] of a buffer whose slot 0
    // holds token swa_pos0
    int64_t j0 = 0, n_sw = 0;
    if (P.swa) {
        const int64_t p = P.q_pos[row];
        const int64_t s0 = P.swa_start ? (int64_t)P.swa_start[b] : 0;
        int64_t lo = p - P.window + 1;
        lo = lo < s0 ? s0 : lo;
        lo = lo < 0 ? 0 : lo;
        const int64_t pos0 = P.swa_pos0[b];
        j0 = lo - pos0 < 0 ? 0 : lo - pos0;
        int64_t j1 = p - pos0;
        j1 = j1 > P.n_swa - 1 ? P.n_swa - 1 : j1;
        n_sw = j1 >= j0 ? j1 - j0 + 1 : 0;
    }
    const int64_t n_slots = P.topk + n_sw;
    const int64_t t_lo = (int64_t)blockIdx.z * P.tiles_per_split * kKT;
    int64_t t_hi = t_lo + (int64_t)P.tiles_per_split * kKT;
    t_hi = t_hi < n_slots ? t_hi : n_slots;

    float acc[kHG][CPT];
#pragma unroll
    for (int hh = 0; hh < kHG; ++hh)
#pragma unroll
        for (int u = 0; u < CPT; ++u) acc[hh][u] = 0.0f;
    float m_run = -INFINITY, l_run = 0.0f;   // per-head state, held by the head's warp
    const int my_h = h0 + warp;
    // the query, positions and SWA range above come from inputs the kernel before does not
    // write; the indices (and the keys they select) from here on may
    pdl_wait();
    pdl_allow_dependents();

    for (int64_t t0 = t_lo; t0 < t_hi; t0 += kKT) {
        if (tid < kKT) {
            const int64_t sl = t0 + tid;
            int64_t src = -1;
            if (sl < P.topk) {
                const int32_t id = P.idx[row * P.topk + sl];
                if (id >= 0 && id < P.n_kv) src = id;
                else if (id != -1) dev_flag(P.d_status, CSA2_DEV_BAD_INDEX);
            } else if (sl < t_hi) {
                src = -(j0 + (sl - P.topk) + 2);
            }
            s_src[tid] = src;
        }
        __syncthreads();
        // gather + dequantise (main KV) or widen (SWA) the tile's keys: 16-value chunks, two
        // per thread and pass, both loaded before either is widened (d_qk = 128: one pass)
        {
            const int nch = P.d_qk / 16, nchunk = kKT * nch;
            for (int c0 = 0; c0 < nchunk; c0 += 2 * kThreads) {
                KvChunk kc[2];
                int at[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int ch = c0 + u * kThreads + tid;
                    const int j = ch / nch, q = ch - j * nch;
                    kc[u] = load_chunk(P, b, ch < nchunk ? s_src[j] : -1, q);
                    at[u] = ch < nchunk ? j * ldk + q * 16 : -1;
                }
#pragma unroll
                for (int u = 0; u < 2; ++u)
                    if (at[u] >= 0) store_chunk(P, kc[u], s_k + at[u]);
            }
        }
        __syncthreads();
        // logits: warp = head, lane = key
        {
            float l = -INFINITY;
            if (my_h < P.H && s_src[lane] != -1) {
                float dot = 0.0f;
                const float *qh = s_q + warp * P.d_qk;
                const float *kj = s_k + lane * ldk;
                for (int c = 0; c < P.d_qk; ++c) dot = fmaf(qh[c], kj[c], dot);
                l = dot * P.sm_scale;
            }
            const float m_new = fmaxf(m_run, warp_max(l));
            float p = 0.0f, corr = 1.0f;
            if (m_new != -INFINITY) {
                p = (l == -INFINITY) ? 0.0f : expf(l - m_new);
                corr = (m_run == -INFINITY) ? 0.0f : expf(m_run - m_new);
            }
            l_run = l_run * corr + warp_sum(p);
            m_run = m_new;
            s_p[warp * kKT + lane] = p;
            if (lane == 0) s_corr[warp] = corr;
        }
        __syncthreads();
        // P.V over the tile: thread owns columns tid + 256u of every head
#pragma unroll
        for (int hh = 0; hh < kHG; ++hh) {
            const float corr = s_corr[hh];
#pragma unroll
            for (int u = 0; u < CPT; ++u) acc[hh][u] *= corr;
        }
        for (int j = 0; j < kKT; ++j) {
            float v[CPT];
#pragma unroll
            for (int u = 0; u < CPT; ++u) {
                const int c = tid + kThreads * u;
                v[u] = c < P.d_v ? s_k[j * ldk + c] : 0.0f;
            }
#pragma unroll
            for (int hh = 0; hh < kHG; ++hh) {
                const float p = s_p[hh * kKT + j];
#pragma unroll
                for (int u = 0; u < CPT; ++u) acc[hh][u] = fmaf(p, v[u], acc[hh][u]);
            }
        }
        __syncthreads();
    }
    if (lane == 0) { s_m[warp] = m_run; s_l[warp] = l_run; }
    __syncthreads();
    if (P.splits > 1) {
        // this span's partial: m and l per head, then the output unnormalised (relative to m)
        float *part = P.part + (((row * gridDim.x + blockIdx.x) * P.splits + blockIdx.z) * kHG) * (int64_t)(P.d_v + 2);
#pragma unroll
        for (int hh = 0; hh < kHG; ++hh) {
            float *ph = part + hh * (int64_t)(P.d_v + 2);
            if (tid == 0) {
                ph[0] = s_m[hh];
                ph[1] = s_l[hh];
            }
#pragma unroll
            for (int u = 0; u < CPT; ++u) {
                const int c = tid + kThreads * u;
                if (c < P.d_v) ph[2 + c] = acc[hh][u];
            }
        }
        return;
    }
#pragma unroll
    for (int hh = 0; hh < kHG; ++hh) {
        const int h = h0 + hh;
        if (h >= P.H) continue;
        const float l = s_l[hh];
        const float inv = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll
        for (int u = 0; u < CPT; ++u) {
            const int c = tid + kThreads * u;
            if (c < P.d_v) {
                const float o = acc[hh][u] * inv;
                // round to nearest even bf16
                uint32_t bits = __float_as_uint(o);
                bits += 0x7fffu + ((bits >> 16) & 1u);
                P.out[(row * P.H + h) * (int64_t)P.d_v + c] = (uint16_t)(bits >> 16);
            }
        }
        if (P.lse && tid == 0) P.lse[row * P.H + h] = l > 0.0f ? s_m[hh] + logf(l) : -INFINITY;
    }
}

// Merge of a split row, one CTA per (head group, row) and one warp per head (at most
// 2 x 152 spans a row: the weights take at most 9.7 KB of shared memory):
//   o = sum_s e^(m_s - M) acc_s / sum_s e^(m_s - M) l_s,  lse = M + ln(sum_s e^(m_s - M) l_s)
template <int NC>           // output columns per lane (d_v <= 32 NC)
__global__ void __launch_bounds__(kThreads) sparse_attn_cc_merge_kernel(AttnParams P)
{
    // warp hh merges head blockIdx.x * kHG + hh: lanes take the spans for M and the sum L,
    // the spans' weights e^(m_s - M) go to shared memory, then lanes take output columns
    static_assert(kThreads == 32 * kHG, "one warp per head");
    extern __shared__ float s_e[];                         // [kHG][splits]
    const int64_t row = blockIdx.y;
    const int S = P.splits;
    const int lane = threadIdx.x & 31, hh = threadIdx.x >> 5;
    const int h = blockIdx.x * kHG + hh;
    pdl_wait();                                            // the spans' partials
    pdl_allow_dependents();
    if (h >= P.H) return;                                  // whole warps; no block barrier follows
    const int64_t stride = kHG * (int64_t)(P.d_v + 2);     // from one span's partial to the next
    const float *ph = P.part + ((row * gridDim.x + blockIdx.x) * S * kHG + hh) * (int64_t)(P.d_v + 2);
    float *se = s_e + hh * S;
    // lane z's first span's (m, l) are read once and kept (spans from 32 on are read again)
    float m0 = -INFINITY, l0 = 0.0f;
    if (lane < S) {
        m0 = ph[lane * stride];
        l0 = ph[lane * stride + 1];
    }
    float M = m0;
    for (int z = lane + 32; z < S; z += 32) M = fmaxf(M, ph[z * stride]);
    M = warp_max(M);
    float L = 0.0f;
    for (int z = lane; z < S; z += 32) {
        const float m = z == lane ? m0 : ph[z * stride];
        const float l = z == lane ? l0 : ph[z * stride + 1];
        const float e = m != -INFINITY ? expf(m - M) : 0.0f;   // a span without keys adds nothing
        se[z] = e;
        if (e != 0.0f) L += e * l;
    }
    L = warp_sum(L);
    __syncwarp();
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    // lane columns c = lane + 32 k; CH spans' values of all of them loaded together (CH x NC
    // registers), then each column's chain advances over those spans in order
    constexpr int CH = NC <= 4 ? 8 : (NC <= 16 ? 4 : 2);
    float o[NC];
#pragma unroll
    for (int k = 0; k < NC; ++k) o[k] = 0.0f;
    for (int z0 = 0; z0 < S; z0 += CH) {
        float v[CH][NC], e[CH];
#pragma unroll
        for (int u = 0; u < CH; ++u) {
            const int z = z0 + u;
            e[u] = z < S ? se[z] : 0.0f;
#pragma unroll
            for (int k = 0; k < NC; ++k) {
                const int c = lane + 32 * k;
                v[u][k] = (z < S && c < P.d_v) ? ph[z * stride + 2 + c] : 0.0f;
            }
        }
#pragma unroll
        for (int u = 0; u < CH; ++u)
            if (e[u] != 0.0f) {
#pragma unroll
                for (int k = 0; k < NC; ++k) o[k] = fmaf(e[u], v[u][k], o[k]);
            }
    }
#pragma unroll
    for (int k = 0; k < NC; ++k) {
        const int c = lane + 32 * k;
        if (c >= P.d_v) break;
        uint32_t bits = __float_as_uint(o[k] * inv);       // round to nearest even bf16
        bits += 0x7fffu + ((bits >> 16) & 1u);
        P.out[(row * P.H + h) * (int64_t)P.d_v + c] = (uint16_t)(bits >> 16);
    }
    if (P.lse && lane == 0) P.lse[row * P.H + h] = L > 0.0f ? M + logf(L) : -INFINITY;
}

// Spans per row: enough CTAs for about two per SM, at most one per 32-key tile of the
// row's largest slot count (its Top-K entries and a full SWA window).
void cc_split(const csa2_attn_args &a, int &splits, int &per)
{
    const int64_t rows = (int64_t)a.batch * a.n_q, hg = (a.n_heads + kHG - 1) / kHG;
    int64_t sw = a.swa ? (a.window < a.n_swa ? a.window : a.n_swa) : 0;
    const int64_t tiles = (a.topk + sw + kKT - 1) / kKT;
    int64_t want = (2 * device_sm_count() + rows * hg - 1) / (rows * hg > 0 ? rows * hg : 1);
    if (want > tiles) want = tiles;
    if (want < 1) want = 1;
    const int64_t p = (tiles + want - 1) / want;
    per = (int)(p > 0 ? p : 1);
    splits = (int)(tiles > 0 ? (tiles + per - 1) / per : 1);
    if (splits < 1) splits = 1;
}

template <int CPT>
cudaError_t launch_cc(const AttnParams &P, int64_t rows, cudaStream_t s)
{
    const size_t smem = sizeof(float) * ((size_t)kKT * (P.d_qk + 1) + (size_t)kHG * P.d_qk + kHG * kKT);
    cudaError_t e = cudaFuncSetAttribute(sparse_attn_cc_kernel<CPT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((P.H + kHG - 1) / kHG), (unsigned)rows, (unsigned)P.splits);
    e = launch_pdl(sparse_attn_cc_kernel<CPT>, grid, dim3(kThreads), smem, s, 1, P);
    if (e != cudaSuccess || P.splits <= 1) return e;
    const dim3 mg(grid.x, grid.y);
    const size_t msm = sizeof(float) * kHG * P.splits;
    const int nc = (P.d_v + 31) / 32;                    // d_v <= d_qk <= 1024
    if (nc <= 1) return launch_pdl(sparse_attn_cc_merge_kernel<1>, mg, dim3(kThreads), msm, s, 1, P);
    if (nc <= 2) return launch_pdl(sparse_attn_cc_merge_kernel<2>, mg, dim3(kThreads), msm, s, 1, P);
    if (nc <= 4) return launch_pdl(sparse_attn_cc_merge_kernel<4>, mg, dim3(kThreads), msm, s, 1, P);
    if (nc <= 8) return launch_pdl(sparse_attn_cc_merge_kernel<8>, mg, dim3(kThreads), msm, s, 1, P);
    if (nc <= 16) return launch_pdl(sparse_attn_cc_merge_kernel<16>, mg, dim3(kThreads), msm, s, 1, P);
    return launch_pdl(sparse_attn_cc_merge_kernel<32>, mg, dim3(kThreads), msm, s, 1, P);
}

} // namespace

size_t sparse_attn_ws_bytes(const csa2_attn_args &a)
{
    if (attn_tc_eligible(a)) return attn_tc_ws_bytes(a);
    int splits, per;
    cc_split(a, splits, per);
    if (splits <= 1) return 0;
    const int64_t rows = (int64_t)a.batch * a.n_q, hg = (a.n_heads + kHG - 1) / kHG;
    return (size_t)rows * hg * splits * kHG * (size_t)(a.d_v + 2) * sizeof(float);
}

cudaError_t launch_sparse_attn(const csa2_attn_args &a, uint16_t *out, float *lse, void *ws,
                               uint32_t *d_status, cudaStream_t s)
{
    AttnParams P;
    P.T = a.n_q;
    P.H = a.n_heads;
    P.d_qk = a.d_qk;
    P.d_v = a.d_v;
    P.topk = a.topk;
    P.window = a.window;
    P.n_swa = a.swa ? a.n_swa : 0;
    P.nv = a.kv_fmt == CSA2_FMT_NVFP4_E4M3_16 ? 1 : 0;
    P.sm_scale = a.sm_scale;
    P.n_kv = a.n_kv;
    P.q = a.q;
    P.kvc = a.kv_codes;
    P.kvs = a.kv_scales;
    P.idx = a.idx;
    P.swa = a.swa;
    P.swa_scales = a.swa_scales;
    P.swa8 = a.swa_fmt == CSA2_SWA_MXFP8 ? 1 : 0;
    P.swa_pos0 = a.swa_pos0;
    P.swa_start = a.swa_start;
    P.q_pos = a.q_pos;
    P.out = out;
    P.lse = lse;
    P.d_status = d_status;
    const int64_t rows = (int64_t)a.batch * a.n_q;
    if (rows == 0 || a.n_heads == 0) return cudaSuccess;
    if (attn_tc_eligible(a)) return launch_attn_tc(a, out, lse, ws, d_status, s);
    cc_split(a, P.splits, P.tiles_per_split);
    P.part = static_cast<float *>(ws);
    const int cpt = (a.d_v + kThreads - 1) / kThreads;
    switch (cpt <= 1 ? 1 : cpt <= 2 ? 2 : 4) {
    case 1: return launch_cc<1>(P, rows, s);
    case 2: return launch_cc<2>(P, rows, s);
    default: return launch_cc<4>(P, rows, s);
    }
}

} // namespace csa2
