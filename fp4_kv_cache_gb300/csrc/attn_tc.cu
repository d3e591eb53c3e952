// attn_tc.cu -- tensor-core CSA2 core attention (csa2_sparse_attn fast path, sm_103a).
//
// DeepSeek-V4.1-Flash report (aipaper.jasonlin.tech) §2.3 / §2.3.1: each query attends its
// selected main-KV entries (dequantised from FP4, §2.4.4) together with the layer's SWA
// window; review page (papers.chlience.com, CSA2 section): the latent is shared by all
// query heads, so K = the whole latent and V = its leading d_v dims.
//
// Orientation: keys are the MMA M dimension.  For a tile of 128 key slots:
//   S^T [128 keys x 64 heads]  = K [keys x 576] . Q^T          (kind::f16, bf16 in, f32 acc)
//   O^T [512 dims x 64 heads] += V^T [dims x keys] . P^T        (P = softmax numerators)
// The dequantised key tile lives in shared memory as nine K-major 128-byte-swizzled chunks
// of 64 dims; the first eight serve as the K-major A operand of S^T and, read MN-major, as
// V^T for O^T, so the latent is never transposed.  S^T (64 columns) and O^T (4 x 64
// columns) accumulate in tensor memory.  Softmax runs with one thread per key: per-head
// maxima and sums are reduced across the 128 threads with a halving shuffle reduction.
// The softmax runs in base 2: logits are scaled by sm_scale * log2(e), so every exponential
// is one exp2f, and lse = (m + log2 l) ln 2.
// A CTA covers its share of one query row's SWA window and a contiguous span of the row's
// index tiles with an online softmax.  The SWA share comes first and runs before the wait
// for the kernel that writes the index entries (Top-K), so only the index tiles remain
// once those arrive.  When a row is split over several CTAs (one index tile each while
// the rows' tiles fit one wave), they form one thread-block cluster: (m, l) go through
// distributed shared memory, O partials through L2 (bulk-copied into the merging CTA's
// shared memory), and each CTA merges a quarter-slice of the output dims.  A tile is
// staged with coalesced reads (consecutive threads, consecutive 8-value pieces of a row);
// the next tile's rows are prefetched into L2 while the current one computes.
#include <cuda_bf16.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"
#include "tc_util.cuh"

namespace csa2 {
namespace {

constexpr int kThreads = 512;          // four warps per TMEM lane quadrant, 16 heads each
constexpr int kHT = 16;               // heads per thread in the softmax and the epilogue
constexpr int kKeys = 128;            // key slots per tile (MMA M)
constexpr int kH = 64;                // heads (MMA N; fewer heads are zero-padded)
constexpr int kDqk = 576, kDv = 512;
constexpr int kChunks = kDqk / 64;    // 9 chunks of 64 dims
constexpr int kChunkBytes = kKeys * 128;          // 16 KB: 128 keys x 64 bf16
constexpr int kQChunkBytes = kH * 128;            // 8 KB: 64 heads x 64 bf16
constexpr uint32_t kTmemCols = 512;   // S^T [0,64), O^T block m at [64 + 64m, 128 + 64m)
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMaxSplits = 7;          // CTAs (one cluster) per split row
constexpr int kPieces = kKeys * (kDqk / 8) / kThreads;   // 18 pieces of 8 values per thread and tile
static_assert(kKeys * (kDqk / 8) == kPieces * kThreads, "pieces do not divide evenly");

struct AttnTcParams {
    int32_t T, H, topk, window, n_swa, splits, tiles_per_split;
    int32_t n_itiles;       // tiles of index slots (128 each); SWA tiles are numbered after them
    float log2_scale;       // logit scale x log2(e): the softmax runs in base 2
    float *part_o;          // split rows: [rows, splits, 4 blocks, H, 128] raw O^T partials
    int64_t n_kv;
    const uint16_t *q;
    const uint8_t *kvc, *kvs;
    const int32_t *idx;
    const uint16_t *swa;    // bf16 rows, or E4M3 bytes when swa8
    const uint8_t *swa_scales;
    int32_t swa8;           // SWA in MXFP8 (E4M3 + E8M0 per 32)
    const int32_t *swa_pos0, *swa_start, *q_pos;
    uint16_t *out;
    float *lse;
    uint32_t *d_status;
};

// smem layout (dynamic, 1024-aligned): K chunks 0..7 | rope chunk / P^T | Q chunks 0..8
constexpr int kOffK = 0;
constexpr int kOffR = 8 * kChunkBytes;                    // 131072
constexpr int kOffQ = kOffR + kChunkBytes;                // 147456
constexpr int kSmemBytes = kOffQ + kChunks * kQChunkBytes; // 221184
// the merge's bulk copies (at most 6 peer blocks of 64 heads x 128 dims, float) reuse it
static_assert(6 * kH * kKeys * 4 <= kSmemBytes, "merge staging does not fit");
static_assert(kMaxSplits <= 7, "merge staging holds at most 6 peer blocks");

__device__ __forceinline__ int sw128(int row, int piece)   // byte offset of 16-byte piece
{
    return (row >> 3) * 1024 + (row & 7) * 128 + ((piece ^ (row & 7)) << 4);
}

__device__ __forceinline__ uint16_t bf16_bits(float v)    // round to nearest even
{
    uint32_t bits = __float_as_uint(v);
    bits += 0x7fffu + ((bits >> 16) & 1u);
    return (uint16_t)(bits >> 16);
}

// distributed shared memory: the same shared-memory offset in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t map_peer(uint32_t local, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v)
{
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Eight E2M1 codes (element 2i in the low nibble of byte i) -> four bf16x2 words of their
// values times sc2, on the ALUs (no table in shared memory).  The bf16 bits of a magnitude
// code c in 0..7 are looked up with byte permutes: high bytes {00,3F,3F,3F,40,40,40,40},
// low bytes {00,00,80,C0,00,40,80,C0} (0, 0.5, 1, 1.5, 2, 3, 4, 6); the code's sign bit
// is copied to bit 15 of its half with a sign-replicating permute.  The product with a
// power of two sc2 is exact while it stays normal.
__device__ __forceinline__ void e2m1x8_to_bf16(uint32_t w, __nv_bfloat162 sc2, uint32_t (&o)[4])
{
    const uint32_t mags = w & 0x77777777u, mhi = mags >> 16, w4 = w << 4;
    const uint32_t h03 = prmt(0x3F3F3F00u, 0x40404040u, mags), l03 = prmt(0xC0800000u, 0xC0804000u, mags);
    const uint32_t h47 = prmt(0x3F3F3F00u, 0x40404040u, mhi), l47 = prmt(0xC0800000u, 0xC0804000u, mhi);
    uint32_t v[4] = {prmt(l03, h03, 0x5140u), prmt(l03, h03, 0x7362u), prmt(l47, h47, 0x5140u),
                     prmt(l47, h47, 0x7362u)};
    const uint32_t sel[4] = {0xC080u, 0xD191u, 0xE2A2u, 0xF3B3u};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        v[k] ^= prmt(w4, w, sel[k]) & 0x80008000u;
        const __nv_bfloat162 x = __hmul2(*reinterpret_cast<const __nv_bfloat162 *>(&v[k]), sc2);
        o[k] = *reinterpret_cast<const uint32_t *>(&x);
    }
}

__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t f16_idesc(int a_mn)
{
    // c = f32, a = b = bf16, A major (0 K, 1 MN), B K-major, N = 64, M = 128
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)(kH >> 3) << 17) |
           ((uint32_t)(kKeys >> 4) << 24);
}

__device__ __forceinline__ void mma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}

__device__ __forceinline__ void cp_async_16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// Reduce N per-thread values (N = 16 or 32) over the 32 lanes of a warp by halving: each
// exchange sends half the values and keeps the other half, so afterwards lane L holds the
// reduction of value index L N / 32 (for N = 16 lanes 2i and 2i + 1 both hold value i).
template <bool MAX, int N>
__device__ __forceinline__ float warp_halving_reduce(float (&v)[N], int lane)
{
    static_assert(N == 16 || N == 32, "16 or 32 values");
    constexpr int kSteps = N == 32 ? 5 : 4;
#pragma unroll
    for (int st = 0; st < kSteps; ++st) {
        const int o = 16 >> st, n = N >> st;
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = upper ? v[i] : v[i + n / 2];
            const float keep = upper ? v[i + n / 2] : v[i];
            const float recv = __shfl_xor_sync(0xffffffffu, send, o);
            v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
        }
    }
    if (N == 16) {
        const float recv = __shfl_xor_sync(0xffffffffu, v[0], 1);
        v[0] = MAX ? fmaxf(v[0], recv) : v[0] + recv;
    }
    return v[0];
}

// NV: the main KV holds E2M1 codes with one E4M3 scale per 16 values (report §2.4.4)
// instead of one E8M0 scale per 32; only the gather and the dequantisation differ.
template <bool NV>
__global__ void __launch_bounds__(kThreads, 1) sparse_attn_tc_kernel(const AttnTcParams P)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ float s_red[4][kH];
    __shared__ float s_m[kH], s_l[kH], s_corr[kH];
    __shared__ uint64_t s_bar;
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ float s_mlx[kMaxSplits][2][kH];   // split row: every rank's (m, l) per head
    __shared__ float s_fac[kMaxSplits][kH];      // split row: e^(m_s - M)
    __shared__ int64_t s_src[kKeys];             // the tile's source rows (see slot_src)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t row = blockIdx.y;
    const int split = blockIdx.x;
    const int64_t b = row / P.T;
    const int H = P.H;
    const int quad = warp & 3, hh0 = kHT * (warp >> 2);  // TMEM lane quadrant, first head
    const int key_row = 32 * quad + lane;                 // this thread's key / dim row
    const int t_begin = split * P.tiles_per_split;
    // index entry of slot `key_row` of an index tile (0 past the entries and for SWA tiles)
    auto slot_id = [&](int tile) -> int32_t {
        const int64_t sl = (int64_t)tile * kKeys + key_row;
        return tile < P.n_itiles && sl < P.topk ? P.idx[row * P.topk + sl] : 0;
    };
    if (tid == 0) {
        tc::mbar_init(&s_bar, 1);
        tc::fence_mbar_init();
        s_abort = 0;
    }
    if (tid < kH) { s_m[tid] = -INFINITY; s_l[tid] = 0.0f; }
    if (warp == 0) {
        tc::tmem_alloc(&s_tmem, kTmemCols);
        tc::tmem_relinquish();
    }
    // Q -> nine K-major chunks (rows = heads), zero rows for heads >= H, and the SWA window
    // bounds: both before the wait for the previous kernel, since only the index entries
    // come from it (the Top-K of this step); the query, its position and the SWA rows are
    // complete before that kernel starts (see csa2_sparse_attn).
    for (int e = tid; e < kH * kChunks * 8; e += kThreads) {
        const int h = e / (kChunks * 8), rem = e % (kChunks * 8), c = rem >> 3, p = rem & 7;
        uint8_t *dst = sm + kOffQ + c * kQChunkBytes + sw128(h, p);
        if (h < H) cp_async_16(dst, P.q + ((row * H + h) * (int64_t)kDqk + c * 64 + p * 8));
        else *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
    }

    // this query's key slots: idx entries, then its SWA window [max(s, p-W+1, 0), p]
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
    // This CTA's tiles, in order: its share of the SWA window -- slots [sw_lo, sw_hi), an
    // equal part for each of the row's CTAs -- which needs nothing from the kernel before, so
    // it runs before the dependency wait (while Top-K still works, and with every CTA's code
    // path warmed up by the time the index entries arrive), then its index tiles
    // [t_begin, t_begin + tiles_per_split).
    const int64_t sw_share = (n_sw + P.splits - 1) / P.splits;
    const int64_t sw_lo = split * sw_share < n_sw ? split * sw_share : n_sw;
    const int64_t sw_hi = sw_lo + sw_share < n_sw ? sw_lo + sw_share : n_sw;
    const int n_sw_t = (int)((sw_hi - sw_lo + kKeys - 1) / kKeys);
    const int n_it = max(0, min(t_begin + P.tiles_per_split, P.n_itiles) - t_begin);
    const int n_v = n_sw_t + n_it;
    auto gtile = [&](int v) -> int { return v < n_sw_t ? P.n_itiles + v : t_begin + (v - n_sw_t); };
    bool waited = false;
    auto wait_prev = [&]() {
        if (!waited) {
            pdl_wait();
            pdl_allow_dependents();
            waited = true;
        }
    };
    __syncthreads();
    const uint32_t tmem = s_tmem;
    uint32_t phase = 0;
    bool any_o = false;

    // Key slot `key_row` of a tile: an index tile's entry, or an SWA tile's slot of the
    // window.  Returns the main-KV row (>= 0), -(SWA slot + 2), or -1 for an empty slot.
    auto slot_src = [&](int tile, int32_t id) -> int64_t {
        if (tile < P.n_itiles) {
            const int64_t sl = (int64_t)tile * kKeys + key_row;
            if (sl >= P.topk) return -1;
            if (id >= 0 && id < P.n_kv) return id;
            if (id != -1) dev_flag(P.d_status, CSA2_DEV_BAD_INDEX);
            return -1;
        }
        const int64_t sl = sw_lo + (int64_t)(tile - P.n_itiles) * kKeys + key_row;
        return sl < sw_hi ? -(j0 + sl + 2) : -1;
    };
    // Staging: thread t < 128 resolves key slot t of the tile to its source row (s_src).
    // Main-KV tiles then go to the threads as 16-value half blocks (8 code bytes, one scale)
    // hb = t + 512 k, k < 9: consecutive threads take consecutive half blocks of a row, so a
    // warp's reads cover one or two rows' contiguous bytes.  A half block decodes to two
    // 16-byte pieces of one chunk row, written in the order given by the chunk's parity,
    // so the eight threads of a store phase (two chunks, four half blocks each) hit eight
    // different bank groups.  SWA tiles go by 8-value pieces p = t + 512 k, k < 18.  The
    // next tile's rows are prefetched into L2 while the current one computes.
    const int64_t kv_row0 = b * P.n_kv, swa_row0 = b * P.n_swa;
    auto piece_dst = [&](int r, int q) -> uint8_t * {
        const int c = q >> 3;
        return sm + (c < 8 ? kOffK + c * kChunkBytes : kOffR) + sw128(r, q & 7);
    };
    auto stage_fp4 = [&]() {
        constexpr int kHalves = kKeys * (kDqk / 16) / kThreads;      // 9 half blocks per thread
        uint2 cw[kHalves];
        uint32_t sc[kHalves], ok = 0;
#pragma unroll
        for (int k = 0; k < kHalves; ++k) {
            const int hb = tid + kThreads * k, r = hb / 36, hq = hb - 36 * r;
            const int64_t src = s_src[r];
            cw[k] = make_uint2(0u, 0u);
            sc[k] = 0u;
            if (src >= 0) {
                const int64_t g = kv_row0 + src;
                cw[k] = *reinterpret_cast<const uint2 *>(P.kvc + g * (kDqk / 2) + hq * 8);
                sc[k] = NV ? P.kvs[g * (kDqk / 16) + hq] : P.kvs[g * (kDqk / 32) + (hq >> 1)];
                ok |= 1u << k;
            }
        }
        uint32_t slow = 0;
#pragma unroll
        for (int k = 0; k < kHalves; ++k) {
            const int hb = tid + kThreads * k, r = hb / 36, hq = hb - 36 * r, c = hq >> 2;
            uint8_t *base = sm + (c < 8 ? kOffK + c * kChunkBytes : kOffR);
            // code value x scale in bf16 is exact: an E4M3 scale has 4 significant bits and a
            // code 2, with every product normal; an E8M0 scale in [2^-119, 2^123] keeps every
            // product normal.  Other E8M0 scales (rare) take the exact float path below.
            const bool have = (ok >> k) & 1u;
            const bool use = have && (NV || (sc[k] >= 8u && sc[k] <= 250u));
            if (have && !use) slow |= 1u << k;
            const unsigned short sbits = NV ? (unsigned short)(__float_as_uint(e4m3_value(sc[k])) >> 16)
                                            : (unsigned short)(sc[k] << 7);
            const __nv_bfloat162 sc2 = __halves2bfloat162(__ushort_as_bfloat16(sbits), __ushort_as_bfloat16(sbits));
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int w = (j + c) & 1;
                uint32_t o[4] = {0u, 0u, 0u, 0u};
                if (use) e2m1x8_to_bf16(w ? cw[k].y : cw[k].x, sc2, o);
                *reinterpret_cast<uint4 *>(base + sw128(r, 2 * (hq & 3) + w)) = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
        if (slow) {
            // exact float products rounded to bf16 once, the half block's codes read again
#pragma unroll 1
            for (int k = 0; k < kHalves; ++k) {
                if (!((slow >> k) & 1u)) continue;
                const int hb = tid + kThreads * k, r = hb / 36, hq = hb - 36 * r, c = hq >> 2;
                uint8_t *base = sm + (c < 8 ? kOffK + c * kChunkBytes : kOffR);
                const int64_t g = kv_row0 + s_src[r];
                const uint8_t *codes = P.kvc + g * (kDqk / 2) + hq * 8;
                const float sf = e8m0_value(P.kvs[g * (kDqk / 32) + (hq >> 1)]);
#pragma unroll 1
                for (int w = 0; w < 2; ++w) {
                    const uint32_t word = *reinterpret_cast<const uint32_t *>(codes + 4 * w);
                    uint32_t o[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t byte = (word >> (8 * i)) & 0xffu;
                        float lo = e2m1_mag(byte & 7u) * sf, hi = e2m1_mag((byte >> 4) & 7u) * sf;
                        if (byte & 8u) lo = -lo;
                        if (byte & 0x80u) hi = -hi;
                        const __nv_bfloat162 bb = __floats2bfloat162_rn(lo, hi);
                        o[i] = *reinterpret_cast<const uint32_t *>(&bb);
                    }
                    *reinterpret_cast<uint4 *>(base + sw128(r, 2 * (hq & 3) + w)) = make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
        }
    };
    // bf16 SWA rows: one 16-byte cp.async per piece
    auto stage_swa16 = [&]() {
#pragma unroll 4
        for (int k = 0; k < kPieces; ++k) {
            const int p = tid + kThreads * k, r = p / 72, q = p - 72 * r;
            const int64_t src = s_src[r];
            uint8_t *dst = piece_dst(r, q);
            if (src <= -2) cp_async_16(dst, P.swa + (swa_row0 + (-src - 2)) * kDqk + q * 8);
            else *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
    };
    // MXFP8 SWA rows: 8 E4M3 code bytes and their scale byte per piece, decoded exactly (the
    // code's bits placed as a float's, times 2^120 to move the exponent bias from 7 to 127 --
    // subnormal codes included -- and times the block's 2^X)
    auto stage_swa8 = [&]() {
#pragma unroll 2
        for (int k = 0; k < kPieces; ++k) {
            const int p = tid + kThreads * k, r = p / 72, q = p - 72 * r;
            const int64_t src = s_src[r];
            uint32_t o[4] = {0u, 0u, 0u, 0u};
            if (src <= -2) {
                const int64_t srw = swa_row0 + (-src - 2);
                const uint2 cw = *reinterpret_cast<const uint2 *>(reinterpret_cast<const uint8_t *>(P.swa) + srw * kDqk + q * 8);
                const float k2 = e8m0_value(P.swa_scales[srw * (kDqk / 32) + (q >> 2)]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t x = i < 2 ? cw.x : cw.y, sh = 16 * (i & 1);
                    const uint32_t b0 = x >> sh, b1 = x >> (sh + 8);
                    const float f0 = __uint_as_float(((b0 & 0x7fu) << 20) | ((b0 & 0x80u) << 24)) * 0x1p120f * k2;
                    const float f1 = __uint_as_float(((b1 & 0x7fu) << 20) | ((b1 & 0x80u) << 24)) * 0x1p120f * k2;
                    const __nv_bfloat162 bb = __floats2bfloat162_rn(f0, f1);
                    o[i] = *reinterpret_cast<const uint32_t *>(&bb);
                }
            }
            *reinterpret_cast<uint4 *>(piece_dst(r, q)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
    };
    // the next tile's source row of key slot `key_row` into L2 (threads < 128)
    auto prefetch_row = [&](int tile, int32_t id) {
        if (tile < P.n_itiles) {
            const int64_t sl = (int64_t)tile * kKeys + key_row;
            if (sl >= P.topk || id < 0 || id >= P.n_kv) return;
            const uint8_t *c = P.kvc + (kv_row0 + id) * (kDqk / 2);
#pragma unroll
            for (int o = 0; o < kDqk / 2; o += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(c + o));
            asm volatile("prefetch.global.L2 [%0];" ::"l"(c + kDqk / 2 - 1));
            const uint8_t *s = P.kvs + (kv_row0 + id) * (NV ? kDqk / 16 : kDqk / 32);
            asm volatile("prefetch.global.L2 [%0];" ::"l"(s));
            asm volatile("prefetch.global.L2 [%0];" ::"l"(s + (NV ? kDqk / 16 : kDqk / 32) - 1));
        } else {
            const int64_t sl = sw_lo + (int64_t)(tile - P.n_itiles) * kKeys + key_row;
            if (sl >= sw_hi) return;
            const int64_t srw = swa_row0 + j0 + sl;
            const int row_bytes = P.swa8 ? kDqk : 2 * kDqk;
            const uint8_t *c = reinterpret_cast<const uint8_t *>(P.swa) + srw * row_bytes;
#pragma unroll 1
            for (int o = 0; o < row_bytes; o += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(c + o));
            asm volatile("prefetch.global.L2 [%0];" ::"l"(c + row_bytes - 1));
            if (P.swa8) asm volatile("prefetch.global.L2 [%0];" ::"l"(P.swa_scales + srw * (kDqk / 32)));
        }
    };
    int32_t id_cur = 0;      // index entry of key slot key_row of the current tile (threads < 128)
    bool have_id = false;
#pragma unroll 1
    for (int v = 0; v < n_v; ++v) {
        const int tile = gtile(v);
        if (tile < P.n_itiles) {
            wait_prev();
            if (!have_id && tid < kKeys) id_cur = slot_id(tile);
        }
        // the next tile's index entries are read a tile ahead (once the wait is behind)
        const int tn = v + 1 < n_v ? gtile(v + 1) : -1;
        const bool nx_idx = tn >= 0 && tn < P.n_itiles && waited;
        const int32_t id_nx = nx_idx && tid < kKeys ? slot_id(tn) : 0;
        if (tid < kKeys) s_src[tid] = slot_src(tile, id_cur);
        __syncthreads();
        // ---- stage the tile's keys into the chunks
        if (tile < P.n_itiles) stage_fp4();
        else if (P.swa8) stage_swa8();
        else stage_swa16();
        if (tid < kKeys && tn >= 0 && (tn >= P.n_itiles || nx_idx)) prefetch_row(tn, id_nx);
        id_cur = id_nx;
        have_id = nx_idx;
        const bool valid = s_src[key_row] != -1;
        cp_async_wait_all();
        tc::fence_proxy_async_smem();
        __syncthreads();
        // ---- S^T = K . Q^T
        if (tid == 0) {
            tc::tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < kChunks; ++c) {
                const uint32_t a0 = tc::smem_u32(sm + (c < 8 ? kOffK + c * kChunkBytes : kOffR));
                const uint32_t b0 = tc::smem_u32(sm + kOffQ + c * kQChunkBytes);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_f16(tmem, tc::smem_desc(a0 + kk * 32, 16, 1024, tc::kSwizzle128B),
                            tc::smem_desc(b0 + kk * 32, 16, 1024, tc::kSwizzle128B), f16_idesc(0),
                            (c | kk) != 0);
            }
            tc::tc_commit(&s_bar);
        }
        __syncwarp();
        if (__syncthreads_or(!tc::mbar_wait(&s_bar, phase, &s_abort))) { s_abort = 1; break; }
        phase ^= 1u;
        tc::tc_fence_after();
        // ---- softmax numerators: thread = (key row, 16 heads)
        float l[kHT];
        {
            uint32_t r[kHT];
            tc::tc_ld_32x32b_x16(tmem + ((uint32_t)(quad * 32) << 16) + hh0, r);
            tc::tc_wait_ld();
#pragma unroll
            for (int j = 0; j < kHT; ++j)
                l[j] = (valid && hh0 + j < H) ? __uint_as_float(r[j]) * P.log2_scale : -INFINITY;
        }
        {
            float v[kHT];
#pragma unroll
            for (int j = 0; j < kHT; ++j) v[j] = l[j];
            const float red = warp_halving_reduce<true, kHT>(v, lane);
            if ((lane & 1) == 0) s_red[quad][hh0 + (lane >> 1)] = red;
        }
        __syncthreads();
        if (tid < kH) {
            const float tmax = fmaxf(fmaxf(s_red[0][tid], s_red[1][tid]), fmaxf(s_red[2][tid], s_red[3][tid]));
            const float m_old = s_m[tid];
            const float m_new = fmaxf(m_old, tmax);
            s_corr[tid] = (m_old == -INFINITY) ? 0.0f : exp2f(m_old - m_new);
            s_m[tid] = m_new;
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kHT; ++j) l[j] = (l[j] == -INFINITY) ? 0.0f : exp2f(l[j] - s_m[hh0 + j]);
        {
            float v[kHT];
#pragma unroll
            for (int j = 0; j < kHT; ++j) v[j] = l[j];
            const float red = warp_halving_reduce<false, kHT>(v, lane);
            if ((lane & 1) == 0) s_red[quad][hh0 + (lane >> 1)] = red;
        }
        // ---- P^T (bf16) into the rope-chunk buffer: [64 heads x 128 keys], two 64-key halves
        {
            uint8_t *pbase = sm + kOffR + (key_row >> 6) * kQChunkBytes;
            const int col = key_row & 63;
            const bool odd = (lane & 1) != 0;
#pragma unroll
            for (int i = 0; i < kHT / 2; ++i) {
                // even lanes store heads hh0..hh0+7 for keys (row, row+1); odd lanes heads
                // hh0+8..hh0+15 for keys (row-1, row)
                const float mine = odd ? l[kHT / 2 + i] : l[i];
                const float send = odd ? l[i] : l[kHT / 2 + i];
                const float other = __shfl_xor_sync(0xffffffffu, send, 1);
                const int h = hh0 + (odd ? kHT / 2 + i : i);
                const int c0 = odd ? col - 1 : col;
                const __nv_bfloat162 pr = odd ? __floats2bfloat162_rn(other, mine)
                                              : __floats2bfloat162_rn(mine, other);
                *reinterpret_cast<__nv_bfloat162 *>(pbase + sw128(h, c0 >> 3) + (c0 & 7) * 2) = pr;
            }
        }
        __syncthreads();
        if (tid < kH) {
            const float tsum = s_red[0][tid] + s_red[1][tid] + s_red[2][tid] + s_red[3][tid];
            s_l[tid] = s_l[tid] * s_corr[tid] + tsum;
        }
        // ---- rescale the running O^T by the per-head correction (thread = dim row, 16 heads)
        if (any_o) {
#pragma unroll 1
            for (int m = 0; m < 4; ++m) {
                uint32_t r[kHT];
                const uint32_t ta = tmem + ((uint32_t)(quad * 32) << 16) + 64 + 64 * m + hh0;
                tc::tc_ld_32x32b_x16(ta, r);
                tc::tc_wait_ld();
#pragma unroll
                for (int j = 0; j < kHT; ++j)
                    r[j] = __float_as_uint(__uint_as_float(r[j]) * s_corr[hh0 + j]);
                tc::tc_st_32x32b_x16(ta, r);
            }
            tc::tc_wait_st();
        }
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();
        __syncthreads();
        // ---- O^T += V^T . P^T  (A = key chunks read MN-major, B = P^T K-major)
        if (tid == 0) {
            tc::tc_fence_after();
#pragma unroll 1
            for (int m = 0; m < 4; ++m) {
                const uint32_t a0 = tc::smem_u32(sm + kOffK + (2 * m) * kChunkBytes);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t b0 = tc::smem_u32(sm + kOffR + (kk >> 2) * kQChunkBytes) + (kk & 3) * 32;
                    mma_f16(tmem + 64 + 64 * m,
                            tc::smem_desc(a0 + kk * 2048, kChunkBytes, 1024, tc::kSwizzle128B),
                            tc::smem_desc(b0, 16, 1024, tc::kSwizzle128B), f16_idesc(1),
                            (any_o || kk > 0) ? 1u : 0u);
                }
            }
            tc::tc_commit(&s_bar);
        }
        __syncwarp();
        if (__syncthreads_or(!tc::mbar_wait(&s_bar, phase, &s_abort))) { s_abort = 1; break; }
        phase ^= 1u;
        tc::tc_fence_after();
        any_o = true;
        __syncthreads();
    }

    wait_prev();             // a CTA with SWA tiles only has not waited yet
    // ---- epilogue: thread = (dim row of each O^T block, its 16 heads)
    const uint32_t lane_t = tmem + ((uint32_t)(quad * 32) << 16);
    if (P.splits == 1) {
        if (tid < kH) s_corr[tid] = s_l[tid] > 0.0f ? 1.0f / s_l[tid] : 0.0f;   // 1/l per head
        __syncthreads();
#pragma unroll 1
        for (int m = 0; m < 4; ++m) {
            const int d = 128 * m + key_row;
            uint32_t r[kHT];
            if (any_o) {
                tc::tc_ld_32x32b_x16(lane_t + 64 + 64 * m + hh0, r);
                tc::tc_wait_ld();
            } else {
#pragma unroll
                for (int j = 0; j < kHT; ++j) r[j] = 0u;
            }
#pragma unroll
            for (int j = 0; j < kHT; ++j)
                if (hh0 + j < H)
                    P.out[(row * H + hh0 + j) * (int64_t)kDv + d] = bf16_bits(__uint_as_float(r[j]) * s_corr[hh0 + j]);
        }
        if (tid < H && P.lse) P.lse[row * H + tid] = s_l[tid] > 0.0f ? (s_m[tid] + log2f(s_l[tid])) * kLn2 : -INFINITY;
    } else {
        // Split row: the row's CTAs form one cluster (rank = split).  Each publishes (m, l)
        // to every rank through distributed shared memory and its raw O^T blocks to the
        // workspace ([row][split][block][head][128 dims]); after one cluster barrier, O^T
        // block m is merged by rank m % S from its own copy (still in tensor memory) and
        // the other ranks' copies, bulk-copied from L2 into its shared memory:
        //   o = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s,  lse = (M + log2 l) ln 2
        const int S = P.splits;
        const int64_t blk_floats = (int64_t)H * kKeys;                 // one block of a rank
        if (tid < kH) {
            const uint32_t lm = tc::smem_u32(&s_mlx[split][0][tid]), ll = tc::smem_u32(&s_mlx[split][1][tid]);
#pragma unroll 1
            for (int c = 0; c < S; ++c) {
                st_cluster_f32(map_peer(lm, (uint32_t)c), s_m[tid]);
                st_cluster_f32(map_peer(ll, (uint32_t)c), s_l[tid]);
            }
        }
#pragma unroll 1
        for (int m = 0; m < 4; ++m) {
            if (m % S == split) continue;
            float *dst = P.part_o + ((row * S + split) * 4 + m) * blk_floats + key_row;
            uint32_t r[kHT];
            if (any_o) {                  // one load of the thread's columns, one wait
                tc::tc_ld_32x32b_x16(lane_t + 64 + 64 * m + hh0, r);
                tc::tc_wait_ld();
            } else {
#pragma unroll
                for (int j = 0; j < kHT; ++j) r[j] = 0u;
            }
#pragma unroll
            for (int j = 0; j < kHT; ++j)
                if (hh0 + j < H) dst[(hh0 + j) * kKeys] = __uint_as_float(r[j]);
        }
        __threadfence();
        tc::tc_fence_before();
        cluster_sync();                   // (m, l) and partials visible to the whole cluster
        tc::tc_fence_after();
        const int n_own = (4 - split + S - 1) / S;                       // blocks m = split + kS
        // The peers' copies of the owned blocks come into shared memory with one bulk copy
        // each (the tiles' buffers are free now), slot k (S - 1) + (peer rank, this one skipped).
        const uint32_t blk_bytes = (uint32_t)blk_floats * 4u;
        const uint32_t n_in = (uint32_t)(n_own * (S - 1));
        if (tid == 0 && n_in > 0) {
            tc::mbar_arrive_expect_tx(&s_bar, n_in * blk_bytes);
            uint32_t slot = 0;
#pragma unroll 1
            for (int k = 0; k < n_own; ++k)
#pragma unroll 1
                for (int sp = 0; sp < S; ++sp)
                    if (sp != split)
                        tc::bulk_load(sm + (slot++) * blk_bytes,
                                      P.part_o + ((row * S + sp) * 4 + split + k * S) * blk_floats, blk_bytes, &s_bar);
        }
        if (tid < kH) {
            float M = -INFINITY;
#pragma unroll 1
            for (int sp = 0; sp < S; ++sp) M = fmaxf(M, s_mlx[sp][0][tid]);
            float L = 0.0f;
#pragma unroll 1
            for (int sp = 0; sp < S; ++sp) {
                const float ms = s_mlx[sp][0][tid];
                const float e = ms == -INFINITY ? 0.0f : exp2f(ms - M);
                s_fac[sp][tid] = e;
                if (ms != -INFINITY) L += e * s_mlx[sp][1][tid];
            }
            s_corr[tid] = L > 0.0f ? 1.0f / L : 0.0f;                 // 1/l per head
            if (split == 0 && tid < H && P.lse) P.lse[row * H + tid] = L > 0.0f ? (M + log2f(L)) * kLn2 : -INFINITY;
        }
        bool have = true;
        if (n_in > 0) {
            if (__syncthreads_or(!tc::mbar_wait(&s_bar, phase, &s_abort))) {
                s_abort = 1;
                tc::mbar_wait_bounded(&s_bar, phase);   // the copies in flight land before exit
                have = false;
            }
            phase ^= 1u;
        } else {
            __syncthreads();
        }
        const float *peer = reinterpret_cast<const float *>(sm) + key_row;
#pragma unroll 1
        for (int k = 0; have && k < n_own; ++k) {
            const int m = split + k * S, d = 128 * m + key_row;
            uint32_t own[kHT];
            if (any_o) {
                tc::tc_ld_32x32b_x16(lane_t + 64 + 64 * m + hh0, own);
                tc::tc_wait_ld();
            } else {
#pragma unroll
                for (int j = 0; j < kHT; ++j) own[j] = 0u;
            }
            float acc[kHT];
#pragma unroll
            for (int j = 0; j < kHT; ++j) acc[j] = 0.0f;
#pragma unroll 1
            for (int sp = 0; sp < S; ++sp) {
                const float *src = peer + (int64_t)(k * (S - 1) + (sp < split ? sp : sp - 1)) * blk_floats;
#pragma unroll
                for (int j = 0; j < kHT; ++j)
                    acc[j] += s_fac[sp][hh0 + j] * (sp == split ? __uint_as_float(own[j])
                                                                : hh0 + j < H ? src[(hh0 + j) * kKeys] : 0.0f);
            }
#pragma unroll
            for (int j = 0; j < kHT; ++j)
                if (hh0 + j < H) P.out[(row * H + hh0 + j) * (int64_t)kDv + d] = bf16_bits(acc[j] * s_corr[hh0 + j]);
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
    if (tid == 0 && s_abort) dev_flag(P.d_status, CSA2_DEV_TIMEOUT);
}

// Index tiles per CTA and CTAs (one cluster) per row: one index tile per CTA while the rows'
// index tiles fit one wave of the GPU's SMs, at most kMaxSplits CTAs a row; the row's SWA
// window is shared out evenly among its CTAs, ahead of their index tiles.
void attn_tc_split(const csa2_attn_args &a, int &splits, int &tiles_per_split, int &n_itiles)
{
    const int64_t rows = (int64_t)a.batch * a.n_q;
    n_itiles = (int)((a.topk + kKeys - 1) / kKeys);
    if (n_itiles == 0) {
        splits = 1;
        tiles_per_split = 0;
        return;
    }
    const int64_t sms = device_sm_count();
    int64_t per = (n_itiles * rows + sms - 1) / sms;     // index tiles per CTA to fill one wave
    if (per < 1) per = 1;
    if (per * kMaxSplits < n_itiles) per = (n_itiles + kMaxSplits - 1) / kMaxSplits;   // one cluster per row
    if (per > n_itiles) per = n_itiles;
    tiles_per_split = (int)per;
    splits = (int)((n_itiles + per - 1) / per);
}

} // namespace

bool attn_tc_eligible(const csa2_attn_args &a)
{
    return a.d_qk == kDqk && a.d_v == kDv && a.n_heads <= kH && ((uintptr_t)a.q & 15) == 0 &&
           (!a.swa || ((uintptr_t)a.swa & (a.swa_fmt == CSA2_SWA_MXFP8 ? 7 : 15)) == 0) &&
           ((uintptr_t)a.kv_codes & 15) == 0 &&
           (a.kv_fmt != CSA2_FMT_NVFP4_E4M3_16 || ((uintptr_t)a.kv_scales & 1) == 0);
}

size_t attn_tc_ws_bytes(const csa2_attn_args &a)
{
    int splits, per, nit;
    attn_tc_split(a, splits, per, nit);
    if (splits <= 1) return 0;
    return (size_t)a.batch * a.n_q * splits * a.n_heads * (size_t)kDv * sizeof(float);
}

cudaError_t launch_attn_tc(const csa2_attn_args &a, uint16_t *out, float *lse, void *ws,
                           uint32_t *d_status, cudaStream_t s)
{
    AttnTcParams P;
    P.T = a.n_q;
    P.H = a.n_heads;
    P.topk = a.topk;
    P.window = a.window;
    P.n_swa = a.swa ? a.n_swa : 0;
    P.log2_scale = a.sm_scale * 1.4426950408889634f;
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
    attn_tc_split(a, P.splits, P.tiles_per_split, P.n_itiles);
    P.part_o = static_cast<float *>(ws);
    const int64_t rows = (int64_t)a.batch * a.n_q;
    const int smem = kSmemBytes + 1024;
    const bool nv = a.kv_fmt == CSA2_FMT_NVFP4_E4M3_16;
    void (*kern)(AttnTcParams) = nv ? sparse_attn_tc_kernel<true> : sparse_attn_tc_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // a row's CTAs form one cluster
    return launch_pdl(kern, dim3((unsigned)P.splits, (unsigned)rows), dim3(kThreads),
                      (size_t)smem, s, (unsigned)P.splits, P);
}

} // namespace csa2
