// exact.cuh -- exact indexer scores for the selection kernels (topk.cu).
//
// DeepSeek-V4.1-Flash report (aipaper.jasonlin.tech) §2.3 / §2.4.4: the indexer ranks
// main-KV entries by scores of MXFP4 indexer queries and keys.  The score is
//     s = sum_h w_h * max(0, d_h),   d_h = q_hat_h . k_hat  (the exact dot),
// with w_h the exact value of the float32 weight.  The selection kernels rank by s
// exactly: float32 scores (within a proven error bound of s) decide every candidate far
// from the K-th score, and the few candidates within the bound are re-scored here with
// nothing rounded.
//
// Representation: a two's-complement integer S of kLimbs 32-bit limbs with s = S * 2^kE0.
// A product term m_w * I_b (m_w < 2^24 the weight's significand, |I_b| < 2^13 the integer
// block dot) sits at exponent e_w + Xq + Xk - 2 >= -149 - 127 - 127 - 2 = -405 and is below
// 2^(104 + 255 - 2 + 37) = 2^394, so 26 limbs from 2^-416 hold any sum of up to 256 of
// them with its sign.  A warp computes one score: lane h handles head h (and h + 32), and
// lane j < 26 owns limb j of the result, accumulating each term's 32-bit slice as a signed
// 64-bit digit; one carry pass at the end gives the limbs.
#pragma once

#include "common.cuh"

namespace csa2 {
namespace exact {

constexpr int kLimbs = 26;
constexpr int kE0 = -416;
constexpr int kMaxH = 64;
constexpr int kMaxWords = 32;          // int8x4 words of one head (head dim <= 128)

// One query row quantised to MXFP4 by the indexer's rule, as the exact pass needs it.
struct QuantQuery {
    int32_t qw[kMaxH * kMaxWords];     // twice the E2M1 values as int8x4 words, head-major
    int32_t qx[kMaxH * 4];             // block exponents X (scale byte - 127)
    int32_t q1[kMaxH * 4];             // sum of |twice value| over each block
    int32_t m_w[kMaxH];                // w_h = m_w * 2^e_w exactly
    int32_t e_w[kMaxH];
    float w[kMaxH];
};

// Quantise query row `q` ([H, d] bf16 bits, 16-byte aligned) into Q with the block exponent
// and rounding of csa2_quant_fp4 and the indexer kernels: thread t loads 8 values (one
// 16-byte load; H * d / 8 <= blockDim threads), the 4 threads of a 32-value block agree on
// its exponent by shuffles.  All threads of the block call; ends with a barrier.
__device__ __forceinline__ void quantise_query(QuantQuery &Q, const uint16_t *q, const float *w, int H, int d)
{
    const int t = threadIdx.x;
    const int nb = d / 32, nw = d / 4;
    const int nchunks = H * d / 8;
    uint4 raw = make_uint4(0, 0, 0, 0);
    if (t < nchunks) raw = reinterpret_cast<const uint4 *>(q)[t];
    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
    float v[8];
    uint32_t amax = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        v[2 * k] = __uint_as_float(w4[k] << 16);
        v[2 * k + 1] = __uint_as_float(w4[k] & 0xffff0000u);
        amax = max(amax, max(__float_as_uint(v[2 * k]) & 0x7fffffffu, __float_as_uint(v[2 * k + 1]) & 0x7fffffffu));
    }
    amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const int X = mx_block_exponent(__uint_as_float(amax >= 0x7f800000u ? 0u : amax));
    const float inv = pow2_neg(X);
    uint32_t word[2] = {0u, 0u};
    int q1 = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const int tw = e2m1_twice(e2m1_encode(v[e], inv));
        word[e >> 2] |= ((uint32_t)tw & 0xffu) << (8 * (e & 3));
        q1 += tw < 0 ? -tw : tw;
    }
    q1 += __shfl_xor_sync(0xffffffffu, q1, 1);
    q1 += __shfl_xor_sync(0xffffffffu, q1, 2);
    if (t < nchunks) {
        const int h = t / (nb * 4), b = (t / 4) % nb, part = t & 3;
        Q.qw[h * nw + b * 8 + part * 2] = (int32_t)word[0];
        Q.qw[h * nw + b * 8 + part * 2 + 1] = (int32_t)word[1];
        if (part == 0) {
            Q.qx[h * 4 + b] = X;
            Q.q1[h * 4 + b] = q1;
        }
    }
    for (int h = t; h < H; h += blockDim.x) {
        const float x = w[h];
        const uint32_t u = __float_as_uint(x);
        const int ef = (int)((u >> 23) & 0xffu);
        int m = (int)(u & 0x7fffffu), e = -149;
        if (ef != 0) { m |= 0x800000; e = ef - 150; }
        Q.m_w[h] = (u >> 31) ? -m : m;
        Q.e_w[h] = e;
        Q.w[h] = x;
    }
    __syncthreads();
}

// Sign of sum_b I[b] * 2^E[b] (|I[b]| < 2^13), exactly: terms from the largest exponent
// down; once the partial sum is at least 2^15 times the next term's unit (a gap of >= 15
// bits, or a partial sum >= 2^40 of its own unit), the remaining terms (fewer than three,
// each below 2^13 of that unit) cannot change its sign.
template <int NB>
__device__ __forceinline__ int dyadic_sign(const int (&I)[NB], const int (&E)[NB])
{
    int ii[NB], ee[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) { ii[b] = I[b]; ee[b] = I[b] ? E[b] : -(1 << 20); }
#pragma unroll
    for (int i = 0; i < NB; ++i)
#pragma unroll
        for (int j = 0; j + 1 < NB - i; ++j)
            if (ee[j] < ee[j + 1]) {
                const int te = ee[j], ti = ii[j];
                ee[j] = ee[j + 1]; ii[j] = ii[j + 1];
                ee[j + 1] = te; ii[j + 1] = ti;
            }
    long long acc = 0;
    int base = 0;
#pragma unroll
    for (int t = 0; t < NB; ++t) {
        if (ii[t] == 0) continue;
        if (acc == 0) { acc = ii[t]; base = ee[t]; continue; }
        const int g = base - ee[t];
        if (g >= 15 || acc >= (1LL << 40) || acc <= -(1LL << 40)) break;
        acc = acc * (1LL << g) + ii[t];
        base = ee[t];
    }
    return acc > 0 ? 1 : (acc < 0 ? -1 : 0);
}

// Signed 32-bit slice of m * 2^(e - kE0) falling on limb `lane` (|m| < 2^63, e >= kE0).
__device__ __forceinline__ long long limb_slice(long long m, int e, int lane)
{
    const int lo = 32 * lane - (e - kE0);
    const unsigned long long a = (unsigned long long)(m < 0 ? -m : m);
    uint32_t s = 0;
    if (lo >= 0 && lo < 64) s = (uint32_t)(a >> lo);
    else if (lo < 0 && lo > -32) s = (uint32_t)(a << (-lo));
    return m < 0 ? -(long long)s : (long long)s;
}

// Four E2M1 codes (the low 16 bits, element 0 in the lowest nibble) as int8x4 of twice
// their values.
__device__ __forceinline__ int32_t twice_codes4(uint32_t x)
{
    uint32_t r = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) r |= ((uint32_t)e2m1_twice((x >> (4 * i)) & 15u) & 0xffu) << (8 * i);
    return (int32_t)r;
}

// Exact score of key row (kc: d/2 code bytes, ks: d/32 scale bytes) against Q, computed by
// the whole warp.  Returns limb `lane` of S (lanes >= kLimbs return 0), with the top limb's
// sign bit flipped, so that comparing limbs as unsigned from the top gives numeric order.
template <int D>
__device__ __noinline__ uint32_t score_key_limb(const QuantQuery &Q, int H, const uint8_t *kc, const uint8_t *ks)
{
    constexpr int NB = D / 32, NW = D / 4;
    const int lane = threadIdx.x & 31;
    const int32_t kw = lane < NW ? twice_codes4(*reinterpret_cast<const uint16_t *>(kc + 2 * lane)) : 0;
    int E_k[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) E_k[b] = (int)ks[b] - 127;
    long long acc = 0;
#pragma unroll 1
    for (int slot = 0; slot < 2; ++slot) {
        const int h = lane + 32 * slot;
        if (__all_sync(0xffffffffu, h >= H)) break;
        const bool live = h < H;
        const int hq = live ? h : 0;
        int I[NB], E[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            int a = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) a = __dp4a(Q.qw[hq * NW + b * 8 + j], __shfl_sync(0xffffffffu, kw, b * 8 + j), a);
            I[b] = a;
            E[b] = Q.qx[hq * 4 + b] + E_k[b] - 2;
        }
        const bool pos = live && Q.m_w[hq] != 0 && dyadic_sign<NB>(I, E) > 0;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const bool has = pos && I[b] != 0;
            const long long mant = has ? (long long)Q.m_w[hq] * I[b] : 0;
            const int e = Q.e_w[hq] + E[b];
            uint32_t mask = __ballot_sync(0xffffffffu, has);
#pragma unroll 1
            while (mask) {
                const int src = __ffs(mask) - 1;
                mask &= mask - 1u;
                const long long m = __shfl_sync(0xffffffffu, mant, src);
                const int ee = __shfl_sync(0xffffffffu, e, src);
                if (lane < kLimbs) acc += limb_slice(m, ee, lane);
            }
        }
    }
    // carries: limb j = (acc_j + carry_j) mod 2^32, carry_{j+1} = floor(./2^32)
    long long carry = 0;
    uint32_t limb = 0;
#pragma unroll 1
    for (int j = 0; j < kLimbs; ++j) {
        const long long v = acc + carry;
        if (lane == j) limb = (uint32_t)v;
        carry = __shfl_sync(0xffffffffu, v >> 32, j);
    }
    if (lane == kLimbs - 1) limb ^= 0x80000000u;
    return lane < kLimbs ? limb : 0u;
}

// Fixed-point form of the exact score for the common case: S = V * 2^E with V a signed
// 128-bit integer and E the smallest exponent among the score's terms.  Each term is
// m * 2^e with |m| < 2^37; a lane's terms (at most 8) are shifted to E by at most 80 bits,
// so a lane's sum stays below 2^120 and the warp's below 2^125.  Returns false (nothing
// decided) when a term lies more than 80 bits above E; the caller then takes the wide
// path.  A score with no terms is V = 0 (E = kNoTerms).  Warp-collective; every lane gets
// the result.
constexpr int kNoTerms = 1 << 30;

__device__ __forceinline__ __int128 shfl_xor_i128(__int128 v, int o)
{
    const unsigned long long lo = (unsigned long long)v, hi = (unsigned long long)(v >> 64);
    const unsigned long long lo2 = __shfl_xor_sync(0xffffffffu, lo, o), hi2 = __shfl_xor_sync(0xffffffffu, hi, o);
    return (__int128)(((unsigned __int128)hi2 << 64) | lo2);
}

// Significant bits of |v| (0 for v = 0).
__device__ __forceinline__ int bits_i128(__int128 v)
{
    const unsigned __int128 a = v < 0 ? (unsigned __int128)(-v) : (unsigned __int128)v;
    const unsigned long long hi = (unsigned long long)(a >> 64), lo = (unsigned long long)a;
    return hi ? 128 - __clzll((long long)hi) : (lo ? 64 - __clzll((long long)lo) : 0);
}

template <int D>
__device__ __noinline__ bool score_fixed(const QuantQuery &Q, int H, const uint8_t *kc, const uint8_t *ks,
                                         __int128 &V, int &E)
{
    constexpr int NB = D / 32, NW = D / 4;
    const int lane = threadIdx.x & 31;
    const int32_t kw = lane < NW ? twice_codes4(*reinterpret_cast<const uint16_t *>(kc + 2 * lane)) : 0;
    int E_k[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) E_k[b] = (int)ks[b] - 127;
    long long tm[2][NB];
    int te[2][NB];
    int emin = kNoTerms;
#pragma unroll
    for (int slot = 0; slot < 2; ++slot) {
        const int h = lane + 32 * slot;
        const bool live = h < H;
        const int hq = live ? h : 0;
        int I[NB], Ex[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            int a = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) a = __dp4a(Q.qw[hq * NW + b * 8 + j], __shfl_sync(0xffffffffu, kw, b * 8 + j), a);
            I[b] = a;
            Ex[b] = Q.qx[hq * 4 + b] + E_k[b] - 2;
        }
        const bool pos = live && Q.m_w[hq] != 0 && dyadic_sign<NB>(I, Ex) > 0;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const bool has = pos && I[b] != 0;
            tm[slot][b] = has ? (long long)Q.m_w[hq] * I[b] : 0;
            te[slot][b] = Q.e_w[hq] + Ex[b];
            if (has) emin = min(emin, te[slot][b]);
        }
        if (H <= 32) {
#pragma unroll
            for (int b = 0; b < NB; ++b) tm[1][b] = 0;
            break;
        }
    }
    E = __reduce_min_sync(0xffffffffu, emin);
    V = 0;
    if (E == kNoTerms) return true;
    bool ok = true;
    __int128 c = 0;
#pragma unroll
    for (int slot = 0; slot < 2; ++slot)
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            if (tm[slot][b] == 0) continue;
            const int sh = te[slot][b] - E;
            if (sh > 80) ok = false;
            else c += (__int128)tm[slot][b] << sh;
        }
    if (!__all_sync(0xffffffffu, ok)) return false;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += shfl_xor_i128(c, o);
    V = c;
    return true;
}

// Brings (V, E) to exponent E_to <= E: V << (E - E_to); false when that would leave more
// than 126 significant bits.
__device__ __forceinline__ bool align_fixed(__int128 &V, int E, int E_to)
{
    if (V == 0) return true;
    const int sh = E - E_to;
    if (sh < 0 || bits_i128(V) + sh > 126) return false;
    V = V << sh;
    return true;
}

// Compares two keys held one limb per lane (as returned by score_key_limb): > 0 when a is
// the larger score, 0 when equal.  Warp-collective.
__device__ __forceinline__ int compare_keys(uint32_t a, uint32_t b)
{
    const uint32_t diff = __ballot_sync(0xffffffffu, a != b);
    if (!diff) return 0;
    const int top = 31 - __clz((int)diff);
    const uint32_t xa = __shfl_sync(0xffffffffu, a, top), xb = __shfl_sync(0xffffffffu, b, top);
    return xa > xb ? 1 : -1;
}

} // namespace exact

// The row's error bound of the float32 scores as an affine function of the score,
// e(x) = c1 max(x, 0) + c0 (see above); it holds for finite scores (a row with another
// score gets no exact pass: the indexer has flagged CSA2_DEV_SCORE_RANGE).
//   every w_h >= 0: A_t = s_t <= (s~_t + eta) / (1 - c), so e(x) = c (x + eta) / (1 - c) + eta;
//   otherwise: one row-wide A from the key scale maxima, e = c A + eta.
// Evaluated in float32 with every operation rounded outward (a float64 unit this slow has
// no place in a per-row prologue); c1 = (H + 4) 2^-24 covers c / (1 - c) and that rounding,
// c0 >= eta = 2^-140 (sum|w| + H) covers the subnormal terms.
struct RowBound {
    float c1, c0;
    __device__ float e(float x) const { return __fmaf_ru(c1, x > 0.0f ? x : 0.0f, c0); }
    // below lo(tau): out; above hi(tau): in (x - e(x) and x + e(x) both rise with x)
    __device__ float lo(float x) const { return __fsub_rd(x, __fmul_ru(2.0f, e(x))); }
    __device__ float hi(float x) const
    {
        const float ex = e(x);
        return __fadd_ru(__fadd_ru(x, ex), e(__fmaf_ru(3.0f, ex, x)));
    }
};

// The bound of a row whose head weights w[0..H) are all >= 0 (neg = false); with a negative
// weight neg = true and the bound needs the key scale maxima (see csa2_topk).  The same
// evaluation serves every kernel that cuts candidates by it, so their cuts agree.
__device__ __forceinline__ RowBound row_bound_nonneg(const float *w, int H, bool &neg)
{
    float sumw = 0.0f;
    neg = false;
    for (int h = 0; h < H; ++h) {
        sumw = __fadd_ru(sumw, fabsf(w[h]));
        neg |= w[h] < 0.0f;
    }
    RowBound rb;
    rb.c1 = (float)(H + 4) * 0x1p-24f;
    rb.c0 = __fmul_ru(__fadd_ru(sumw, (float)H), 0x1p-140f);
    return rb;
}

} // namespace csa2
