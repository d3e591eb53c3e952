// common.cuh -- device helpers shared by the CSA2 kernels of libcsa2.so.
//
// MXFP4 (E2M1 elements, E8M0 scale per 32; DeepSeek-V4.1-Flash report,
// aipaper.jasonlin.tech §2.4.4, which names the OCP MXFP4 format for indexer queries and
// keys), the order-preserving key used by selection, and exact float32 rounding of a
// sum of scaled integers (the indexer's per-head dot).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/csa2.h"

namespace csa2 {

// ------------------------------------------------------------------ status helpers
__device__ __forceinline__ void dev_flag(uint32_t *d_status, uint32_t bits)
{
    if (d_status) atomicOr(d_status, bits);
}

// ------------------------------------------------------------------ MXFP4 codec
// floor(log2(a)) for finite a > 0, from the float's bits (subnormals included).
__device__ __forceinline__ int floor_log2_f32(float a)
{
    uint32_t u = __float_as_uint(a);
    int e = (int)((u >> 23) & 0xffu);
    if (e != 0) return e - 127;
    return -149 + (31 - __clz((int)(u & 0x7fffffu)));
}

// Shared scale exponent X of a block with maximum magnitude amax (finite, >= 0):
// floor(log2 amax) - 2 clamped to [-127, 127]; 0 for an all-zero block.
__device__ __forceinline__ int mx_block_exponent(float amax)
{
    if (!(amax > 0.0f)) return 0;
    int x = floor_log2_f32(amax) - 2;
    return x < -127 ? -127 : (x > 127 ? 127 : x);
}

// 2^-X as a float for X in [-127, 125] (normal, exact).
__device__ __forceinline__ float pow2_neg(int X)
{
    int b = 127 - X;
    b = b < 1 ? 1 : (b > 254 ? 254 : b);
    return __uint_as_float((uint32_t)b << 23);
}

// E2M1 code of x at block scale 2^X (inv = 2^-X): magnitude rounded to the nearest of
// {0, .5, 1, 1.5, 2, 3, 4, 6}, ties to the even code, saturating; bit 3 = sign bit of x.
// |x| * inv is exact whenever it can reach a rounding boundary (it is >= 2^-126 there).
__device__ __forceinline__ uint32_t e2m1_encode(float x, float inv)
{
    float v = fabsf(x) * inv;
    uint32_t c = v <= 0.25f ? 0u
               : v < 0.75f  ? 1u
               : v <= 1.25f ? 2u
               : v < 1.75f  ? 3u
               : v <= 2.5f  ? 4u
               : v < 3.5f   ? 5u
               : v <= 5.0f  ? 6u
                            : 7u;
    return c | ((__float_as_uint(x) >> 28) & 8u);
}

// The E2M1 codes of two already scaled values (a to the low nibble, b to the high one) by
// the hardware conversion: round to nearest, ties to even, saturating at 6, sign kept --
// the rule of e2m1_encode, checked against it on the GPU over every rounding boundary.
__device__ __forceinline__ uint32_t e2m1x2_cvt(float a_scaled, float b_scaled)
{
    uint16_t d;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u16.u8 %0, t;\n\t}"
        : "=h"(d) : "f"(b_scaled), "f"(a_scaled));
    return d;
}

// Magnitude of an E2M1 code's low 3 bits, as float.
__device__ __forceinline__ float e2m1_mag(uint32_t c3)
{
    // 0, .5, 1, 1.5, 2, 3, 4, 6: exponent field e = c3>>1, mantissa bit m = c3&1
    uint32_t e = (c3 >> 1) & 3u, m = c3 & 1u;
    return e == 0 ? 0.5f * (float)m : __uint_as_float(((e + 126u) << 23) | (m << 22));
}

// 2^(sb - 127) as float for a scale byte sb (sb = 0 gives the subnormal 2^-127).
__device__ __forceinline__ float e8m0_value(uint32_t sb)
{
    return sb == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(sb << 23);
}

// ------------------------------------------------------------------ E4M3 block scales
// (report §2.4.4: the main KV keeps E2M1 values with one E4M3 scale per 16.)
// Value of an E4M3 byte: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent field
// 0 is subnormal (m x 2^-9); 0x7F / 0xFF are NaN.
__device__ __forceinline__ float e4m3_value(uint32_t byte)
{
    const uint32_t e = (byte >> 3) & 15u, m = byte & 7u;
    float mag = e == 0 ? (float)m * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
    if ((byte & 0x7fu) == 0x7fu) mag = __uint_as_float(0x7fc00000u);
    return (byte & 0x80u) ? -mag : mag;
}

// Scale byte of a 16-value block with maximum magnitude amax (finite, >= 0): amax / 6
// rounded to the nearest E4M3 value, ties to even, clamped to 448.  The float32 quotient
// rounds onto an E4M3 midpoint only when the exact quotient is that midpoint (the
// midpoints have 5 significant bits), so the two roundings give the exact one.
__device__ __forceinline__ uint32_t e4m3_block_scale(float amax)
{
    const float t = __fdiv_rn(amax, 6.0f);
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(d) : "f"(t));
    return (uint32_t)(d & 0xffu);
}

// ------------------------------------------------------------------ MXFP8 (E4M3) SWA
// (report §2.4.4: the SWA KV cache stays in FP8; OCP MX with E4M3 elements.)
// Shared exponent X of a 32-value block with maximum magnitude amax (finite, >= 0):
// floor(log2 amax) - 8 clamped to [-127, 127]; 0 for an all-zero block.
__device__ __forceinline__ int mx8_block_exponent(float amax)
{
    if (!(amax > 0.0f)) return 0;
    const int x = floor_log2_f32(amax) - 8;
    return x < -127 ? -127 : (x > 127 ? 127 : x);
}

// E4M3 code of an already scaled value by the hardware conversion: round to nearest, ties
// to even, saturating at +-448, sign kept (also for results that round to zero).
__device__ __forceinline__ uint32_t e4m3_cvt(float v)
{
    uint16_t d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %1;" : "=h"(d) : "f"(v));
    return (uint32_t)(d & 0xffu);
}

// Twice the signed E2M1 value of a code, an integer in [-12, 12].
__device__ __forceinline__ int e2m1_twice(uint32_t c)
{
    const int m = (int)(2.0f * e2m1_mag(c & 7u));
    return (c & 8u) ? -m : m;
}

// ------------------------------------------------------------------ selection key
// Order-preserving 32-bit key of a float score: larger key = better; -0 == +0; NaN = 0
// (below every number, including -inf).
__device__ __forceinline__ uint32_t score_key(float s)
{
    uint32_t u = __float_as_uint(s);
    if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// The float a key stands for (the inverse of score_key on numbers).
__device__ __forceinline__ float key_value(uint32_t key)
{
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// ------------------------------------------------------------------ exact rounding
// float32 round-to-nearest-even of sum_b I[b] * 2^E[b] (|I[b]| < 2^20, E in [-300, 260]).
//
// Fast case: every nonzero term normal, exponents within 9 of each other and far from
// overflow, so every partial sum is exact in float32 whatever the order.  Otherwise the
// terms are added exactly in a wide two's-complement integer and rounded once.
struct WideAcc {
    static constexpr int kWords = 20;     // 640 bits
    static constexpr int kBase = -330;    // weight of bit 0
    uint32_t w[kWords];
};

static __device__ __noinline__ float wide_sum_round_f32(int n, const int *I, const int *E)
{
    WideAcc a;
#pragma unroll 1
    for (int i = 0; i < WideAcc::kWords; ++i) a.w[i] = 0u;
#pragma unroll 1
    for (int t = 0; t < n; ++t) {
        if (I[t] == 0) continue;
        uint64_t mag = (uint64_t)(I[t] < 0 ? -(int64_t)I[t] : (int64_t)I[t]);
        int sh = E[t] - WideAcc::kBase;
        int word = sh >> 5, bit = sh & 31;
        uint32_t part[3];
        part[0] = (uint32_t)(mag << bit);
        part[1] = (uint32_t)((mag << bit) >> 32);
        part[2] = bit ? (uint32_t)(mag >> (64 - bit)) : 0u;
        // add or subtract part << (32*word)
        uint64_t carry = 0;
        if (I[t] > 0) {
#pragma unroll 1
            for (int i = word; i < WideAcc::kWords; ++i) {
                uint64_t v = (uint64_t)a.w[i] + (i - word < 3 ? part[i - word] : 0u) + carry;
                a.w[i] = (uint32_t)v;
                carry = v >> 32;
            }
        } else {
            uint64_t borrow = 0;
#pragma unroll 1
            for (int i = word; i < WideAcc::kWords; ++i) {
                uint64_t sub = (uint64_t)(i - word < 3 ? part[i - word] : 0u) + borrow;
                borrow = (uint64_t)a.w[i] < sub ? 1u : 0u;
                a.w[i] = (uint32_t)((uint64_t)a.w[i] - sub);
            }
        }
    }
    const bool neg = (a.w[WideAcc::kWords - 1] >> 31) != 0;
    if (neg) {                      // magnitude = two's complement negation
        uint64_t c = 1;
#pragma unroll 1
        for (int i = 0; i < WideAcc::kWords; ++i) {
            uint64_t v = (uint64_t)(~a.w[i]) + c;
            a.w[i] = (uint32_t)v;
            c = v >> 32;
        }
    }
    int msb = -1;
#pragma unroll 1
    for (int i = WideAcc::kWords - 1; i >= 0 && msb < 0; --i)
        if (a.w[i]) msb = 32 * i + 31 - __clz((int)a.w[i]);
    if (msb < 0) return 0.0f;
    auto bit_at = [&](int i) -> uint32_t {
        return (i < 0) ? 0u : ((a.w[i >> 5] >> (i & 31)) & 1u);
    };
    int keep_lo = msb - 23;                                   // 24 significant bits
    if (keep_lo + WideAcc::kBase < -149) keep_lo = -149 - WideAcc::kBase;   // subnormal
    uint32_t m = 0;
#pragma unroll 1
    for (int i = msb; i >= keep_lo; --i) m = (m << 1) | bit_at(i);
    uint32_t rnd = bit_at(keep_lo - 1), sticky = 0;
#pragma unroll 1
    for (int i = keep_lo - 2; i >= 0 && !sticky; --i) sticky |= bit_at(i);
    if (rnd && (sticky || (m & 1u))) ++m;
    // value = m * 2^(keep_lo + kBase), m <= 2^24: scale in two exact steps
    int e = keep_lo + WideAcc::kBase;
    float f = (float)m;                                        // exact
    if (e > 0) {
        int e1 = e > 127 ? 127 : e;
        f *= __uint_as_float((uint32_t)(e1 + 127) << 23);
        if (e - e1 > 0) f *= __uint_as_float((uint32_t)(min(e - e1, 127) + 127) << 23);  // inf
    } else if (e < 0) {
        // m * 2^e with the result normal or an exact subnormal: first to [2^-100] range
        int e1 = e < -100 ? -100 : e;
        f *= __uint_as_float((uint32_t)(e1 + 127) << 23);
        if (e - e1 < 0) f *= __uint_as_float((uint32_t)(e - e1 + 127) << 23);
    }
    return neg ? -f : f;
}

template <int NB>
__device__ __forceinline__ float dyadic_sum_f32(const int (&I)[NB], const int (&E)[NB])
{
    int emin = 1 << 20, emax = -(1 << 20);
#pragma unroll
    for (int b = 0; b < NB; ++b)
        if (I[b] != 0) { emin = min(emin, E[b]); emax = max(emax, E[b]); }
    if (emax < emin) return 0.0f;
    if (emin >= -126 && emax <= 100 && emax - emin <= 9) {
        float s = 0.0f;
#pragma unroll
        for (int b = 0; b < NB; ++b)
            s += (float)I[b] * __uint_as_float((uint32_t)(min(max(E[b], -126), 127) + 127) << 23);
        return s;
    }
    return wide_sum_round_f32(NB, I, E);
}

// ------------------------------------------------------------------ dependent launch
// A kernel launched with programmatic dependent launch waits here until the previous
// kernel in the stream has completed and its writes are visible (immediately, when there
// is no such kernel); pdl_allow_dependents lets the next kernel in the stream start its
// own set-up early.  The indexer, Top-K, attention and RoPE cache-write kernels call it
// (the indexer then streams the cache rows written before this step while the cache write
// runs); the other conversion kernels let the next kernel start only when they finish.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

} // namespace csa2
