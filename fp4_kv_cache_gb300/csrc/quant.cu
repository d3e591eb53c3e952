// quant.cu -- 4-bit cache codec kernels (csa2_quant_fp4 / csa2_dequant_fp4).
//
// DeepSeek-V4.1-Flash report (aipaper.jasonlin.tech) §2.4.4: indexer queries and keys use
// OCP MXFP4 -- E2M1 values with one power-of-two (E8M0) scale per 32 -- the main KV keeps
// E2M1 values with one E4M3 scale per 16, and cached values are dequantised before
// attention.  MXFP4 scalar kernel: one warp quantises one 32-value block per step: lane i
// holds element i, the block maximum is a warp max over the magnitude bits, and lane
// pairs merge their nibbles (element 2i in the low nibble).
#include "common.cuh"
#include "internal.h"
#include <cuda_bf16.h>

namespace csa2 {
namespace {

template <bool BF16>
__global__ void __launch_bounds__(256) quant_mxfp4_kernel(const void *__restrict__ x, int64_t rows,
                                                          int64_t cols, int64_t ldx,
                                                          uint8_t *__restrict__ codes, int64_t ldc,
                                                          uint8_t *__restrict__ scales, int64_t lds,
                                                          uint32_t *d_status)
{
    const int lane = threadIdx.x & 31;
    const int64_t nblk_row = cols / 32;
    const int64_t total = rows * nblk_row;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t blk = warp0; blk < total; blk += nwarps) {
        const int64_t r = blk / nblk_row, kb = blk % nblk_row;
        const int64_t col = kb * 32 + lane;
        float v;
        if (BF16) {
            uint16_t bits = static_cast<const uint16_t *>(x)[r * ldx + col];
            v = __uint_as_float((uint32_t)bits << 16);
        } else {
            v = static_cast<const float *>(x)[r * ldx + col];
        }
        const uint32_t mag_bits = __float_as_uint(v) & 0x7fffffffu;
        const uint32_t amax_bits = __reduce_max_sync(0xffffffffu, mag_bits);
        if (amax_bits >= 0x7f800000u && lane == 0) dev_flag(d_status, CSA2_DEV_NONFINITE);
        const int X = mx_block_exponent(__uint_as_float(amax_bits >= 0x7f800000u ? 0u : amax_bits));
        const uint32_t c = e2m1_encode(v, pow2_neg(X));
        const uint32_t c_hi = __shfl_down_sync(0xffffffffu, c, 1);
        if ((lane & 1) == 0) codes[r * ldc + kb * 16 + (lane >> 1)] = (uint8_t)(c | (c_hi << 4));
        if (lane == 0) scales[r * lds + kb] = (uint8_t)(X + 127);
    }
}

// Vectorised variant: four lanes share a 32-value block, each lane converts 8 values
// (one 16-byte bf16 load or two 16-byte f32 loads) and stores their 8 nibbles as one
// 32-bit word.  Needs 16-byte aligned rows of x and 4-byte aligned rows of codes.
template <bool BF16>
__global__ void __launch_bounds__(256) quant_mxfp4_vec_kernel(const void *__restrict__ x, int64_t rows,
                                                              int64_t cols, int64_t ldx,
                                                              uint8_t *__restrict__ codes, int64_t ldc,
                                                              uint8_t *__restrict__ scales, int64_t lds,
                                                              uint32_t *d_status)
{
    pdl_wait();                                   // x may come from the kernel before
    const int64_t nblk_row = cols / 32;
    const int64_t total = rows * nblk_row * 4;                 // lanes of work
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t total32 = (total + 31) & ~int64_t(31);
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total32; t += stride) {
        const bool act = t < total;
        const int64_t grp = t >> 2;
        const int sub = (int)(t & 3);
        const int64_t r = act ? grp / nblk_row : 0, kb = act ? grp % nblk_row : 0;
        float v[8];
        if (act) {
            if (BF16) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(x) +
                                                                   r * ldx + kb * 32 + sub * 8);
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    v[2 * i] = __uint_as_float(w[i] << 16);
                    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
                }
            } else {
                const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(x) +
                                                                     r * ldx + kb * 32 + sub * 8);
                const float4 a = src[0], b = src[1];
                v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
                v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = 0.0f;
        }
        uint32_t amax = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = max(amax, __float_as_uint(v[i]) & 0x7fffffffu);
        amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        if (!act) continue;
        const bool finite = amax < 0x7f800000u;
        if (!finite && sub == 0) dev_flag(d_status, CSA2_DEV_NONFINITE);
        const int X = mx_block_exponent(__uint_as_float(finite ? amax : 0u));
        const float inv = pow2_neg(X);
        uint32_t word = 0;
#pragma unroll
        for (int i = 0; i < 8; i += 2) word |= e2m1x2_cvt(v[i] * inv, v[i + 1] * inv) << (4 * i);
        *reinterpret_cast<uint32_t *>(codes + r * ldc + kb * 16 + sub * 4) = word;
        if (sub == 0) scales[r * lds + kb] = (uint8_t)(X + 127);
    }
}

// Several jobs in one launch: their 4-lane block groups are laid end to end (each job's
// lane count is a multiple of 4, so no group straddles two jobs) and every lane finds its
// job from the running lane counts; the per-lane work is the vectorised kernel's.
struct QuantBatchParams {
    const void *x[4];
    uint8_t *codes[4], *scales[4];
    int64_t nblk[4], ldx[4], ldc[4], lds[4];
    int64_t lanes_end[4];          // running total of 4 x blocks over jobs 0..j
    int bf16[4];
    int n;
};

__global__ void __launch_bounds__(256) quant_mxfp4_batch_kernel(const __grid_constant__ QuantBatchParams B,
                                                                uint32_t *d_status)
{
    pdl_wait();                                   // x may come from the kernel before
    const int64_t total = B.lanes_end[B.n - 1];
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t total32 = (total + 31) & ~int64_t(31);
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total32; t += stride) {
        const bool act = t < total;
        int j = 0;
#pragma unroll
        for (int k = 0; k < 3; ++k) j += (k + 1 < B.n && t >= B.lanes_end[k]) ? 1 : 0;
        const int64_t tl = act ? t - (j > 0 ? B.lanes_end[j - 1] : 0) : 0;
        const int64_t grp = tl >> 2;
        const int sub = (int)(tl & 3);
        const int64_t nblk = B.nblk[j];
        const int64_t r = grp / nblk, kb = grp % nblk;
        float v[8];
        if (act && B.bf16[j]) {
            const uint4 raw = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(B.x[j]) +
                                                               r * B.ldx[j] + kb * 32 + sub * 8);
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[2 * i] = __uint_as_float(w[i] << 16);
                v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
            }
        } else if (act) {
            const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(B.x[j]) +
                                                                 r * B.ldx[j] + kb * 32 + sub * 8);
            const float4 a = src[0], b = src[1];
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
            v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = 0.0f;
        }
        uint32_t amax = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = max(amax, __float_as_uint(v[i]) & 0x7fffffffu);
        amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        if (!act) continue;
        const bool finite = amax < 0x7f800000u;
        if (!finite && sub == 0) dev_flag(d_status, CSA2_DEV_NONFINITE);
        const int X = mx_block_exponent(__uint_as_float(finite ? amax : 0u));
        const float inv = pow2_neg(X);
        uint32_t word = 0;
#pragma unroll
        for (int i = 0; i < 8; i += 2) word |= e2m1x2_cvt(v[i] * inv, v[i + 1] * inv) << (4 * i);
        *reinterpret_cast<uint32_t *>(B.codes[j] + r * B.ldc[j] + kb * 16 + sub * 4) = word;
        if (sub == 0) B.scales[j][r * B.lds[j] + kb] = (uint8_t)(X + 127);
    }
}

// ---------------------------------------------------------------- E2M1 + E4M3 per 16
// The report's main-KV format (§2.4.4): one E4M3 scale per 16 values, no global scale.
// Scale = amax/6 rounded to E4M3 (e4m3_block_scale); element code = the E2M1 rounding of
// x / scale.  The float32 quotient x / scale rounds onto an E2M1 midpoint only when the
// exact quotient is that midpoint (x has <= 24 significant bits, scale x midpoint <= 7),
// so the hardware conversion of the quotient gives the exact rounding.  A zero scale
// leaves only the sign bits.

// Two lanes share a 16-value block; each converts 8 values (one 16-byte bf16 load or two
// 16-byte f32 loads) and stores their 8 nibbles as one 32-bit word.  Needs 16-byte aligned
// rows of x and 4-byte aligned rows of codes.
template <bool BF16>
__global__ void __launch_bounds__(256) quant_nvfp4_vec_kernel(const void *__restrict__ x, int64_t rows,
                                                              int64_t cols, int64_t ldx,
                                                              uint8_t *__restrict__ codes, int64_t ldc,
                                                              uint8_t *__restrict__ scales, int64_t lds,
                                                              uint32_t *d_status)
{
    pdl_wait();                                   // x may come from the kernel before
    const int64_t nblk_row = cols / 16;
    const int64_t total = rows * nblk_row * 2;                 // lanes of work
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t total32 = (total + 31) & ~int64_t(31);
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total32; t += stride) {
        const bool act = t < total;
        const int64_t grp = t >> 1;
        const int sub = (int)(t & 1);
        const int64_t r = act ? grp / nblk_row : 0, kb = act ? grp % nblk_row : 0;
        float v[8];
        if (act) {
            if (BF16) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(x) +
                                                                   r * ldx + kb * 16 + sub * 8);
                const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    v[2 * i] = __uint_as_float(w[i] << 16);
                    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
                }
            } else {
                const float4 *src = reinterpret_cast<const float4 *>(static_cast<const float *>(x) +
                                                                     r * ldx + kb * 16 + sub * 8);
                const float4 a = src[0], b = src[1];
                v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
                v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = 0.0f;
        }
        uint32_t amax = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = max(amax, __float_as_uint(v[i]) & 0x7fffffffu);
        amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        if (!act) continue;
        const bool finite = amax < 0x7f800000u;
        if (!finite && sub == 0) dev_flag(d_status, CSA2_DEV_NONFINITE);
        const uint32_t sb = e4m3_block_scale(__uint_as_float(finite ? amax : 0u));
        const float sc = e4m3_value(sb);
        uint32_t word = 0;
        if (sc > 0.0f) {
#pragma unroll
            for (int i = 0; i < 8; i += 2)
                word |= e2m1x2_cvt(__fdiv_rn(v[i], sc), __fdiv_rn(v[i + 1], sc)) << (4 * i);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) word |= (__float_as_uint(v[i]) >> 31) << (4 * i + 3);
        }
        *reinterpret_cast<uint32_t *>(codes + r * ldc + kb * 8 + sub * 4) = word;
        if (sub == 0) scales[r * lds + kb] = (uint8_t)sb;
    }
}

// Rows without the vector kernel's alignment: one warp takes two 16-value blocks per step
// (lane = element), block maximum by shuffles within each half-warp.
template <bool BF16>
__global__ void __launch_bounds__(256) quant_nvfp4_kernel(const void *__restrict__ x, int64_t rows,
                                                          int64_t cols, int64_t ldx,
                                                          uint8_t *__restrict__ codes, int64_t ldc,
                                                          uint8_t *__restrict__ scales, int64_t lds,
                                                          uint32_t *d_status)
{
    const int lane = threadIdx.x & 31, e16 = lane & 15;
    const int64_t nblk_row = cols / 16;
    const int64_t total = rows * nblk_row;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t pair = warp0; pair * 2 < total; pair += nwarps) {
        const int64_t blk = pair * 2 + (lane >> 4);
        const bool act = blk < total;
        const int64_t r = act ? blk / nblk_row : 0, kb = act ? blk % nblk_row : 0;
        const int64_t col = kb * 16 + e16;
        float v = 0.0f;
        if (act) {
            if (BF16) v = __uint_as_float((uint32_t)static_cast<const uint16_t *>(x)[r * ldx + col] << 16);
            else v = static_cast<const float *>(x)[r * ldx + col];
        }
        uint32_t amax = __float_as_uint(v) & 0x7fffffffu;
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const bool finite = amax < 0x7f800000u;
        if (act && !finite && e16 == 0) dev_flag(d_status, CSA2_DEV_NONFINITE);
        const uint32_t sb = e4m3_block_scale(__uint_as_float(finite ? amax : 0u));
        const float sc = e4m3_value(sb);
        const uint32_t c = sc > 0.0f ? (e2m1x2_cvt(__fdiv_rn(v, sc), 0.0f) & 15u)
                                     : ((__float_as_uint(v) >> 28) & 8u);
        const uint32_t c_hi = __shfl_down_sync(0xffffffffu, c, 1);
        if (act && (lane & 1) == 0) codes[r * ldc + kb * 8 + (e16 >> 1)] = (uint8_t)(c | (c_hi << 4));
        if (act && e16 == 0) scales[r * lds + kb] = (uint8_t)sb;
    }
}

template <bool BF16, bool NV>
__global__ void __launch_bounds__(256) dequant_fp4_kernel(const uint8_t *__restrict__ codes,
                                                          int64_t ldc,
                                                          const uint8_t *__restrict__ scales,
                                                          int64_t lds, int64_t rows, int64_t cols,
                                                          void *__restrict__ y, int64_t ldy)
{
    const int64_t total = rows * cols;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / cols, c = i % cols;
        const uint32_t byte = codes[r * ldc + c / 2];
        const uint32_t code = (c & 1) ? (byte >> 4) : (byte & 15u);
        float v = e2m1_mag(code & 7u) * (NV ? e4m3_value(scales[r * lds + c / 16])
                                            : e8m0_value(scales[r * lds + c / 32]));
        if (code & 8u) v = -v;
        if (BF16)
            static_cast<uint16_t *>(y)[r * ldy + c] = (uint16_t)(__float_as_uint(v) >> 16);
        else
            static_cast<float *>(y)[r * ldy + c] = v;
    }
}

// ---------------------------------------------------------------- MXFP8 (E4M3) SWA codec
// One warp per 32-value block: the block maximum by a warp reduction, X = floor(log2 amax)
// - 8, each lane's value times 2^-X (exact: a power of two, and any product below 2^-126
// lies far below the first E4M3 rounding boundary 2^-10) converted by the hardware.
template <bool BF16>
__global__ void __launch_bounds__(256) quant_mxfp8_kernel(const void *__restrict__ x, int64_t rows,
                                                          int64_t cols, int64_t ldx,
                                                          uint8_t *__restrict__ codes, int64_t ldc,
                                                          uint8_t *__restrict__ scales, int64_t lds,
                                                          uint32_t *d_status)
{
    const int lane = threadIdx.x & 31;
    const int64_t nblk_row = cols / 32;
    const int64_t total = rows * nblk_row;
    const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    pdl_wait();
    for (int64_t blk = warp0; blk < total; blk += nwarps) {
        const int64_t r = blk / nblk_row, kb = blk % nblk_row;
        const int64_t col = kb * 32 + lane;
        float v;
        if (BF16) v = __uint_as_float((uint32_t)static_cast<const uint16_t *>(x)[r * ldx + col] << 16);
        else v = static_cast<const float *>(x)[r * ldx + col];
        const uint32_t amax_bits = __reduce_max_sync(0xffffffffu, __float_as_uint(v) & 0x7fffffffu);
        if (amax_bits >= 0x7f800000u && lane == 0) dev_flag(d_status, CSA2_DEV_NONFINITE);
        const int X = mx8_block_exponent(__uint_as_float(amax_bits >= 0x7f800000u ? 0u : amax_bits));
        codes[r * ldc + col] = (uint8_t)e4m3_cvt(v * pow2_neg(X));
        if (lane == 0) scales[r * lds + kb] = (uint8_t)(X + 127);
    }
}

template <bool BF16>
__global__ void __launch_bounds__(256) dequant_mxfp8_kernel(const uint8_t *__restrict__ codes, int64_t ldc,
                                                            const uint8_t *__restrict__ scales, int64_t lds,
                                                            int64_t rows, int64_t cols, void *__restrict__ y,
                                                            int64_t ldy)
{
    const int64_t total = rows * cols;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / cols, c = i % cols;
        // E4M3 value (at most 4 significant bits) x 2^(e - 127): exact in float32
        const float v = e4m3_value(codes[r * ldc + c]) * e8m0_value(scales[r * lds + c / 32]);
        if (BF16)
            static_cast<uint16_t *>(y)[r * ldy + c] = (uint16_t)(__float_as_uint(v) >> 16);
        else
            static_cast<float *>(y)[r * ldy + c] = v;
    }
}

// ---------------------------------------------------------------- RoPE + quantise
// The cache write of report §2.4.4 (quantise after RoPE, one format for both parts): every
// lane takes 8 values of one block (one 16-byte bf16 load), rotates the pairs that fall in
// the trailing rope_dim channels with the caller's cos/sin row, and quantises like the
// vector kernels above.  Jobs are laid end to end; each job's lane run starts on a multiple
// of 4 so that a block's lanes (4 for MXFP4, 2 for E2M1 + E4M3/16) share an aligned group.
struct RopeQuantParams {
    const uint16_t *x[4];
    const int32_t *pos[4];
    const float *cs[4];
    uint8_t *codes[4], *scales[4];
    int64_t cols[4], nblk[4], blocks[4], ldx[4], ldc[4], lds[4], n_pos[4];
    int64_t lanes_end[4];          // running total of each job's lanes, rounded up to 4
    int32_t rope[4], nv[4];
    int n;
};

__global__ void __launch_bounds__(256) rope_quant_kernel(const __grid_constant__ RopeQuantParams B,
                                                         uint32_t *d_status)
{
    pdl_wait();                                   // x and pos may come from the kernel before
    pdl_allow_dependents();                       // the indexer streams older rows meanwhile
    const int64_t total = B.lanes_end[B.n - 1];
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t total32 = (total + 31) & ~int64_t(31);
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < total32; t += stride) {
        int j = 0;
#pragma unroll
        for (int k = 0; k < 3; ++k) j += (k + 1 < B.n && t >= B.lanes_end[k]) ? 1 : 0;
        const int64_t tl = t < total ? t - (j > 0 ? B.lanes_end[j - 1] : 0) : 0;
        const bool nv = B.nv[j] != 0;
        const int64_t grp = nv ? tl >> 1 : tl >> 2;
        const int sub = (int)(tl & (nv ? 1 : 3));
        const bool act = t < total && grp < B.blocks[j];
        const int64_t nblk = B.nblk[j];
        const int64_t r = act ? grp / nblk : 0, kb = act ? grp % nblk : 0;
        const int G = nv ? 16 : 32;
        const int64_t col = kb * G + sub * 8;
        float v[8];
        if (act) {
            const uint4 raw = *reinterpret_cast<const uint4 *>(B.x[j] + r * B.ldx[j] + col);
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                v[2 * i] = __uint_as_float(w[i] << 16);
                v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
            }
            const int rope = B.rope[j];
            const int64_t c0 = B.cols[j] - rope;
            if (rope > 0 && col + 8 > c0) {
                const int64_t p = B.pos[j][r];
                if (p < 0 || p >= B.n_pos[j]) {
                    dev_flag(d_status, CSA2_DEV_BAD_INDEX);
                } else {
                    const float *cs = B.cs[j] + p * rope;
                    const int half = rope >> 1;
#pragma unroll
                    for (int e = 0; e < 8; e += 2) {
                        if (col + e >= c0) {          // c0 and col + e are even: a whole pair
                            const int i = (int)((col + e - c0) >> 1);
                            const float c = cs[i], sn = cs[half + i], a = v[e], b = v[e + 1];
                            v[e] = __fsub_rn(__fmul_rn(a, c), __fmul_rn(b, sn));
                            v[e + 1] = __fadd_rn(__fmul_rn(a, sn), __fmul_rn(b, c));
                        }
                    }
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = 0.0f;
        }
        uint32_t amax = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = max(amax, __float_as_uint(v[i]) & 0x7fffffffu);
        amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        const uint32_t amax4 = max(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        if (!nv) amax = amax4;
        if (!act) continue;
        const bool finite = amax < 0x7f800000u;
        if (!finite && sub == 0) dev_flag(d_status, CSA2_DEV_NONFINITE);
        const float amax_f = __uint_as_float(finite ? amax : 0u);
        uint32_t word = 0, sbyte;
        if (nv) {
            sbyte = e4m3_block_scale(amax_f);
            const float sc = e4m3_value(sbyte);
            if (sc > 0.0f) {
#pragma unroll
                for (int i = 0; i < 8; i += 2)
                    word |= e2m1x2_cvt(__fdiv_rn(v[i], sc), __fdiv_rn(v[i + 1], sc)) << (4 * i);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) word |= (__float_as_uint(v[i]) >> 31) << (4 * i + 3);
            }
        } else {
            const int X = mx_block_exponent(amax_f);
            const float inv = pow2_neg(X);
#pragma unroll
            for (int i = 0; i < 8; i += 2) word |= e2m1x2_cvt(v[i] * inv, v[i + 1] * inv) << (4 * i);
            sbyte = (uint32_t)(X + 127);
        }
        *reinterpret_cast<uint32_t *>(B.codes[j] + r * B.ldc[j] + kb * (G / 2) + sub * 4) = word;
        if (sub == 0) B.scales[j][r * B.lds[j] + kb] = (uint8_t)sbyte;
    }
}

int grid_for(int64_t work_items, int per_block)
{
    int64_t g = (work_items + per_block - 1) / per_block;
    if (g < 1) g = 1;
    const int64_t gmax = (int64_t)device_sm_count() * 16;
    if (g > gmax) g = gmax;
    return (int)g;
}

} // namespace

cudaError_t launch_quant_mxfp4(const void *x, bool x_bf16, int64_t rows, int64_t cols, int64_t ldx,
                               uint8_t *codes, int64_t ldc, uint8_t *scales, int64_t lds,
                               uint32_t *d_status, cudaStream_t s)
{
    if (rows == 0 || cols == 0) return cudaSuccess;
    const size_t esz = x_bf16 ? 2 : 4;
    const bool vec = ((uintptr_t)x % 16 == 0) && ((ldx * (int64_t)esz) % 16 == 0) &&
                     ((uintptr_t)codes % 4 == 0) && (ldc % 4 == 0);
    if (vec) {
        const int grid = grid_for(rows * (cols / 32) * 4, 256);
        if (x_bf16)
            return launch_pdl(quant_mxfp4_vec_kernel<true>, dim3(grid), dim3(256), 0, s, 1, x, rows, cols, ldx,
                              codes, ldc, scales, lds, d_status);
        return launch_pdl(quant_mxfp4_vec_kernel<false>, dim3(grid), dim3(256), 0, s, 1, x, rows, cols, ldx,
                          codes, ldc, scales, lds, d_status);
    }
    const int grid = grid_for(rows * (cols / 32), 8);
    if (x_bf16)
        quant_mxfp4_kernel<true><<<grid, 256, 0, s>>>(x, rows, cols, ldx, codes, ldc, scales, lds,
                                                      d_status);
    else
        quant_mxfp4_kernel<false><<<grid, 256, 0, s>>>(x, rows, cols, ldx, codes, ldc, scales, lds,
                                                       d_status);
    return cudaGetLastError();
}

bool quant_job_vec_ok(const QuantJobDesc &j)
{
    const size_t esz = j.x_bf16 ? 2 : 4;
    return ((uintptr_t)j.x % 16 == 0) && ((j.ldx * (int64_t)esz) % 16 == 0) && ((uintptr_t)j.codes % 4 == 0) &&
           (j.ldc % 4 == 0);
}

cudaError_t launch_quant_mxfp4_batch(const QuantJobDesc *jobs, int n_jobs, uint32_t *d_status, cudaStream_t s)
{
    if (n_jobs < 1 || n_jobs > 4) return cudaErrorInvalidValue;
    QuantBatchParams B = {};
    int64_t acc = 0;
    int n = 0;
    for (int k = 0; k < n_jobs; ++k) {
        const QuantJobDesc &j = jobs[k];
        if (!quant_job_vec_ok(j)) return cudaErrorInvalidValue;
        if (j.rows == 0 || j.cols == 0) continue;
        B.x[n] = j.x;
        B.codes[n] = j.codes;
        B.scales[n] = j.scales;
        B.nblk[n] = j.cols / 32;
        B.ldx[n] = j.ldx;
        B.ldc[n] = j.ldc;
        B.lds[n] = j.lds;
        B.bf16[n] = j.x_bf16 ? 1 : 0;
        acc += j.rows * (j.cols / 32) * 4;
        B.lanes_end[n] = acc;
        ++n;
    }
    if (n == 0) return cudaSuccess;
    B.n = n;
    for (int k = n; k < 4; ++k) B.lanes_end[k] = acc;
    return launch_pdl(quant_mxfp4_batch_kernel, dim3(grid_for(acc, 256)), dim3(256), 0, s, 1, B, d_status);
}

cudaError_t launch_quant_nvfp4(const void *x, bool x_bf16, int64_t rows, int64_t cols, int64_t ldx,
                               uint8_t *codes, int64_t ldc, uint8_t *scales, int64_t lds,
                               uint32_t *d_status, cudaStream_t s)
{
    if (rows == 0 || cols == 0) return cudaSuccess;
    const size_t esz = x_bf16 ? 2 : 4;
    const bool vec = ((uintptr_t)x % 16 == 0) && ((ldx * (int64_t)esz) % 16 == 0) &&
                     ((uintptr_t)codes % 4 == 0) && (ldc % 4 == 0);
    if (vec) {
        const int grid = grid_for(rows * (cols / 16) * 2, 256);
        if (x_bf16)
            return launch_pdl(quant_nvfp4_vec_kernel<true>, dim3(grid), dim3(256), 0, s, 1, x, rows, cols, ldx,
                              codes, ldc, scales, lds, d_status);
        return launch_pdl(quant_nvfp4_vec_kernel<false>, dim3(grid), dim3(256), 0, s, 1, x, rows, cols, ldx,
                          codes, ldc, scales, lds, d_status);
    }
    const int grid = grid_for(rows * (cols / 16), 16);
    if (x_bf16)
        quant_nvfp4_kernel<true><<<grid, 256, 0, s>>>(x, rows, cols, ldx, codes, ldc, scales, lds, d_status);
    else
        quant_nvfp4_kernel<false><<<grid, 256, 0, s>>>(x, rows, cols, ldx, codes, ldc, scales, lds, d_status);
    return cudaGetLastError();
}

cudaError_t launch_rope_quant(const RopeQuantJobDesc *jobs, int n_jobs, uint32_t *d_status, cudaStream_t s)
{
    if (n_jobs < 1 || n_jobs > 4) return cudaErrorInvalidValue;
    RopeQuantParams B = {};
    int64_t acc = 0;
    int n = 0;
    for (int k = 0; k < n_jobs; ++k) {
        const RopeQuantJobDesc &j = jobs[k];
        if (j.rows == 0 || j.cols == 0) continue;
        const int G = j.nvfp4 ? 16 : 32;
        B.x[n] = j.x;
        B.pos[n] = j.pos;
        B.cs[n] = j.cos_sin;
        B.codes[n] = j.codes;
        B.scales[n] = j.scales;
        B.cols[n] = j.cols;
        B.nblk[n] = j.cols / G;
        B.blocks[n] = j.rows * (j.cols / G);
        B.ldx[n] = j.ldx;
        B.ldc[n] = j.ldc;
        B.lds[n] = j.lds;
        B.n_pos[n] = j.n_pos;
        B.rope[n] = j.rope_dim;
        B.nv[n] = j.nvfp4 ? 1 : 0;
        acc += (B.blocks[n] * (G / 8) + 3) & ~int64_t(3);
        B.lanes_end[n] = acc;
        ++n;
    }
    if (n == 0) return cudaSuccess;
    B.n = n;
    for (int k = n; k < 4; ++k) B.lanes_end[k] = acc;
    return launch_pdl(rope_quant_kernel, dim3(grid_for(acc, 256)), dim3(256), 0, s, 1, B, d_status);
}

cudaError_t launch_quant_mxfp8(const void *x, bool x_bf16, int64_t rows, int64_t cols, int64_t ldx,
                               uint8_t *codes, int64_t ldc, uint8_t *scales, int64_t lds,
                               uint32_t *d_status, cudaStream_t s)
{
    if (rows == 0 || cols == 0) return cudaSuccess;
    const int grid = grid_for(rows * (cols / 32), 8);
    if (x_bf16)
        return launch_pdl(quant_mxfp8_kernel<true>, dim3(grid), dim3(256), 0, s, 1, x, rows, cols, ldx, codes,
                          ldc, scales, lds, d_status);
    return launch_pdl(quant_mxfp8_kernel<false>, dim3(grid), dim3(256), 0, s, 1, x, rows, cols, ldx, codes, ldc,
                      scales, lds, d_status);
}

cudaError_t launch_dequant_mxfp8(const uint8_t *codes, int64_t ldc, const uint8_t *scales, int64_t lds,
                                 int64_t rows, int64_t cols, void *y, bool y_bf16, int64_t ldy, cudaStream_t s)
{
    if (rows == 0 || cols == 0) return cudaSuccess;
    const int grid = grid_for(rows * cols, 256);
    if (y_bf16) dequant_mxfp8_kernel<true><<<grid, 256, 0, s>>>(codes, ldc, scales, lds, rows, cols, y, ldy);
    else dequant_mxfp8_kernel<false><<<grid, 256, 0, s>>>(codes, ldc, scales, lds, rows, cols, y, ldy);
    return cudaGetLastError();
}

cudaError_t launch_dequant_fp4(const uint8_t *codes, int64_t ldc, const uint8_t *scales,
                               int64_t lds, int64_t rows, int64_t cols, bool nvfp4, void *y,
                               bool y_bf16, int64_t ldy, cudaStream_t s)
{
    if (rows == 0 || cols == 0) return cudaSuccess;
    const int grid = grid_for(rows * cols, 256);
    if (nvfp4) {
        if (y_bf16)
            dequant_fp4_kernel<true, true><<<grid, 256, 0, s>>>(codes, ldc, scales, lds, rows, cols, y, ldy);
        else
            dequant_fp4_kernel<false, true><<<grid, 256, 0, s>>>(codes, ldc, scales, lds, rows, cols, y, ldy);
    } else {
        if (y_bf16)
            dequant_fp4_kernel<true, false><<<grid, 256, 0, s>>>(codes, ldc, scales, lds, rows, cols, y, ldy);
        else
            dequant_fp4_kernel<false, false><<<grid, 256, 0, s>>>(codes, ldc, scales, lds, rows, cols, y, ldy);
    }
    return cudaGetLastError();
}

} // namespace csa2
