"""Pins of the oracle's MXFP8 (E4M3 + E8M0 per 32) SWA codec (CPU only).

Report (aipaper.jasonlin.tech) §2.4.4 keeps the SWA KV cache in FP8 because it is sensitive
to quantisation; the pages name no FP8 layout.  The reading (include/csa2.h,
csa2_swa_format): OCP MX v1.0 with E4M3 elements -- one E8M0 scale per 32 values,
X = floor(log2 amax) - 8, elements rounded to the nearest E4M3 value with ties to the even
code, saturating at 448, sign bit kept.  Pins: the E4M3 decode of every byte against
PyTorch's float8_e4m3fn; the quantiser against a Fraction brute force on random blocks
(subnormal elements, zeros, -0, wide scales) and against PyTorch's float8_e4m3fn rounding
of the scaled block; hand-derived ties and saturation; idempotence; exactness in bf16.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import tiny
from fp4_kv_cache_gb300 import synth


def test_e4m3_decode_every_byte_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = oracle.dequant_mxfp8(np.tile(codes[None, :], (1, 1))[:, :256].reshape(8, 32),
                               np.full((8, 1), 127, np.uint8)).reshape(-1)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2          # 0x7F and 0xFF
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[1] == 2.0 ** -9


def _frac_block(row):
    return [Fraction(float(v)) for v in row], [bool(np.signbit(v)) for v in row]


@pytest.mark.parametrize("seed,lo,hi", [(0, -4, 4), (1, -30, 30), (2, -126, 100), (3, -140, -120)])
def test_quantiser_matches_fraction_bruteforce(seed, lo, hi):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((24, 32)).astype(np.float32)
    x *= np.exp2(rng.integers(lo, hi + 1, size=(24, 1))).astype(np.float32)
    x[0] = 0.0
    x[1, :16] = -0.0
    x[2, ::5] *= np.float32(2.0 ** -14)                   # elements far below the block maximum
    x = synth.bf16_to_f32(synth.f32_to_bf16_bits(x))
    codes, scales = oracle.quant_mxfp8(x)
    for r in range(x.shape[0]):
        sb, c = tiny.quant_block_mxfp8(*_frac_block(x[r]))
        assert scales[r, 0] == sb, r
        assert list(codes[r]) == c, r


def test_quantiser_matches_torch_rounding_of_the_scaled_block():
    # library special case: with X fixed, each element below 448 * 2^X is
    # float8_e4m3fn(x / 2^X) (torch rounds to nearest even); the others saturate to +-448
    rng = np.random.default_rng(5)
    x = rng.standard_normal((200, 32)).astype(np.float32) * np.float32(37.0)
    codes, scales = oracle.quant_mxfp8(x)
    X = scales.astype(np.int64) - 127
    scaled = x / np.exp2(X).astype(np.float32)
    small = np.abs(scaled) < 448.0
    assert small.mean() > 0.9 and (~small).sum() > 0
    ref = torch.from_numpy(np.where(small, scaled, 0)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes[small], ref[small])
    assert np.all(codes[~small] & 0x7F == 0x7E)


def test_ties_and_saturation():
    # X = 0 (block maximum in [256, 512)); midpoints between neighbours go to the even code
    x = np.zeros((1, 32), np.float64)
    x[0, 0] = 300.0                       # fixes X = 0
    x[0, 1] = 1.0625                      # between 1.0 (0x38) and 1.125 (0x39): even -> 1.0
    x[0, 2] = 1.1875                      # between 1.125 (0x39) and 1.25 (0x3A): even -> 1.25
    x[0, 3] = -2.0 ** -10                 # half the smallest subnormal: ties to 0, sign kept
    x[0, 4] = 3.0 * 2.0 ** -10            # between 2^-9 (0x01) and 2^-8 (0x02): even -> 2^-8
    x[0, 5] = 440.0                       # between 416 (0x7D) and 448 (0x7E): even -> 448
    x[0, 6] = 432.0                       # midpoint of 416 and 448: even code 0x7E
    x[0, 7] = 300.0
    codes, scales = oracle.quant_mxfp8(x)
    assert scales[0, 0] == 127
    assert list(codes[0, 1:7]) == [0x38, 0x3A, 0x80, 0x02, 0x7E, 0x7E]
    # saturation: a block maximum of 500 has X = 0 and saturates to 448
    y = np.zeros((1, 32), np.float64)
    y[0, 0], y[0, 1] = 500.0, -511.0
    c2, s2 = oracle.quant_mxfp8(y)
    assert s2[0, 0] == 127 and c2[0, 0] == 0x7E and c2[0, 1] == 0xFE
    assert oracle.dequant_mxfp8(c2, s2)[0, 0] == 448.0
    # an all-zero block gets X = 0 and zero codes (with the sign bits of the inputs)
    z = np.zeros((1, 32), np.float64)
    z[0, 3] = -0.0
    c3, s3 = oracle.quant_mxfp8(z)
    assert s3[0, 0] == 127 and c3[0, 3] == 0x80 and np.all(np.delete(c3[0], 3) == 0)


def test_idempotent_and_exact_in_bf16():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((300, 64)) * np.exp2(rng.integers(-20, 20, size=(300, 1)))
    c, s = oracle.quant_mxfp8(x)
    y = oracle.dequant_mxfp8(c, s)
    c2, s2 = oracle.quant_mxfp8(y)
    assert np.array_equal(c2, c) and np.array_equal(s2, s)
    y32 = y.astype(np.float32)
    assert np.array_equal(y32.astype(np.float64), y)                      # exact in float32
    assert np.all(y32.view(np.uint32) & 0xFFFF == 0)                       # and in bf16
