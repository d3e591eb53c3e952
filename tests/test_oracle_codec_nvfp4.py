"""Pins of the oracle's E2M1 + E4M3/16 main-KV codec (CPU only).

The report (DeepSeek-V4.1-Flash, aipaper.jasonlin.tech, §2.4.4) stores the main KV as
E2M1 values with an E4M3 scale per 16 and no global scale; the review page's byte
ledger ("四位缓存") counts 256 B of codes and 32 B of scales for 512 channels.  How a
block's scale is chosen is not stated: the oracle maps the block maximum onto 6, the
largest E2M1 value, rounding amax/6 to the nearest E4M3 value.

Pins: E4M3 decoding of all 256 bytes against PyTorch's float8_e4m3fn (a library
routine), the scale rounding against PyTorch's float32 -> float8_e4m3fn conversion at
every E4M3 rounding boundary, a Fraction brute-force quantiser on random blocks,
hand-derived tie cases, the zero-scale and saturation edges, exhaustive dequantisation.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import tiny
from fp4_kv_cache_gb300 import synth

torch = pytest.importorskip("torch")


def _pack(codes):
    codes = np.asarray(codes, np.uint8)
    return (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)


def _torch_e4m3(byte_values):
    b = torch.tensor(np.asarray(byte_values, np.uint8))
    return b.view(torch.float8_e4m3fn).float().numpy().astype(np.float64)


def test_e4m3_decode_all_bytes_matches_library():
    # code 2 (value 1.0) in every element, so y = the scale's value
    codes = _pack([2] * 16)[None]
    ref = _torch_e4m3(range(256))
    for sb in range(256):
        y = oracle.dequant_nvfp4(codes, np.array([[sb]], np.uint8))[0]
        if np.isnan(ref[sb]):
            assert sb & 0x7F == 0x7F and np.all(np.isnan(y))
            assert tiny.e4m3_value(sb) is None
        else:
            assert np.all(y == ref[sb]), sb
            assert Fraction(float(y[0])) == tiny.e4m3_value(sb)
    assert ref[0x7E] == 448.0 and ref[0x01] == 2.0 ** -9 and ref[0x08] == 2.0 ** -6


def _scale_byte(amax):
    x = np.zeros((1, 16))
    x[0, 3] = amax
    return int(oracle.quant_nvfp4(x)[1][0, 0])


def test_scale_rounding_matches_library_at_every_boundary():
    vals = _torch_e4m3(range(0x7F))            # finite non-negative E4M3 values, ascending
    assert np.all(np.diff(vals) > 0)
    amaxes = []
    for lo, hi in zip(vals[:-1], vals[1:]):
        mid6 = np.float32(6.0 * 0.5 * (lo + hi))   # exact: <= 7 significant bits
        for a in (np.nextafter(mid6, np.float32(0)), mid6, np.nextafter(mid6, np.float32(np.inf))):
            amaxes.append(a)
        amaxes.append(np.float32(6.0 * hi))
    amaxes += [np.float32(v) for v in (1e-30, 6 * 2.0 ** -10, 2687.9, 2688.0, 2784.0, 2785.0, 1e9)]
    n_checked = 0
    for a in amaxes:
        sb = _scale_byte(float(a))
        t32 = np.float32(a) / np.float32(6.0)    # IEEE division: the E4M3 decision it feeds
        if t32 <= 464.0:                         # the library rounds to nearest even there
            lib = int(torch.tensor([float(t32)], dtype=torch.float32)
                      .to(torch.float8_e4m3fn).view(torch.uint8)[0])
            assert sb == lib, (float(a), sb, lib)
            n_checked += 1
        else:                                    # library: NaN; this format clamps to 448
            assert sb == 0x7E
        # and the exact rational rule agrees
        assert sb == tiny.quant_block_nvfp4([Fraction(float(a))] + [Fraction(0)] * 15,
                                            [False] * 16)[0]
    assert n_checked > 3 * 125


def _random_blocks16(rng, n):
    rows = []
    for _ in range(n):
        e = rng.integers(-16, 14)
        v = rng.standard_normal(16).astype(np.float32) * np.float32(2.0 ** int(e))
        kind = rng.integers(0, 6)
        if kind == 0:
            v[rng.integers(0, 16, 3)] = 0.0
        elif kind == 1:
            v[rng.integers(0, 16, 3)] = -0.0
        elif kind == 2:
            v[:] = 0.0
            v[rng.integers(0, 16)] = -0.0
        elif kind == 3:
            v *= np.float32(2.0 ** float(rng.integers(-12, 12)))
        rows.append(synth.bf16_to_f32(synth.f32_to_bf16_bits(v)))
    return np.stack(rows)


def test_quant_matches_fraction_bruteforce():
    rng = np.random.default_rng(21)
    x = _random_blocks16(rng, 400)
    codes, scales = oracle.quant_nvfp4(x)
    for r in range(x.shape[0]):
        xs = [Fraction(float(v)) for v in x[r]]
        sb, cs = tiny.quant_block_nvfp4(xs, [bool(np.signbit(v)) for v in x[r]])
        assert scales[r, 0] == sb, r
        assert tiny.unpack_codes(codes[r]) == cs, r


def test_quant_fp32_rows_match_bruteforce():
    rng = np.random.default_rng(22)
    x = (rng.standard_normal((60, 48)) * 2.0 ** rng.integers(-12, 10, (60, 1))).astype(np.float32)
    codes, scales = oracle.quant_nvfp4(x.astype(np.float64))
    for r in range(x.shape[0]):
        for b in range(3):
            blk = x[r, 16 * b:16 * b + 16]
            sb, cs = tiny.quant_block_nvfp4([Fraction(float(v)) for v in blk],
                                            [bool(np.signbit(v)) for v in blk])
            assert scales[r, b] == sb
            assert tiny.unpack_codes(codes[r, 8 * b:8 * b + 8]) == cs


# element value / scale -> expected code (E2M1 grid, round-half-to-even on the code)
TIES = [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6),
        (0.3, 1), (0.74, 1), (0.76, 2), (2.6, 5), (4.9, 6), (5.1, 7)]


@pytest.mark.parametrize("scale_byte", [0x38, 0x3C, 0x4F, 0x03, 0x7E])
def test_known_answer_ties(scale_byte):
    s = tiny.e4m3_value(scale_byte)
    x = np.zeros(16, np.float64)
    x[0] = float(6 * s)                         # amax = 6 s: the scale is exactly s
    for i, (v, _) in enumerate(TIES):
        x[1 + i] = float(Fraction(v) * s) if v in (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0) \
            else v * float(s)
    codes, scales = oracle.quant_nvfp4(x[None])
    assert scales[0, 0] == scale_byte
    un = tiny.unpack_codes(codes[0])
    assert un[0] == 7
    for i, (v, c) in enumerate(TIES):
        assert un[1 + i] == c, (v, scale_byte)
    codes_n, _ = oracle.quant_nvfp4(-x[None])
    assert all(u == c | 8 for u, c in zip(tiny.unpack_codes(codes_n[0]), un))


def test_zero_scale_block_and_negative_zero():
    x = np.zeros((4, 16))
    x[1, :] = -0.0
    x[2, 0], x[2, 1] = 6 * 2.0 ** -10, -1e-4   # amax/6 = 2^-10: tie between 0 and 2^-9 -> 0
    x[3, 0] = 6 * 2.0 ** -10 * (1 + 2.0 ** -20)  # just above the tie -> smallest subnormal
    codes, scales = oracle.quant_nvfp4(x)
    assert list(scales[:, 0]) == [0, 0, 0, 1]
    assert np.all(codes[0] == 0) and np.all(codes[1] == 0x88)
    un = tiny.unpack_codes(codes[2])
    assert un[0] == 0 and un[1] == 8 and all(u == 0 for u in un[2:])
    assert tiny.unpack_codes(codes[3])[0] == 5            # x / 2^-9 = 3.0000... -> 3


def test_saturation_and_max_magnitude():
    x = np.zeros((1, 16))
    x[0, 0], x[0, 1] = 1e6, -2688.0
    codes, scales = oracle.quant_nvfp4(x)
    assert scales[0, 0] == 0x7E
    un = tiny.unpack_codes(codes[0])
    assert un[0] == 7 and un[1] == 15
    y = oracle.dequant_nvfp4(codes, scales)
    assert y[0, 0] == 6 * 448.0 and y[0, 1] == -2688.0   # report §2.4.4: 448 x 6 = 2688


def test_dequant_exhaustive_codes_and_scales():
    codes = np.array(list(range(16)), np.uint8)
    packed = _pack(codes)[None]
    for sb in range(256):
        if sb & 0x7F == 0x7F:
            continue
        y = oracle.dequant_nvfp4(packed, np.array([[sb]], np.uint8))[0]
        for i, c in enumerate(codes.tolist()):
            assert Fraction(float(y[i])) == tiny.e2m1_value(c) * tiny.e4m3_value(sb), (c, sb)


def test_dequant_is_exact_in_bf16():
    # every E2M1 x E4M3 product has at most 6 significant bits and lies in [2^-10, 2688]:
    # the bf16 rounding of each value is the value itself
    codes = np.array(list(range(16)), np.uint8)
    packed = _pack(codes)[None]
    for sb in range(0x7F):
        y = oracle.dequant_nvfp4(packed, np.array([[sb]], np.uint8))[0].astype(np.float32)
        back = synth.bf16_to_f32(synth.f32_to_bf16_bits(y))
        assert np.array_equal(back, y)


def test_main_kv_helpers_pick_the_format():
    rng = np.random.default_rng(3)
    x = synth.bf16_to_f32(synth.f32_to_bf16_bits(rng.standard_normal((5, 576)).astype(np.float32)))
    c1, s1 = oracle.quant_main_kv(x, "nvfp4")
    c2, s2 = oracle.quant_main_kv(x, "mxfp4")
    assert s1.shape == (5, 36) and s2.shape == (5, 18)
    assert np.array_equal(oracle.dequant_main_kv(c1, s1), oracle.dequant_nvfp4(c1, s1))
    assert np.array_equal(oracle.dequant_main_kv(c2, s2), oracle.dequant_mxfp4(c2, s2))
    # the per-16 scale is never coarser than a power of two: its error is no larger
    err16 = np.abs(oracle.dequant_nvfp4(c1, s1) - x).max()
    assert err16 <= np.abs(x).max() / 4
