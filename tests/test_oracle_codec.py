"""Pins of the oracle's MXFP4 codec against the format definition (CPU only).

The report (DeepSeek-V4.1-Flash, aipaper.jasonlin.tech, §2.4.4) names OCP MXFP4 for
the indexer; the OCP rule fixes the scale X = floor(log2 amax) - 2 and RNE element
rounding with saturation.  Pins: the golden code table, exhaustive code x scale
dequantisation against an independent Fraction evaluation, hand-derived tie cases,
a Fraction brute-force quantiser, idempotence, saturation, zero and -0 blocks.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import tiny
from fp4_kv_cache_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_codes():
    out = {}
    for line in open(os.path.join(GOLDEN, "e2m1_code_values.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        c, v = line.split()
        out[int(c)] = v
    return out


def _pack(codes):
    codes = np.asarray(codes, np.uint8)
    return (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)


def test_golden_code_table():
    g = _golden_codes()
    for c in range(16):
        codes = _pack([c] * 32)
        y = oracle.dequant_mxfp4(codes[None], np.array([[127]], np.uint8))[0]
        expect = float(g[c])
        assert y[0] == expect and np.signbit(y[0]) == g[c].startswith("-")
        assert tiny.e2m1_value(c) == Fraction(g[c])


def test_dequant_exhaustive_codes_and_scales():
    codes = np.array(list(range(16)) * 2, np.uint8)
    packed = _pack(codes)
    for e in range(0, 255):
        y = oracle.dequant_mxfp4(packed[None], np.array([[e]], np.uint8))[0]
        for i, c in enumerate(codes.tolist()):
            exact = tiny.e2m1_value(c) * Fraction(2) ** (e - 127)
            assert y[i] == float(exact), (c, e)
            assert np.signbit(y[i]) == bool(c & 8)


# element value / 2^X -> expected code, by the E2M1 grid and round-half-to-even
TIES = [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6),
        (0.2, 0), (0.3, 1), (0.74, 1), (0.76, 2), (1.3, 3), (2.4, 4), (2.6, 5),
        (3.4, 5), (3.6, 6), (4.9, 6), (5.1, 7), (6.0, 7), (7.5, 7)]


@pytest.mark.parametrize("X", [-127, -20, -1, 0, 3, 60])
def test_known_answer_ties(X):
    # element 0 fixes amax = 4 * 2^X (floor(log2) = X + 2, so the scale is exactly X),
    # except where a tie value above is larger; use 7.75*2^X then (still floor(log2)=X+2)
    x = np.zeros(32, np.float64)
    x[0] = 7.75 * 2.0 ** X
    for i, (v, _) in enumerate(TIES):
        x[1 + i] = v * 2.0 ** X
    codes, scales = oracle.quant_mxfp4(x[None])
    assert scales[0, 0] == X + 127
    unpacked = tiny.unpack_codes(codes[0])
    assert unpacked[0] == 7          # 7.75 saturates to 6
    for i, (v, c) in enumerate(TIES):
        assert unpacked[1 + i] == c, (v, X)
    # negated block: same magnitudes, sign bit set
    codes_n, _ = oracle.quant_mxfp4(-x[None])
    un = tiny.unpack_codes(codes_n[0])
    assert all(u == c | 8 for u, c in zip(un, unpacked))


def _random_blocks(rng, n):
    """bf16-valued blocks with a wide spread of magnitudes, zeros and -0."""
    rows = []
    for _ in range(n):
        e = rng.integers(-140, 105)
        v = rng.standard_normal(32).astype(np.float32) * np.float32(2.0 ** int(e))
        kind = rng.integers(0, 6)
        if kind == 0:
            v[rng.integers(0, 32, 5)] = 0.0
        elif kind == 1:
            v[rng.integers(0, 32, 5)] = -0.0
        elif kind == 2:
            v[:] = 0.0
            v[rng.integers(0, 32)] = -0.0
        elif kind == 3:
            v *= np.float32(2.0 ** float(rng.integers(-10, 10)))
        rows.append(synth.bf16_to_f32(synth.f32_to_bf16_bits(v)))
    return np.stack(rows)


def test_quant_matches_fraction_bruteforce():
    rng = np.random.default_rng(11)
    x = _random_blocks(rng, 300)
    codes, scales = oracle.quant_mxfp4(x)
    for r in range(x.shape[0]):
        xs = [Fraction(float(v)) for v in x[r]]
        sb, cs = tiny.quant_block(xs, [bool(np.signbit(v)) for v in x[r]])
        assert scales[r, 0] == sb
        assert tiny.unpack_codes(codes[r]) == cs


def test_quant_fp32_subnormal_and_huge():
    x = np.zeros((3, 32), np.float64)
    x[0, :] = np.float32(1e-45)                 # smallest fp32 subnormal: X clamps at -127
    x[1, 0] = float(np.finfo(np.float32).max)   # X = 125
    x[2, 3] = -float(np.finfo(np.float32).tiny)
    codes, scales = oracle.quant_mxfp4(x)
    for r in range(3):
        xs = [Fraction(float(v)) for v in x[r]]
        sb, cs = tiny.quant_block(xs, [bool(np.signbit(v)) for v in x[r]])
        assert scales[r, 0] == sb and tiny.unpack_codes(codes[r]) == cs
    assert scales[0, 0] == 0 and scales[1, 0] == 125 + 127


def test_idempotent_roundtrip():
    rng = np.random.default_rng(5)
    x = _random_blocks(rng, 500)
    c1, s1 = oracle.quant_mxfp4(x)
    y = oracle.dequant_mxfp4(c1, s1)
    c2, s2 = oracle.quant_mxfp4(y)
    # values are reproduced exactly, always
    assert np.array_equal(oracle.dequant_mxfp4(c2, s2), y)
    # codes and scales too, for every block with a nonzero code: its scale X puts the
    # block maximum at code 6 or 7, so requantising finds the same X.  A block whose
    # scale clamped at 2^-127 can round to all zeros and then takes the zero-block scale.
    nonzero = np.any((c1 & 0x77) != 0, axis=1)
    assert nonzero.sum() > 300
    assert np.array_equal(c1[nonzero], c2[nonzero]) and np.array_equal(s1[nonzero], s2[nonzero])


def test_zero_block_and_negative_zero():
    x = np.zeros((2, 32))
    x[1, :] = -0.0
    codes, scales = oracle.quant_mxfp4(x)
    assert list(scales[:, 0]) == [127, 127]
    assert np.all(codes[0] == 0) and np.all(codes[1] == 0x88)


def test_max_magnitude():
    # largest finite MXFP4 value: code 7 (6) at scale byte 254 -> 6 * 2^127
    y = oracle.dequant_mxfp4(np.full((1, 16), 0x77, np.uint8), np.array([[254]], np.uint8))
    assert y[0, 0] == 6.0 * 2.0 ** 127
