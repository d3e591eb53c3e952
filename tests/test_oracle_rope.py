"""Pins of the oracle's RoPE-before-quantisation step (CPU only).

Report §2.4.4 (DeepSeek-V4.1-Flash, aipaper.jasonlin.tech): the main-KV cache is quantised
after RoPE, and the RoPE and non-RoPE channels share one format.  The pages print no RoPE
formula, so the rotation is pinned by what a rotation must satisfy: the identity and
quarter-turn special cases, pair locality (only the trailing rope_dim channels, and only
within a pair), norm preservation, composition of angles against an fp64 rotation, and
the float32 rounding rule (one rounding per product and per sum) on exact cases.
"""
import numpy as np
import pytest

import oracle
from fp4_kv_cache_gb300 import synth


def _table(n_pos, rope_dim, base=10000.0):
    """Synthetic RoPE table [n_pos, rope_dim]: cosines then sines of p * base^(-2i/R)."""
    i = np.arange(rope_dim // 2, dtype=np.float64)
    ang = np.arange(n_pos, dtype=np.float64)[:, None] * base ** (-2.0 * i / rope_dim)[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def _rows(rng, n, cols):
    return synth.bf16_to_f32(synth.f32_to_bf16_bits(rng.standard_normal((n, cols)).astype(np.float32)))


def test_identity_and_quarter_turn():
    rng = np.random.default_rng(0)
    x = _rows(rng, 5, 96)
    R = 32
    ident = np.concatenate([np.ones((1, R // 2)), np.zeros((1, R // 2))], axis=1).astype(np.float32)
    quarter = np.concatenate([np.zeros((1, R // 2)), np.ones((1, R // 2))], axis=1).astype(np.float32)
    pos = np.zeros(5, np.int64)
    assert np.array_equal(oracle.rope_rotate(x, pos, ident, R), x)
    y = oracle.rope_rotate(x, pos, quarter, R)
    c0 = 96 - R
    assert np.array_equal(y[:, :c0], x[:, :c0])
    assert np.array_equal(y[:, c0::2], -x[:, c0 + 1::2])      # (a, b) -> (-b, a)
    assert np.array_equal(y[:, c0 + 1::2], x[:, c0::2])


def test_pair_locality():
    R, cols = 64, 576
    tab = _table(50, R)
    for ch in (0, 511, 512, 513, 574, 575):
        x = np.zeros((1, cols), np.float32)
        x[0, ch] = 1.0
        y = oracle.rope_rotate(x, np.array([37]), tab, R)
        changed = set(np.nonzero(y[0])[0].tolist())
        if ch < cols - R:
            assert changed == {ch} and y[0, ch] == 1.0
        else:
            first = ch - (ch - (cols - R)) % 2                 # the pair's even channel
            assert changed and changed <= {first, first + 1}


def test_norm_preserved_and_composition():
    rng = np.random.default_rng(1)
    R, cols, n = 64, 128, 200
    x = _rows(rng, n, cols)
    theta = rng.uniform(-np.pi, np.pi, (n, R // 2))
    def tab_of(th):
        return np.concatenate([np.cos(th), np.sin(th)], axis=1).astype(np.float32)
    pos = np.arange(n)
    y = oracle.rope_rotate(x, pos, tab_of(theta), R)
    c0 = cols - R
    n_in = x[:, c0::2] ** 2 + x[:, c0 + 1::2] ** 2
    n_out = y[:, c0::2].astype(np.float64) ** 2 + y[:, c0 + 1::2].astype(np.float64) ** 2
    assert np.allclose(n_out, n_in, rtol=2e-6, atol=1e-30)
    # rotating by theta1 then theta2 matches an fp64 rotation by theta1 + theta2
    theta2 = rng.uniform(-np.pi, np.pi, (n, R // 2))
    z = oracle.rope_rotate(y, pos, tab_of(theta2), R)
    a, b = x[:, c0::2].astype(np.float64), x[:, c0 + 1::2].astype(np.float64)
    t = theta + theta2
    assert np.allclose(z[:, c0::2], a * np.cos(t) - b * np.sin(t), atol=1e-5)
    assert np.allclose(z[:, c0 + 1::2], a * np.sin(t) + b * np.cos(t), atol=1e-5)


def test_float32_rounding_rule():
    # a*c - b*s with products that are not float32-exact: one rounding per product, one per
    # difference (a fused multiply-add would give a different bit pattern here)
    a = np.float32(1.0 + 2.0 ** -23)
    c = np.float32(1.0 - 2.0 ** -24)
    b = np.float32(1.0)
    s = np.float32(1.0 - 2.0 ** -23)
    x = np.array([[a, b]], np.float32)
    tab = np.array([[c, s]], np.float32)
    y = oracle.rope_rotate(x, np.array([0]), tab, 2)
    p1 = np.float32(np.float64(a) * np.float64(c))          # exact product, rounded once
    p2 = np.float32(np.float64(b) * np.float64(s))
    assert y[0, 0] == np.float32(np.float64(p1) - np.float64(p2))
    fused = np.float32(np.float64(a) * np.float64(c) - np.float64(p2))
    assert y[0, 0] != fused                                  # the case separates the two rules


@pytest.mark.parametrize("fmt", ["mxfp4", "nvfp4"])
def test_rope_quant_is_quant_of_rotated(fmt):
    rng = np.random.default_rng(2)
    x = _rows(rng, 40, 576)
    tab = _table(1000, 64)
    pos = rng.integers(0, 1000, 40)
    c, s = oracle.rope_quant(x, pos, tab, 64, fmt)
    y = oracle.rope_rotate(x, pos, tab, 64)
    c2, s2 = oracle.quant_main_kv(y.astype(np.float64), fmt)
    assert np.array_equal(c, c2) and np.array_equal(s, s2)
    # non-RoPE channels' blocks are those of the plain quantiser
    g = 32 if fmt == "mxfp4" else 16
    c3, s3 = oracle.quant_main_kv(x.astype(np.float64), fmt)
    nb = (576 - 64) // g
    assert np.array_equal(s[:, :nb], s3[:, :nb]) and np.array_equal(c[:, : nb * g // 2], c3[:, : nb * g // 2])


def test_rounding_rule_against_exact_rationals():
    # every rotated value is RN32(RN32(a c) -/+ RN32(b s)), evaluated here with exact
    # rationals and the brute-force float32 rounding of oracle/tiny.py
    from fractions import Fraction
    from oracle import tiny
    rng = np.random.default_rng(9)
    R, cols, n = 8, 24, 40
    x = _rows(rng, n, cols) * np.float32(2.0) ** rng.integers(-30, 30, (n, 1)).astype(np.float32)
    tab = _table(64, R)
    pos = rng.integers(0, 64, n)
    y = oracle.rope_rotate(x, pos, tab, R)
    c0 = cols - R
    for r in range(n):
        for i in range(R // 2):
            a, b = Fraction(float(x[r, c0 + 2 * i])), Fraction(float(x[r, c0 + 2 * i + 1]))
            c, s = Fraction(float(tab[pos[r], i])), Fraction(float(tab[pos[r], R // 2 + i]))
            ac, bs = tiny.rn32(a * c), tiny.rn32(b * s)
            as_, bc = tiny.rn32(a * s), tiny.rn32(b * c)
            assert y[r, c0 + 2 * i] == tiny.rn32(Fraction(float(ac)) - Fraction(float(bs)))
            assert y[r, c0 + 2 * i + 1] == tiny.rn32(Fraction(float(as_)) + Fraction(float(bc)))
