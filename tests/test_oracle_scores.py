"""Pins of the oracle's indexer score (CPU only).

Score (the workload definition; the report, aipaper.jasonlin.tech §2.3, says only that
the indexer scores main-KV entries from indexer Q and indexer K):
    s = sum_h w_h * ReLU(q_h . k)
with q, k MXFP4 (report §2.4.4), each head dot rounded once to float32 and the head
sum a float32 fma chain (or, for the prefill-chunk kernel, eight partial chains over the
heads h = j mod 8 added in a fixed tree).  Pins: an exact Fraction brute force on tiny inputs
(typical and extreme scales, so both the double path and the wide-integer path of the
C oracle run), hand-derived rounding cases where a tiny term breaks a tie, and the
textbook case H = 1, w = 1 where the score is the plain dot product.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import tiny
from fp4_kv_cache_gb300 import synth


def _rand_mx(rng, rows, d, scale_lo, scale_hi):
    codes = rng.integers(0, 256, size=(rows, d // 2), dtype=np.uint8)
    scales = rng.integers(scale_lo, scale_hi + 1, size=(rows, d // 32)).astype(np.uint8)
    return codes, scales


@pytest.mark.parametrize("H,d,lo,hi,seed", [
    (1, 32, 120, 134, 0), (4, 64, 120, 134, 1), (3, 96, 110, 140, 2),
    (2, 64, 0, 254, 3), (4, 128, 0, 254, 4), (2, 128, 60, 200, 5)])
def test_scores_match_fraction_bruteforce(H, d, lo, hi, seed):
    rng = np.random.default_rng(seed)
    N = 20
    kc, ks = _rand_mx(rng, N, d, lo, hi)
    qc, qs = _rand_mx(rng, H, d, lo, hi)
    w = rng.standard_normal(H).astype(np.float32)
    w[0] = abs(w[0])
    if H > 2:
        w[2] = 0.0
    pos = np.arange(N, dtype=np.int64)
    got = oracle.index_scores(qc, qs, w, kc, ks, pos)
    got8 = oracle.index_scores(qc, qs, w, kc, ks, pos, order="split8")
    dots = oracle.head_dots(qc, qs, kc, ks, pos)
    for t in range(N):
        for g, order in ((got, "chain"), (got8, "split8")):
            exp = np.float32(tiny.score(qc, qs, w, kc[t], ks[t], order))
            if np.isnan(exp):
                assert np.isnan(g[t])            # NaN payloads differ between platforms
            else:
                assert g[t].view(np.uint32) == exp.view(np.uint32), (order, t, g[t], exp)
        kv = tiny.exact_vector(kc[t], ks[t])
        for h in range(H):
            qv = tiny.exact_vector(qc[h], qs[h])
            D = tiny.rn32(sum((a * b for a, b in zip(qv, kv)), Fraction(0)))
            assert dots[t, h].view(np.uint32) == np.float32(D).view(np.uint32)


def _one_hot_block_row(vals):
    """Per block: a single element of code `c` at position 0 (others +0)."""
    d = 32 * len(vals)
    codes = np.zeros(d, np.uint8)
    for b, c in enumerate(vals):
        codes[32 * b] = c
    return (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)


@pytest.mark.parametrize("sign_tiny,tiny_exp,expect", [
    (+1, -200, 2.0 ** 30 + 2.0 ** 7),   # wide-integer path: sticky bit rounds the tie up
    (-1, -200, 2.0 ** 30),              # negative tiny term: below the midpoint
    (+1, -2, 2.0 ** 30 + 2.0 ** 7),     # double path (span 32)
    (0, 0, 2.0 ** 30),                  # exact midpoint, ties to even
])
def test_rounding_tie_broken_by_tiny_term(sign_tiny, tiny_exp, expect):
    # three blocks, one product each: 2^30 + 2^6 + sign * 2^tiny_exp.  2^30 + 2^6 is the
    # midpoint between float32 neighbours 2^30 and 2^30 + 2^7.  A product of codes 2 and 2
    # (1 x 1) in a block with scale bytes (a, b) is 2^(a-127 + b-127).
    q_codes = [2, 2, 10 if sign_tiny < 0 else (2 if sign_tiny > 0 else 0)]
    qc = _one_hot_block_row(q_codes)[None]
    kc = _one_hot_block_row([2, 2, 2])[None]
    qs = np.array([[127 + 30, 127 + 6, 127]], np.uint8)
    ks = np.array([[127, 127, 127 + tiny_exp]], np.uint8) if tiny_exp >= -127 else \
        np.array([[127, 127, 0]], np.uint8)
    if tiny_exp < -127:
        qs[0, 2] = 127 + tiny_exp + 127
    D = oracle.head_dots(qc, qs, kc, ks, np.array([0]))[0, 0]
    assert float(D) == expect
    s = oracle.index_scores(qc, qs, np.array([1.0], np.float32), kc, ks, np.array([0]))[0]
    assert float(s) == expect


def test_textbook_single_head_dot():
    # H = 1, w = 1 and a positive dot: the score is the plain dot product of the
    # dequantised vectors (numpy float64 dot, exact here, then float32).
    rng = np.random.default_rng(7)
    d, N = 128, 64
    k = synth.bf16_to_f32(synth.f32_to_bf16_bits(rng.standard_normal((N, d)).astype(np.float32)))
    q = synth.bf16_to_f32(synth.f32_to_bf16_bits(rng.standard_normal((1, d)).astype(np.float32)))
    kc, ks = oracle.quant_mxfp4(k)
    qc, qs = oracle.quant_mxfp4(q)
    kd = oracle.dequant_mxfp4(kc, ks)
    qd = oracle.dequant_mxfp4(qc, qs)[0]
    s = oracle.index_scores(qc, qs, np.array([1.0], np.float32), kc, ks, np.arange(N))
    ref = kd @ qd
    checked = 0
    for t in range(N):
        if ref[t] > 0:
            assert np.float64(np.float32(ref[t])) == ref[t]       # representable here
            assert s[t] == np.float32(ref[t])
            checked += 1
        else:
            assert s[t] == 0.0
    assert checked > 10
    # w = (1, 0) on two heads with the same query row: the second head drops out
    q2c, q2s = np.repeat(qc, 2, 0), np.repeat(qs, 2, 0)
    s2 = oracle.index_scores(q2c, q2s, np.array([1.0, 0.0], np.float32), kc, ks, np.arange(N))
    assert np.array_equal(s2, s)


def test_head_weight_power_of_two_scaling():
    # scaling every w_h by 2 doubles every score exactly (no rounding changes)
    rng = np.random.default_rng(8)
    kc, ks = _rand_mx(rng, 50, 128, 122, 130)
    qc, qs = _rand_mx(rng, 8, 128, 122, 130)
    w = rng.random(8).astype(np.float32)
    pos = np.arange(50)
    s1 = oracle.index_scores(qc, qs, w, kc, ks, pos)
    s2 = oracle.index_scores(qc, qs, w * np.float32(2), kc, ks, pos)
    assert np.array_equal(s2, s1 * np.float32(2))


def test_visibility_rule():
    # ratio m: entry j covers tokens [j*m, j*m+m-1]; only complete entries are visible
    assert oracle.n_visible(4095, 1, 4096) == 4096
    assert oracle.n_visible(0, 1, 10) == 1
    assert oracle.n_visible(0, 2, 10) == 0
    assert oracle.n_visible(1, 2, 10) == 1
    assert oracle.n_visible(131072, 2, 67584) == 65536
    assert oracle.n_visible(135167, 2, 67584) == 67584
    assert oracle.n_visible(10 ** 9, 1, 77) == 77
