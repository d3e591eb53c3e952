"""Brute-force exact reference for tiny inputs (TEST INFRASTRUCTURE).

Written independently of ``csa2_oracle.c`` with Python ``fractions.Fraction`` so
that it can pin the C oracle: every value here is an exact rational, every
rounding an explicit integer round-half-even.  Slow by design: only for inputs
of a few dozen positions.

Format facts used (DeepSeek-V4.1-Flash report, aipaper.jasonlin.tech, §2.4.4:
indexer queries and keys in OCP MXFP4; main KV in E2M1 with an E4M3 scale per 16):
E2M1 = 1 sign bit, 2 exponent bits with bias 1, 1 mantissa bit; E8M0 scale =
2^(byte - 127); blocks of 32.  E4M3 = 1 sign bit, 4 exponent bits with bias 7,
3 mantissa bits, no infinities, 0x7F/0xFF NaN; blocks of 16.
"""
from __future__ import annotations

from fractions import Fraction
from typing import List, Sequence

import numpy as np

TWO = Fraction(2)


def e2m1_value(code: int) -> Fraction:
    """Value of a 4-bit E2M1 code from its bit fields."""
    s = -1 if code & 8 else 1
    e = (code >> 1) & 3
    m = code & 1
    if e == 0:
        mag = Fraction(m, 2)                       # subnormal: 0.m * 2^(1-1)
    else:
        mag = (1 + Fraction(m, 2)) * TWO ** (e - 1)
    return s * mag


def floor_log2(a: Fraction) -> int:
    """Largest k with 2^k <= a (a > 0)."""
    k = a.numerator.bit_length() - a.denominator.bit_length()
    while TWO ** k > a:
        k -= 1
    while TWO ** (k + 1) <= a:
        k += 1
    return k


def quant_block(xs: Sequence[Fraction], signs: Sequence[bool]):
    """OCP MXFP4 of one block of 32 exact values -> (scale byte, [codes]).

    ``signs`` carries the sign bit of each input (so -0.0 keeps it)."""
    amax = max(abs(x) for x in xs)
    X = 0 if amax == 0 else min(127, max(-127, floor_log2(amax) - 2))
    codes = []
    grid = [abs(e2m1_value(c)) for c in range(8)]
    for x, neg in zip(xs, signs):
        v = abs(x) / TWO ** X
        if v >= 6:
            c = 7
        else:
            best = min(range(8), key=lambda c: (abs(v - grid[c]), c % 2))   # ties -> even code
            c = best
        codes.append(c | (8 if neg else 0))
    return X + 127, codes


def e4m3_value(byte: int):
    """Value of an E4M3 byte from its bit fields (None for the NaN codes)."""
    e, m = (byte >> 3) & 15, byte & 7
    if e == 15 and m == 7:
        return None
    mag = Fraction(m, 8) * TWO ** -6 if e == 0 else (1 + Fraction(m, 8)) * TWO ** (e - 7)
    return -mag if byte & 0x80 else mag


def quant_block_nvfp4(xs: Sequence[Fraction], signs: Sequence[bool]):
    """One block of 16 exact values in E2M1 + E4M3 -> (scale byte, [codes]).

    Scale: the finite non-negative E4M3 value nearest to amax/6 (ties to the even
    code; beyond 448 the nearest is 448).  Elements: the E2M1 magnitude nearest to
    |x|/scale (ties to the even code), all zero when the scale is 0."""
    amax = max(abs(x) for x in xs)
    t = amax / 6
    sb = min(range(0x7F), key=lambda c: (abs(t - e4m3_value(c)), c % 2))
    s = e4m3_value(sb)
    grid = [abs(e2m1_value(c)) for c in range(8)]
    codes = []
    for x, neg in zip(xs, signs):
        if s == 0:
            c = 0
        else:
            v = abs(x) / s
            c = min(range(8), key=lambda c: (abs(v - grid[c]), c % 2))
        codes.append(c | (8 if neg else 0))
    return sb, codes


def rn32(x: Fraction) -> np.float32:
    """Round an exact rational to float32 (nearest, ties to even; subnormals; inf)."""
    if x == 0:
        return np.float32(0.0)
    neg = x < 0
    a = -x if neg else x
    e = floor_log2(a)
    q = max(e, -126) - 23                           # weight of the last kept bit
    scaled = a / TWO ** q
    n = scaled.numerator // scaled.denominator
    rem = scaled - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    val = n * TWO ** q
    if val >= TWO ** 128:
        f = np.float32(np.inf)
    else:
        f = np.float32(float(val))                  # exactly representable
    return -f if neg else f


def fma32(a: np.float32, b: np.float32, c: np.float32) -> np.float32:
    """float32 fused multiply-add: one rounding of the exact a*b + c.

    Infinite or NaN operands give the IEEE special result (no rounding involved)."""
    if not (np.isfinite(a) and np.isfinite(b) and np.isfinite(c)):
        with np.errstate(invalid="ignore", over="ignore"):
            return np.float32(np.float64(a) * np.float64(b) + np.float64(c))
    return rn32(Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c)))


def dequant(codes: List[int], scale_byte: int) -> List[Fraction]:
    sc = TWO ** (scale_byte - 127)
    return [e2m1_value(c) * sc for c in codes]


def unpack_codes(packed: np.ndarray) -> List[int]:
    """uint8 [D/2] -> D codes, element 2i from the low nibble."""
    out = []
    for byte in packed.tolist():
        out.append(byte & 15)
        out.append(byte >> 4)
    return out


def exact_vector(codes_packed: np.ndarray, scales: np.ndarray) -> List[Fraction]:
    codes = unpack_codes(codes_packed)
    vals = []
    for b, sb in enumerate(scales.tolist()):
        vals += dequant(codes[32 * b: 32 * b + 32], sb)
    return vals


def score(qc, qs, w, kc, ks, order: str = "chain") -> np.float32:
    """float32 score from R_h = max(RN32(q_h . k), 0): "chain" = fma32 chain over heads of
    (w_h, R_h); "split8" = eight fma32 chains over the heads h = j mod 8, added as
    ((p0 + p1) + (p2 + p3)) + ((p4 + p5) + (p6 + p7)) with float32 roundings."""
    kv = exact_vector(kc, ks)
    s = np.float32(0.0)
    p = [np.float32(0.0)] * 8
    for h in range(qc.shape[0]):
        qv = exact_vector(qc[h], qs[h])
        D = rn32(sum((a * b for a, b in zip(qv, kv)), Fraction(0)))
        R = D if D > 0 else np.float32(0.0)
        if order == "chain":
            s = fma32(np.float32(w[h]), R, s)
        else:
            p[h % 8] = fma32(np.float32(w[h]), R, p[h % 8])
    if order == "chain":
        return s
    add = lambda a, b: fma32(np.float32(1.0), a, b)           # one rounding of a + b
    return add(add(add(p[0], p[1]), add(p[2], p[3])), add(add(p[4], p[5]), add(p[6], p[7])))


def topk_positions(scores: Sequence[float], positions: Sequence[int], k: int) -> List[int]:
    """k best by (score descending, position ascending); returned ascending, -1 padded."""
    order = sorted(range(len(positions)), key=lambda i: (-float(scores[i]), positions[i]))
    sel = sorted(positions[i] for i in order[:k])
    return sel + [-1] * (k - len(sel))


def score_exact(qc, qs, w, kc, ks) -> Fraction:
    """The exact score sum_h w_h * max(0, q_h . k) as a Fraction (w_h the exact value of
    each float32 weight; nothing rounded)."""
    kv = exact_vector(kc, ks)
    s = Fraction(0)
    for h in range(qc.shape[0]):
        qv = exact_vector(qc[h], qs[h])
        d = sum((a * b for a, b in zip(qv, kv)), Fraction(0))
        if d > 0:
            s += Fraction(float(np.float32(w[h]))) * d
    return s


def topk_exact_positions(values: Sequence[Fraction], positions: Sequence[int], k: int) -> List[int]:
    """k best by (exact value descending, position ascending); ascending, -1 padded."""
    order = sorted(range(len(positions)), key=lambda i: (-values[i], positions[i]))
    sel = sorted(positions[i] for i in order[:k])
    return sel + [-1] * (k - len(sel))


def quant_block_mxfp8(xs: Sequence[Fraction], signs: Sequence[bool]):
    """OCP MXFP8 (E4M3 elements) of one block of 32 exact values -> (scale byte, [codes]):
    X = floor(log2 amax) - 8 clamped to [-127, 127] (0 for a zero block); each element the
    finite E4M3 magnitude nearest to |x| / 2^X (ties to the even code, beyond 448 the
    nearest is 448), with the sign bit of x."""
    amax = max(abs(x) for x in xs)
    X = 0 if amax == 0 else min(127, max(-127, floor_log2(amax) - 8))
    grid = [e4m3_value(c) for c in range(0x7F)]
    codes = []
    for x, neg in zip(xs, signs):
        v = abs(x) / TWO ** X
        c = min(range(0x7F), key=lambda c: (abs(v - grid[c]), c % 2))
        codes.append(c | (0x80 if neg else 0))
    return X + 127, codes
