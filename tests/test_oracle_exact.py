"""Pins of the oracle's exact indexer score and of the selections made on it (CPU only).

Score (the workload definition; the report, aipaper.jasonlin.tech §2.3, says only that
the indexer scores main-KV entries from indexer Q and indexer K, both MXFP4 by §2.4.4):
    s = sum_h w_h * max(0, q_hat_h . k_hat)
computed exactly -- no product, dot or sum rounded -- and used to rank positions
(Top-512, report §4.2.1) and blocks of 8 (report §2.3.2).  Pins:
  * an exact ``fractions.Fraction`` brute force on tiny inputs, over typical and
    full-range scale bytes, negative, zero, subnormal and huge weights;
  * properties exact arithmetic has and a rounded chain lacks: invariance under a
    permutation of the heads, additivity in the weights, exact scaling by 2^k;
  * the textbook case H = 1, w = 1 (the plain dot product);
  * a hand-built pair of positions whose float32 scores tie while their exact scores
    do not, where only the exact ranking picks the right one;
  * the error bound the GPU selection relies on: the float32 chain the library writes
    out is within (H + 2) 2^-24 A + 2^-149 (sum|w_h| + H) of the exact score, where
    A = sum_h |w_h| max(0, q_h . k);
  * selections against ``sorted()`` on the Fraction values, the pool bound and
    Top-K inside the pool (I1), Reindex over a Full layer's own pool (I2).
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import tiny
from fp4_kv_cache_gb300 import synth


def _rand_mx(rng, rows, d, lo, hi):
    codes = rng.integers(0, 256, size=(rows, d // 2), dtype=np.uint8)
    scales = rng.integers(lo, hi + 1, size=(rows, d // 32)).astype(np.uint8)
    return codes, scales


def _weights(rng, H, kind):
    if kind == "unit":
        return rng.random(H).astype(np.float32)
    if kind == "normal":
        return rng.standard_normal(H).astype(np.float32)
    if kind == "extreme":
        w = rng.standard_normal(H).astype(np.float32)
        w[0] = np.float32(1e-45)                  # smallest subnormal
        if H > 1:
            w[1] = np.float32(-3.0e38)
        if H > 2:
            w[2] = 0.0
        if H > 3:
            w[3] = np.float32(2.0 ** -140)
        return w
    raise ValueError(kind)


def _frac(limbs_row):
    return oracle.exact_fraction(limbs_row)


@pytest.mark.parametrize("H,d,lo,hi,wkind,seed", [
    (1, 32, 120, 134, "unit", 0), (4, 64, 120, 134, "unit", 1), (3, 96, 110, 140, "normal", 2),
    (2, 64, 0, 254, "normal", 3), (4, 128, 0, 255, "extreme", 4), (5, 128, 60, 200, "extreme", 5),
    (8, 128, 125, 129, "normal", 6)])
def test_exact_scores_match_fraction_bruteforce(H, d, lo, hi, wkind, seed):
    rng = np.random.default_rng(100 + seed)
    N = 16
    kc, ks = _rand_mx(rng, N, d, lo, hi)
    qc, qs = _rand_mx(rng, H, d, lo, hi)
    w = _weights(rng, H, wkind)
    ex = oracle.index_scores_exact(qc, qs, w, kc, ks, np.arange(N))
    for t in range(N):
        assert _frac(ex[t]) == tiny.score_exact(qc, qs, w, kc[t], ks[t]), t


def test_exact_score_textbook_single_head():
    # H = 1, w = 1: the exact score is the plain dot product of the dequantised vectors
    # when it is positive (numpy float64 dot, exact for these small dyadic values), else 0
    rng = np.random.default_rng(7)
    d, N = 128, 64
    k = synth.bf16_to_f32(synth.f32_to_bf16_bits(rng.standard_normal((N, d)).astype(np.float32)))
    q = synth.bf16_to_f32(synth.f32_to_bf16_bits(rng.standard_normal((1, d)).astype(np.float32)))
    kc, ks = oracle.quant_mxfp4(k)
    qc, qs = oracle.quant_mxfp4(q)
    ref = oracle.dequant_mxfp4(kc, ks) @ oracle.dequant_mxfp4(qc, qs)[0]
    ex = oracle.index_scores_exact(qc, qs, np.array([1.0], np.float32), kc, ks, np.arange(N))
    for t in range(N):
        assert _frac(ex[t]) == (Fraction(float(ref[t])) if ref[t] > 0 else 0)


def test_exact_score_head_permutation_invariant():
    # exact addition does not depend on the order of the heads (a float32 chain does)
    rng = np.random.default_rng(11)
    H, d, N = 16, 128, 300
    kc, ks = _rand_mx(rng, N, d, 118, 136)
    qc, qs = _rand_mx(rng, H, d, 118, 136)
    w = rng.random(H).astype(np.float32) * np.exp2(rng.integers(-20, 4, H)).astype(np.float32)
    perm = rng.permutation(H)
    a = oracle.index_scores_exact(qc, qs, w, kc, ks, np.arange(N))
    b = oracle.index_scores_exact(qc[perm], qs[perm], w[perm], kc, ks, np.arange(N))
    assert np.array_equal(a, b)
    f1 = oracle.index_scores(qc, qs, w, kc, ks, np.arange(N))
    f2 = oracle.index_scores(qc[perm], qs[perm], w[perm], kc, ks, np.arange(N))
    assert not np.array_equal(f1, f2)        # the chain's rounding does depend on it


def test_exact_score_additive_in_weights():
    # s(w1 + w2) = s(w1) + s(w2) for weights on disjoint heads (w1 + w2 exact in float32),
    # and s(2^k w) = 2^k s(w): a dropped or doubled term breaks these
    rng = np.random.default_rng(12)
    H, d, N = 8, 128, 200
    kc, ks = _rand_mx(rng, N, d, 100, 150)
    qc, qs = _rand_mx(rng, H, d, 100, 150)
    w = rng.standard_normal(H).astype(np.float32)
    m = np.arange(H) % 2 == 0
    w1, w2 = np.where(m, w, 0).astype(np.float32), np.where(m, 0, w).astype(np.float32)
    pos = np.arange(N)
    s = oracle.index_scores_exact(qc, qs, w, kc, ks, pos)
    s1 = oracle.index_scores_exact(qc, qs, w1, kc, ks, pos)
    s2 = oracle.index_scores_exact(qc, qs, w2, kc, ks, pos)
    s8 = oracle.index_scores_exact(qc, qs, w * np.float32(8), kc, ks, pos)
    for t in range(N):
        assert oracle.exact_int(s[t]) == oracle.exact_int(s1[t]) + oracle.exact_int(s2[t])
        assert oracle.exact_int(s8[t]) == 8 * oracle.exact_int(s[t])


def _one_hot_codes(d, entries):
    """Packed E2M1 codes of one row: code c at element i for (i, c) in entries."""
    codes = np.zeros(d, np.uint8)
    for i, c in entries:
        codes[i] = c
    return (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)


def test_float32_tie_resolved_by_exact_score():
    # two heads, w = (1, 2^-30); both positions have d_0 = 1, and d_1 = 1 at position 0,
    # d_1 = 2 at position 1.  Exact scores 1 + 2^-30 < 1 + 2^-29, but both round to 1.0 in
    # float32, where the tie goes to position 0.  The exact Top-1 is position 1.
    d = 32
    qc = np.stack([_one_hot_codes(d, [(0, 2)]), _one_hot_codes(d, [(1, 2)])])   # code 2 = 1.0
    qs = np.full((2, 1), 127, np.uint8)
    kc = np.stack([_one_hot_codes(d, [(0, 2), (1, 2)]), _one_hot_codes(d, [(0, 2), (1, 4)])])   # 4 = 2.0
    ks = np.full((2, 1), 127, np.uint8)
    w = np.array([1.0, 2.0 ** -30], np.float32)
    pos = np.arange(2)
    f = oracle.index_scores(qc, qs, w, kc, ks, pos)
    assert f[0] == f[1] == np.float32(1.0)
    ex = oracle.index_scores_exact(qc, qs, w, kc, ks, pos)
    assert _frac(ex[0]) == 1 + Fraction(1, 2 ** 30) and _frac(ex[1]) == 1 + Fraction(1, 2 ** 29)
    assert list(oracle.topk(f, pos, 1)) == [0]
    assert list(oracle.topk_exact(ex, pos, 1)) == [1]
    assert list(oracle.block_candidates_exact(ex, 2, 1, 1)) == [1]


def _bound(w, A, H):
    """Error bound of the float32 scores the library writes out (any summation order of
    the heads, each per-head dot rounded once): (H + 2) 2^-24 A + 2^-149 (sum|w| + H)."""
    return Fraction(H + 2, 2 ** 24) * A + Fraction(1, 2 ** 149) * (
        sum(abs(Fraction(float(x))) for x in w) + H)


@pytest.mark.parametrize("H,lo,hi,wkind,seed", [
    (32, 120, 134, "unit", 0), (32, 120, 134, "normal", 1), (8, 0, 254, "normal", 2),
    (4, 0, 254, "extreme", 3), (64, 124, 130, "normal", 4), (16, 1, 40, "unit", 5)])
def test_float32_scores_within_error_bound(H, lo, hi, wkind, seed):
    rng = np.random.default_rng(300 + seed)
    d, N = 128, 400
    kc, ks = _rand_mx(rng, N, d, lo, hi)
    qc, qs = _rand_mx(rng, H, d, lo, hi)
    w = _weights(rng, H, wkind)
    # cancellation: pairs of heads with the same query and opposite weights
    if wkind == "normal" and H >= 4:
        qc[1], qs[1], w[1] = qc[0], qs[0], -w[0] * np.float32(1.0000001)
    pos = np.arange(N)
    ex = oracle.index_scores_exact(qc, qs, w, kc, ks, pos)
    A = oracle.index_scores_exact(qc, qs, np.abs(w), kc, ks, pos)
    for order in ("chain", "split8"):                 # both orders the library writes
        f = oracle.index_scores(qc, qs, w, kc, ks, pos, order=order)
        checked = 0
        for t in range(N):
            if not np.isfinite(f[t]):
                continue                      # overflow: outside the bound's domain
            err = abs(Fraction(float(f[t])) - _frac(ex[t]))
            assert err <= _bound(w, _frac(A[t]), H), (order, t)
            checked += 1
        assert checked >= 20


def test_exact_topk_and_blocks_match_sorted_bruteforce():
    # heavy ties: positions share key rows from a small palette, so exact scores repeat
    rng = np.random.default_rng(21)
    H, d, n = 4, 64, 700
    pal_c, pal_s = _rand_mx(rng, 9, d, 124, 130)
    which = rng.integers(0, 9, n)
    kc, ks = pal_c[which], pal_s[which]
    qc, qs = _rand_mx(rng, H, d, 124, 130)
    w = rng.random(H).astype(np.float32)
    pos = np.arange(n)
    ex = oracle.index_scores_exact(qc, qs, w, kc, ks, pos)
    vals = [_frac(ex[t]) for t in range(n)]
    for k in (1, 37, 200, 700, 900):
        assert list(oracle.topk_exact(ex, pos, k)) == tiny.topk_exact_positions(vals, list(pos), k)
    # blocks of 8 (a partial last block uses its visible positions), nb of them
    for n_vis, nb in ((n, 10), (597, 30), (64, 8)):
        nblk = (n_vis + 7) // 8
        bv = [max(vals[p] for p in range(8 * b, min(8 * b + 8, n_vis))) for b in range(nblk)]
        order = sorted(range(nblk), key=lambda b: (-bv[b], b))[:nb]
        exp = sorted(order) + [-1] * (nb - min(nb, nblk))
        assert list(oracle.block_candidates_exact(ex[:n_vis], n_vis, 8, nb)) == exp


def test_exact_pool_contains_topk_and_reindex_reproduces_full():
    # I1 on exact scores: every Top-512 position lies in the Top-2,048 block pool, and
    # |pool| <= 16,384.  I2: Reindex with the Full layer's own (q, w) over its pool
    # selects the Full layer's Top-K.
    w = synth.WORKLOADS["hier_indexer_1m"].scaled(n_keys=60000, q_pos0=59999, palette=300,
                                                  palette_zero=4)
    qi, ww, _ = synth.gen_queries(w)
    kc, ks = oracle.quant_mxfp4(synth.bf16_to_f32(synth.gen_index_keys(w, 0)))
    q = synth.bf16_to_f32(qi[0, 0])
    idx, blocks, _ = oracle.full_indexer(q, ww[0, 0], kc, ks, 59999, 1, want_blocks=True,
                                         want_f32=False)
    pool = oracle.pool_positions(blocks, 8, 60000)
    assert pool.size <= 16384
    assert np.all(np.isin(idx[idx >= 0], pool))
    idx_re, _, _ = oracle.reindex_indexer(q, ww[0, 0], kc, ks, 59999, 1, blocks, want_f32=False)
    assert np.array_equal(idx, idx_re)
