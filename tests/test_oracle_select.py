"""Pins of the oracle's Top-K, block pool and Reindex selection (CPU only).

Report (aipaper.jasonlin.tech) §2.3.2 and §4.2.1: Top-512 per query; the decoder's
first Full layer also gives each block of 8 positions the maximum index score of its
positions and keeps the best blocks (at most 2,048, so at most 16,384 positions);
Reindex layers score only the pool and pick their own Top-512 inside it.  Review page
(papers.chlience.com): the two selections come from the same global scores; the
official code scores the full range and then masks to the candidates.
Pins: Python ``sorted`` brute force, closed cases (n <= K, all-equal scores), the
pool bound, Top-K contained in the pool (I1), and Reindex over a Full layer's own
pool reproducing that layer's Top-K (I2).
"""
import numpy as np
import pytest

import oracle
from oracle import tiny
from fp4_kv_cache_gb300 import synth


def _tie_scores(rng, n, levels):
    return rng.integers(0, levels, n).astype(np.float32) * np.float32(0.25)


@pytest.mark.parametrize("n,k,levels", [(40, 8, 5), (100, 100, 3), (30, 64, 4), (500, 37, 1000),
                                        (64, 1, 2)])
def test_topk_matches_sorted_bruteforce(n, k, levels):
    rng = np.random.default_rng(n + k)
    s = _tie_scores(rng, n, levels)
    pos = np.arange(n, dtype=np.int64)
    got = oracle.topk(s, pos, k)
    assert list(got) == tiny.topk_positions(list(s), list(pos), k)


def test_topk_closed_cases():
    pos = np.arange(300)
    # fewer visible than K: all of them, ascending, then -1
    got = oracle.topk(np.random.default_rng(0).random(300).astype(np.float32), pos, 512)
    assert list(got[:300]) == list(range(300)) and np.all(got[300:] == -1)
    # all-equal scores: the lowest positions win
    got = oracle.topk(np.ones(5000, np.float32), np.arange(5000), 512)
    assert list(got) == list(range(512))
    # empty
    assert np.all(oracle.topk(np.zeros(0, np.float32), np.zeros(0, np.int64), 4) == -1)
    # -0 and +0 tie (position decides); NaN ranks below every number
    s = np.array([0.0, -0.0, np.nan, -1.0, 0.0], np.float32)
    assert list(oracle.topk(s, np.arange(5), 3)) == [0, 1, 4]
    assert list(oracle.topk(s, np.arange(5), 4)) == [0, 1, 3, 4]


def _blocks_bruteforce(s, n_vis, block, nb):
    nblk = (n_vis + block - 1) // block
    bs = []
    for b in range(nblk):
        vals = [float(s[p]) for p in range(b * block, min((b + 1) * block, n_vis))]
        bs.append(max(vals))
    order = sorted(range(nblk), key=lambda b: (-bs[b], b))[:nb]
    sel = sorted(order)
    return sel + [-1] * (nb - len(sel))


@pytest.mark.parametrize("n_vis,block,nb,levels", [(203, 8, 7, 6), (64, 8, 8, 3), (61, 8, 20, 50),
                                                   (1000, 8, 100, 4)])
def test_block_candidates_bruteforce(n_vis, block, nb, levels):
    rng = np.random.default_rng(n_vis)
    s = _tie_scores(rng, n_vis, levels)
    got = oracle.block_candidates(s, n_vis, block, nb)
    assert list(got) == _blocks_bruteforce(s, n_vis, block, nb)


def test_pool_bound_and_topk_inside_pool():
    # I1: every Top-K position lies in the pool (its block scores >= the K-th score and
    # at most K blocks can beat it; both selections break ties by lower position), and
    # |pool| <= 2,048 * 8 = 16,384.
    rng = np.random.default_rng(3)
    for trial in range(20):
        n = int(rng.integers(1000, 40000))
        levels = int(rng.choice([3, 50, 100000]))
        s = _tie_scores(rng, n, levels)
        pos = np.arange(n)
        idx = oracle.topk(s, pos, 512)
        blocks = oracle.block_candidates(s, n, 8, 2048)
        pool = oracle.pool_positions(blocks, 8, n)
        assert pool.size <= 16384
        sel = idx[idx >= 0]
        assert np.all(np.isin(sel, pool))
        if n <= 2048 * 8:
            assert pool.size == n          # at most 2,048 blocks: the pool is everything


def test_reindex_over_own_pool_reproduces_full():
    # I2: Reindex with the Full layer's own (q, w) over that layer's pool gives the Full
    # layer's Top-K (the pool contains it when it keeps at least K blocks, and the pool's
    # positions keep their scores).
    w = synth.WORKLOADS["tiny_full_decode"].scaled(n_keys=20000, q_pos0=19999, idx_heads=8,
                                                   idx_dim=128)
    qi, ww, _ = synth.gen_queries(w)
    k = synth.bf16_to_f32(synth.gen_index_keys(w, 0))
    kc, ks = oracle.quant_mxfp4(k)
    q = synth.bf16_to_f32(qi[0, 0])
    idx_full, blocks, s = oracle.full_indexer(q, ww[0, 0], kc, ks, 19999, 1, want_blocks=True,
                                              nb=600)
    idx_re, _, _ = oracle.reindex_indexer(q, ww[0, 0], kc, ks, 19999, 1, blocks)
    assert np.array_equal(idx_full, idx_re)
    # a different query over the same pool selects inside the pool only
    q2 = synth.bf16_to_f32(synth.gen_queries(w.scaled(seed=99))[0][0, 0])
    idx2, _, pool = oracle.reindex_indexer(q2, ww[0, 0], kc, ks, 19999, 1, blocks)
    assert np.all(np.isin(idx2[idx2 >= 0], pool)) and pool.size <= 600 * 8
