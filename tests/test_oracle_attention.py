"""Pins of the oracle's core attention and SWA window (CPU only).

Report (aipaper.jasonlin.tech) §2.3 / §2.3.1: each query attends the selected main-KV
entries together with the layer's SWA KV, in all three modes; the main KV is a latent
shared by every query head (review page, papers.chlience.com, CSA2 section), so V is
the latent's leading d_v dims.  Report §3.2.2: for a replay starting at s, a query at i
attends SWA keys in [max(s, i-W+1), i].  Review page: Reuse reuses the KV and the
position set, but the output still changes with the layer's own query.
Pins: closed forms (one key, equal logits, two keys), torch's float64
scaled_dot_product_attention on a dense case, duplicate/permutation invariants, the
SWA interval, and the Reuse data-flow facts.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from fp4_kv_cache_gb300 import synth


def test_single_key_gives_v():
    rng = np.random.default_rng(0)
    q = rng.standard_normal((1, 4, 64))
    k = rng.standard_normal((1, 64))
    out, lse = oracle.attention_rows(q, [k], 0.125, 48)
    for h in range(4):
        assert np.array_equal(out[0, h], k[0, :48])
        assert lse[0, h] == pytest.approx(0.125 * float(q[0, h] @ k[0]), rel=1e-15, abs=1e-15)


def test_equal_logits_give_mean():
    rng = np.random.default_rng(1)
    keys = rng.standard_normal((37, 32))
    out, lse = oracle.attention_rows(np.zeros((1, 3, 32)), [keys], 0.3, 32)
    assert np.allclose(out[0], keys.mean(0)[None, :], rtol=0, atol=1e-14)
    assert np.allclose(lse[0], math.log(37), rtol=0, atol=1e-14)


def test_two_keys_sigmoid():
    # keys e0 and e1 (unit vectors), q = (a, b): p0 = 1 / (1 + exp(b - a)) with scale 1
    a, b = 1.3, -0.4
    keys = np.zeros((2, 4)); keys[0, 0] = 1.0; keys[1, 1] = 1.0
    keys[0, 2], keys[1, 2] = 10.0, -6.0          # the value coordinate read back
    q = np.array([[[a, b, 0.0, 0.0]]])
    out, lse = oracle.attention_rows(q, [keys], 1.0, 4)
    p0 = 1.0 / (1.0 + math.exp(b - a))
    assert out[0, 0, 2] == pytest.approx(10.0 * p0 - 6.0 * (1 - p0), rel=1e-14)
    assert lse[0, 0] == pytest.approx(math.log(math.exp(a) + math.exp(b)), rel=1e-14)


def test_empty_key_list():
    out, lse = oracle.attention_rows(np.ones((1, 2, 32)), [np.zeros((0, 32))], 1.0, 16)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


@pytest.mark.parametrize("H,n,dqk,dv", [(16, 200, 128, 128), (8, 640, 576, 512)])
def test_dense_case_matches_torch_sdpa(H, n, dqk, dv):
    rng = np.random.default_rng(H + n)
    q = rng.standard_normal((2, H, dqk))
    keys = [rng.standard_normal((n, dqk)), rng.standard_normal((n // 2, dqk))]
    scale = 1.0 / math.sqrt(dqk)
    out, lse = oracle.attention_rows(q, keys, scale, dv)
    for r in range(2):
        kt = torch.from_numpy(keys[r])[None, None].expand(1, H, -1, -1)
        vt = torch.from_numpy(keys[r][:, :dv])[None, None].expand(1, H, -1, -1)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q[r])[None, :, None, :], kt, vt, scale=scale)[0, :, 0]
        assert np.allclose(out[r], ref.numpy(), rtol=1e-10, atol=1e-12)


def test_duplicates_and_permutation():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((1, 5, 64))
    k = rng.standard_normal((10, 64))
    o1, l1 = oracle.attention_rows(q, [k], 0.2, 64)
    o2, l2 = oracle.attention_rows(q, [k[::-1].copy()], 0.2, 64)
    assert np.allclose(o1, o2, rtol=0, atol=1e-13) and np.allclose(l1, l2, atol=1e-13)
    # a key listed twice counts twice: same as raising its weight by a factor of 2
    o3, l3 = oracle.attention_rows(q, [np.concatenate([k, k[:1]])], 0.2, 64)
    lg = 0.2 * (q[0] @ k.T)
    wts = np.exp(lg - lg.max(1, keepdims=True))
    wts[:, 0] *= 2
    ref = (wts @ k) / wts.sum(1, keepdims=True)
    assert np.allclose(o3[0], ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("s", [0, 37, 4000, 5000])
def test_swa_interval(s):
    # buffer slots hold tokens pos0 .. pos0 + n_slots - 1
    W, pos0, n_slots = 128, 3900, 128 + 63
    for i in range(pos0 + W - 1, pos0 + n_slots):
        j0, j1 = oracle.swa_keys_range(i, pos0, n_slots, W, s)
        toks = [pos0 + j for j in range(j0, j1 + 1)]
        expect = [t for t in range(max(s, i - W + 1), i + 1)]
        assert toks == expect


def test_swa_window_is_truncated_at_sequence_start():
    j0, j1 = oracle.swa_keys_range(5, -122, 128, 128, 0)
    assert (j0, j1) == (122, 127)                       # tokens 0..5


def test_reuse_output_follows_the_layer_query():
    # a Full layer and a Reuse layer over the same selection: the Reuse output equals the
    # Full output for the same query and differs for another query
    w = synth.WORKLOADS["tiny_full_decode"]
    qi, ww, qa = synth.gen_queries(w)
    kidx = synth.bf16_to_f32(synth.gen_index_keys(w, 0))
    kc, ks = oracle.quant_mxfp4(kidx)
    kv = synth.bf16_to_f32(synth.gen_main_kv(w, 0))
    kvc, kvs = oracle.quant_mxfp4(kv)
    swa = synth.bf16_to_f32(synth.gen_swa(w, 0)).astype(np.float64)
    n_slots, pos0 = synth.swa_layout(w)
    idx, _, _ = oracle.full_indexer(synth.bf16_to_f32(qi[0, 0]), ww[0, 0], kc, ks, w.q_pos0, 1)
    assert np.all(idx >= 0) and np.all(np.diff(idx) > 0)
    keys = oracle.gather_keys(idx, kvc, kvs, swa, w.q_pos0, pos0, w.window, 0)
    assert keys.shape[0] == 512 + 128
    scale = 1.0 / math.sqrt(w.d_qk)
    q1 = synth.bf16_to_f32(qa[0, 0])[None].astype(np.float64)
    o_full, _ = oracle.attention_rows(q1, [keys], scale, w.d_v)
    o_reuse, _ = oracle.attention_rows(q1, [keys], scale, w.d_v)
    assert np.array_equal(o_full, o_reuse)
    q2 = synth.bf16_to_f32(synth.gen_queries(w.scaled(seed=5))[2][0, 0])[None].astype(np.float64)
    o_other, _ = oracle.attention_rows(q2, [keys], scale, w.d_v)
    assert np.abs(o_other - o_full).max() > 1e-3
