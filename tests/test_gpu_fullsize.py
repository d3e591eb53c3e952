"""Full-size parity: each workload at its full size, launched as the benchmark launches
it, checked against the oracle on every row it can afford (all rows for the decode
workloads, a deterministic sample of 256 queries for the 4,096-query prefill chunk).
Selections are compared with the oracle's ranking by the exact indexer score."""
import math

import numpy as np
import pytest
import torch

import oracle
from fp4_kv_cache_gb300 import csa2, synth, workload
from fp4_kv_cache_gb300.layers import Cache, LayerInput, full_layer, reindex_layer, reuse_layer

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
W = synth.WORKLOADS


def f32(bits):
    return synth.bf16_to_f32(bits)


def _cache(dw, ratio_m=1):
    return Cache(dw["kv_codes"], dw["kv_scales"], dw["k_codes"], dw["k_scales"], ratio_m)


def _cache_kv(dw, ratio_m=1):
    """Cache view for a Reuse layer: main KV only (no indexer K needed)."""
    return Cache(dw["kv_codes"], dw["kv_scales"], None, None, ratio_m)


def _inp(dw):
    return LayerInput(dw["q_attn"], dw["swa"], dw["swa_pos0"], dw["q_pos"], dw["q_idx"], dw["w_idx"])


def _check_attention_rows(w, out, lse, idx_np, rows_bt, swa_start=0):
    qpos = synth.q_positions(w)
    n_slots, pos0 = synth.swa_layout(w)
    _, _, qa = synth.gen_queries(w)
    worst = 0.0
    by_b = {}
    for b, t in rows_bt:
        by_b.setdefault(b, []).append(t)
    for b, ts in by_b.items():
        kv = f32(synth.gen_main_kv(w, b))
        swa = f32(synth.gen_swa(w, b)).astype(np.float64)
        for t in ts:
            sel = idx_np[b, t]
            sel = sel[(sel >= 0) & (sel < w.n_keys)]
            kc, ks = oracle.quant_mxfp4(kv[sel])              # only the rows attention reads
            keys = oracle.gather_keys(np.arange(sel.size), kc, ks, swa, int(qpos[b, t]), pos0,
                                      w.window, swa_start)
            o_ref, l_ref = oracle.attention_rows(f32(qa[b, t])[None].astype(np.float64), [keys],
                                                 1.0 / math.sqrt(w.d_qk), w.d_v)
            o = out[b, t].float().cpu().numpy().astype(np.float64)
            err = np.abs(o - o_ref[0]).max(-1) / np.maximum(np.abs(o_ref[0]).max(-1), 1e-6)
            assert err.max() <= 1e-2, (b, t, err.max())
            assert np.abs(lse[b, t].cpu().numpy() - l_ref[0]).max() <= 1e-3
            worst = max(worst, err.max())
    return worst


def _oracle_full(w, b, t, qi, ww, kc, ks, qpos, want_blocks=False, nb=2048, want_f32=False):
    return oracle.full_indexer(f32(qi[b, t]), ww[b, t], kc, ks, int(qpos[b, t]), w.ratio_m, w.topk,
                               w.block, nb, want_blocks=want_blocks, want_f32=want_f32)


def test_full_decode_64k():
    """Full-mode decode layer, batch 32 x 65,536 positions: every row's Top-512 bit-exact,
    every row's attention within 1e-2."""
    w = W["full_decode_64k"]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dw = workload.build(w, device=DEV, d_status=st)
    res = full_layer(_cache(dw), _inp(dw), w.topk, w.window, w.d_v, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    qi, ww, _ = synth.gen_queries(w)
    qpos = synth.q_positions(w)
    idx_gpu = res.idx.cpu().numpy()
    recall = []
    for b in range(w.batch):
        kc, ks = oracle.quant_mxfp4(f32(synth.gen_index_keys(w, b, qi[b], ww[b])))
        idx_ref, _, _ = _oracle_full(w, b, 0, qi, ww, kc, ks, qpos)
        assert np.array_equal(idx_gpu[b, 0], idx_ref), b
    _check_attention_rows(w, res.out, res.lse, idx_gpu, [(b, 0) for b in range(w.batch)])


def test_reuse_and_reindex_128k():
    """Reuse (given indices) and Reindex (pool of 2,048 blocks) at batch 64 x 131,072."""
    w = W["reuse_reindex_decode_128k"]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dw = workload.build(w, device=DEV, d_status=st)
    cache, x = _cache(dw), _inp(dw)
    re = reindex_layer(cache, x, dw["pool"], w.topk, w.window, w.d_v, d_status=st)
    ru = reuse_layer(cache, x, dw["reuse_idx"], w.window, w.d_v, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    qi, ww, _ = synth.gen_queries(w)
    qpos = synth.q_positions(w)
    pool = dw["pool"].cpu().numpy()
    for b in range(w.batch):                        # every row's Reindex selection
        kc, ks = oracle.quant_mxfp4(f32(synth.gen_index_keys(w, b, qi[b], ww[b])))
        idx_ref, _, _ = oracle.reindex_indexer(f32(qi[b, 0]), ww[b, 0], kc, ks, int(qpos[b, 0]), 1,
                                               pool[b, 0], w.topk, w.block, want_f32=False)
        assert np.array_equal(re.idx[b, 0].cpu().numpy(), idx_ref), b
    sample = list(range(0, 64, 4))
    _check_attention_rows(w, ru.out, ru.lse, dw["reuse_idx"].cpu().numpy(), [(b, 0) for b in sample])
    _check_attention_rows(w, re.out, re.lse, re.idx.cpu().numpy(), [(b, 0) for b in sample[::2]])


def test_hierarchical_indexer_1m():
    """Decoder's first Full layer at 1,048,576 positions with heavy ties: Top-512 and the
    Top-2,048 block pool bit-exact on all 4 rows; the pool holds the Top-512."""
    w = W["hier_indexer_1m"]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dw = workload.build(w, kv=False, device=DEV, d_status=st)
    scores, row_len, args = csa2.index_score(dw["q_idx"], dw["w_idx"], dw["k_codes"], dw["k_scales"],
                                             dw["q_pos"], 1, None, w.block, st, want_args=True)
    idx = csa2.topk(scores, w.topk, row_len, d_status=st, exact=args)
    blocks = csa2.block_candidates(scores, w.n_blocks, row_len, w.block, st, exact=args)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    qi, ww, _ = synth.gen_queries(w)
    qpos = synth.q_positions(w)
    for b in range(w.batch):
        kc, ks = oracle.quant_mxfp4(f32(synth.gen_index_keys(w, b, qi[b], ww[b])))
        idx_ref, blocks_ref, s_ref = _oracle_full(w, b, 0, qi, ww, kc, ks, qpos, True, w.n_blocks, True)
        assert np.array_equal(idx[b, 0].cpu().numpy(), idx_ref), b
        assert np.array_equal(blocks[b, 0].cpu().numpy(), blocks_ref), b
        pool = oracle.pool_positions(blocks_ref, w.block, w.n_keys)
        assert pool.size <= 16384 and np.all(np.isin(idx_ref, pool))
        # the tie-break decided: the 512th score value repeats beyond the selection
        kth = np.sort(s_ref)[::-1][w.topk - 1]
        assert (s_ref == kth).sum() > (s_ref[idx_ref] == kth).sum()


def test_prefill_chunk_sampled():
    """Encoder Full layer prefill chunk at ratio 2 (4,096 queries after 65,536 entries):
    GPU runs the whole chunk; a deterministic query sample is checked."""
    w = W["prefill_chunk_m2"]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dw = workload.build(w, device=DEV, d_status=st)
    res = full_layer(_cache(dw, 2), _inp(dw), w.topk, w.window, w.d_v, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    qi, ww, _ = synth.gen_queries(w)
    qpos = synth.q_positions(w)
    kc, ks = oracle.quant_mxfp4(f32(synth.gen_index_keys(w, 0, qi[0], ww[0])))
    # 256 queries: the first and last 8, and every 17th from 8 on; 64 of them for attention
    sample = sorted(set(list(range(8)) + list(range(4088, 4096)) + list(range(8, 4088, 17))))
    assert len(sample) == 256
    idx_gpu = res.idx.cpu().numpy()
    for t in sample:
        nvis = oracle.n_visible(int(qpos[0, t]), 2, w.n_keys)
        assert int((idx_gpu[0, t] >= 0).sum()) == min(w.topk, nvis)
        idx_ref, _, _ = _oracle_full(w, 0, t, qi, ww, kc, ks, qpos)
        assert np.array_equal(idx_gpu[0, t], idx_ref), t
    _check_attention_rows(w, res.out, res.lse, idx_gpu, [(0, t) for t in sample[::4]])


def test_swa_replay_prefill():
    """Decoder SWA bounded replay (report §3.2.2): 128 tokens replayed from s = 131,072, each
    attending its given Top-512 entries and the SWA keys [max(s, i - W + 1), i] -- query
    s + j sees j + 1 of them; the 127 buffered tokens before s are never attended."""
    w = W["swa_replay_prefill"]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dw = workload.build(w, kidx=False, device=DEV, d_status=st)
    x = LayerInput(dw["q_attn"], dw["swa"], dw["swa_pos0"], dw["q_pos"], swa_start=dw["swa_start"])
    res = reuse_layer(_cache_kv(dw), x, dw["reuse_idx"], w.window, w.d_v, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    n_slots, pos0 = synth.swa_layout(w)
    qpos = synth.q_positions(w)
    for t in (0, 5, 127):
        j0, j1 = oracle.swa_keys_range(int(qpos[0, t]), pos0, n_slots, w.window, w.swa_start)
        assert j1 - j0 + 1 == min(w.window, t + 1)
    rows = [(b, t) for b in (0, w.batch - 1) for t in list(range(0, 128, 2)) + [127]]
    worst = _check_attention_rows(w, res.out, res.lse, dw["reuse_idx"].cpu().numpy(), rows, w.swa_start)
    assert worst <= 1e-2
