"""GPU parity of every step of the CSA2 path against the CPU oracle (needs a GB300).

The bar (workload definition): indices, block ids and FP4 codes bit-exact, with
selections ranked by the EXACT indexer score; the float32 scores the indexer writes out
bit-exact too (both sides compute that approximation in the same float32 precision); attention
within 1e-2 relative error per (query, head) row:
    max_c |o_gpu - o_ref| / max(max_c |o_ref|, 1e-6) <= 1e-2,
a row-normwise reading of "max relative error" so that near-zero elements do not blow
the ratio up; lse within 1e-3 absolute.  Every input comes from the seeded generator;
the oracle quantises, scores, selects and attends with its own code.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
from fp4_kv_cache_gb300 import csa2, synth, workload

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
ATTN_TOL = 1e-2
LSE_TOL = 1e-3


def f32(bits):
    return synth.bf16_to_f32(bits)


def status():
    return torch.zeros(1, dtype=torch.int32, device=DEV)


def same_f32(a, b):
    """bitwise float32 equality, NaNs compared as NaN."""
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    nan = np.isnan(a) & np.isnan(b)
    return np.array_equal(a.view(np.uint32)[~nan], b.view(np.uint32)[~nan]) and \
        np.array_equal(np.isnan(a), np.isnan(b))


# ------------------------------------------------------------------ codec
def _codec_inputs(rows, cols, seed, as_bf16):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, cols)).astype(np.float32)
    x *= np.exp2(rng.integers(-140, 100, size=(rows, 1))).astype(np.float32)
    x[0] = 0.0
    x[1] = -0.0
    x[2, ::3] = np.float32(1e-45)                       # fp32 subnormals
    x[3] = np.float32(3.0e38) * np.sign(x[3])
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.75], np.float32)
    x[4, :] = 0.0
    x[4, : cols] = np.resize(ties, cols)
    if as_bf16:
        bits = synth.f32_to_bf16_bits(x)
        return bits, synth.bf16_to_f32(bits)
    return x, x


@pytest.mark.parametrize("cols,as_bf16", [(64, True), (576, True), (128, False), (32, False)])
def test_quant_dequant_parity(cols, as_bf16):
    raw, x = _codec_inputs(3001, cols, cols + as_bf16, as_bf16)
    xt = workload.bf16_tensor(raw, DEV) if as_bf16 else torch.from_numpy(raw).to(DEV)
    st = status()
    codes, scales = csa2.quant_fp4(xt, st)
    c_ref, s_ref = oracle.quant_mxfp4(x)
    assert np.array_equal(codes.cpu().numpy(), c_ref)
    assert np.array_equal(scales.cpu().numpy(), s_ref)
    assert int(st.item()) == 0
    # dequantisation: exact in float32, and in bf16 (scale bytes here are <= 252)
    y_ref = oracle.dequant_mxfp4(c_ref, s_ref).astype(np.float32)
    y32 = csa2.dequant_fp4(codes, scales, torch.float32).cpu().numpy()
    assert np.array_equal(y32.view(np.uint32), y_ref.view(np.uint32))
    y16 = csa2.dequant_fp4(codes, scales, torch.bfloat16).view(torch.int16).cpu().numpy()
    assert np.all(y_ref.view(np.uint32) & 0xFFFF == 0)
    assert np.array_equal(y16.view(np.uint16), (y_ref.view(np.uint32) >> 16).astype(np.uint16))
    # FP4 round trip on the GPU: quantising the dequantised values gives the same codes
    c2, s2 = csa2.quant_fp4(torch.from_numpy(y32).to(DEV))
    # (per 32-value block: a block whose scale clamped at 2^-127 may round to all zeros,
    # and then takes the zero-block scale)
    assert np.array_equal(c2.cpu().numpy(), c_ref)
    nz = np.any((c_ref.reshape(c_ref.shape[0], -1, 16) & 0x77) != 0, axis=2)
    assert np.array_equal(s2.cpu().numpy()[nz], s_ref[nz])


@pytest.mark.parametrize("cols,as_bf16", [(576, True), (48, False), (16, True)])
def test_quant_dequant_nvfp4_parity(cols, as_bf16):
    # E2M1 + E4M3/16 (the report's main-KV format): codes and scale bytes bit-exact, and
    # every dequantised value exact in float32 and bf16
    raw, x = _codec_inputs(2001, cols, 100 + cols + as_bf16, as_bf16)
    rng = np.random.default_rng(cols)
    x_small = rng.standard_normal((400, cols)).astype(np.float32)
    x_small *= np.exp2(rng.integers(-16, 14, size=(400, 1))).astype(np.float32)   # E4M3 range
    if as_bf16:
        bits_small = synth.f32_to_bf16_bits(x_small)
        raw, x = np.concatenate([raw, bits_small]), np.concatenate([x, f32(bits_small)])
    else:
        raw = x = np.concatenate([x, x_small])
    xt = workload.bf16_tensor(raw, DEV) if as_bf16 else torch.from_numpy(raw).to(DEV)
    st = status()
    codes, scales = csa2.quant_fp4(xt, st, fmt=csa2.FMT_NVFP4_E4M3_16)
    c_ref, s_ref = oracle.quant_nvfp4(x)
    assert scales.shape[-1] == cols // 16
    assert np.array_equal(scales.cpu().numpy(), s_ref)
    assert np.array_equal(codes.cpu().numpy(), c_ref)
    assert int(st.item()) == 0
    y_ref = oracle.dequant_nvfp4(c_ref, s_ref).astype(np.float32)
    y32 = csa2.dequant_fp4(codes, scales, torch.float32).cpu().numpy()
    assert np.array_equal(y32.view(np.uint32), y_ref.view(np.uint32))
    y16 = csa2.dequant_fp4(codes, scales, torch.bfloat16).view(torch.int16).cpu().numpy()
    assert np.all(y_ref.view(np.uint32) & 0xFFFF == 0)
    assert np.array_equal(y16.view(np.uint16), (y_ref.view(np.uint32) >> 16).astype(np.uint16))
    # row-strided, unaligned rows take the scalar kernel: same bytes
    wide = torch.zeros((xt.shape[0], cols + 1), dtype=xt.dtype, device=DEV)
    wide[:, :cols] = xt
    c_u = torch.empty_like(codes)
    s_u = torch.empty_like(scales)
    csa2.csa2_quant_fp4(wide[:, :cols], c_u, s_u, st, fmt=csa2.FMT_NVFP4_E4M3_16)
    assert np.array_equal(c_u.cpu().numpy(), c_ref) and np.array_equal(s_u.cpu().numpy(), s_ref)


@pytest.mark.parametrize("cols,as_bf16", [(576, True), (64, False), (32, True)])
def test_quant_dequant_mxfp8_parity(cols, as_bf16):
    # MXFP8 SWA codec (report §2.4.4 keeps the SWA cache in FP8): codes and scale bytes
    # bit-exact, every dequantised value exact in float32 and bf16 (moderate scales)
    raw, x = _codec_inputs(2001, cols, 300 + cols + as_bf16, as_bf16)
    xt = workload.bf16_tensor(raw, DEV) if as_bf16 else torch.from_numpy(raw).to(DEV)
    st = status()
    codes, scales = csa2.quant_fp8(xt, st)
    c_ref, s_ref = oracle.quant_mxfp8(x)
    assert np.array_equal(scales.cpu().numpy(), s_ref)
    assert np.array_equal(codes.cpu().numpy(), c_ref)
    assert int(st.item()) == 0
    y_ref = oracle.dequant_mxfp8(c_ref, s_ref).astype(np.float32)
    y32 = csa2.dequant_fp8(codes, scales, torch.float32).cpu().numpy()
    assert np.array_equal(y32.view(np.uint32), y_ref.view(np.uint32))
    ok = (s_ref >= 127 - 100) & (s_ref <= 127 + 100)                # bf16-normal products
    rows_ok = ok.all(axis=1)
    y16 = csa2.dequant_fp8(codes, scales, torch.bfloat16).view(torch.int16).cpu().numpy()
    assert np.array_equal(y16.view(np.uint16)[rows_ok],
                          (y_ref.view(np.uint32) >> 16).astype(np.uint16)[rows_ok])
    x[3] = np.float32(np.inf)
    bad = torch.from_numpy(np.ascontiguousarray(x[:8], np.float32)).to(DEV)
    st2 = status()
    csa2.quant_fp8(bad, st2)
    torch.cuda.synchronize()
    assert int(st2.item()) & csa2.DEV_NONFINITE


def test_nvfp4_scale_rounding_boundaries():
    # block maxima at, and one float32 step either side of, 6 x every E4M3 rounding midpoint,
    # plus the zero-scale and clamp edges: the GPU's scale bytes and codes match the oracle's
    vals = oracle.dequant_nvfp4(np.full((0x7F, 8), 0x22, np.uint8),        # code 2 = 1.0
                                np.arange(0x7F, dtype=np.uint8)[:, None])[:, 0]   # E4M3 values
    amax = []
    for lo, hi in zip(vals[:-1], vals[1:]):
        m = np.float32(3.0 * (lo + hi))
        amax += [np.nextafter(m, np.float32(0)), m, np.nextafter(m, np.float32(np.inf))]
    amax += [np.float32(v) for v in (0.0, 1e-30, 6 * 2.0 ** -10, 2688.0, 2785.0, 1e30)]
    amax = np.asarray(amax, np.float32)
    x = np.zeros((amax.size, 16), np.float32)
    x[:, 5] = amax
    x[:, 6] = -amax * np.float32(0.3)
    x[:, 7] = amax * np.float32(0.75 / 6.0)
    st = status()
    codes, scales = csa2.quant_fp4(torch.from_numpy(x).to(DEV), st, fmt=csa2.FMT_NVFP4_E4M3_16)
    c_ref, s_ref = oracle.quant_nvfp4(x.astype(np.float64))
    assert np.array_equal(scales.cpu().numpy(), s_ref)
    assert np.array_equal(codes.cpu().numpy(), c_ref)
    assert int(st.item()) == 0


def _rope_table(n_pos, rope_dim, base=10000.0):
    """Synthetic RoPE table [n_pos, rope_dim]: cosines then sines of p * base^(-2i/R)."""
    i = np.arange(rope_dim // 2, dtype=np.float64)
    ang = np.arange(n_pos, dtype=np.float64)[:, None] * base ** (-2.0 * i / rope_dim)[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def test_rope_quant_parity():
    # report §2.4.4: the cache is quantised after RoPE.  One launch, four jobs: main-KV rows
    # (512 + 64 rotated channels) in both formats, a 128-channel key block with 64 rotated
    # channels, and a block with no rotation; codes and scales bit-exact against the oracle;
    # one row's position lies outside the table (flagged, quantised unrotated)
    rng = np.random.default_rng(77)
    n_pos = 4096
    tab = _rope_table(n_pos, 64)
    tab_d = torch.from_numpy(tab).to(DEV)
    specs = [(333, 576, 64, csa2.FMT_MXFP4), (129, 576, 64, csa2.FMT_NVFP4_E4M3_16),
             (70, 128, 64, csa2.FMT_MXFP4), (17, 512, 0, csa2.FMT_NVFP4_E4M3_16)]
    st = status()
    call, refs = [], []
    for rows, cols, R, fmt in specs:
        g = csa2.FMT_BLOCK[fmt]
        x = rng.standard_normal((rows, cols)).astype(np.float32)
        x *= np.exp2(rng.integers(-12, 8, size=(rows, 1))).astype(np.float32)
        bits = synth.f32_to_bf16_bits(x)
        pos = rng.integers(0, n_pos, rows).astype(np.int32)
        pos[0], pos[-1] = 0, n_pos - 1
        codes = torch.full((rows, cols // 2 + 8), 0xAB, dtype=torch.uint8, device=DEV)   # strided rows
        scales = torch.full((rows, cols // g + 4), 0xAB, dtype=torch.uint8, device=DEV)
        xt = workload.bf16_tensor(bits, DEV)
        pos_d = torch.from_numpy(pos).to(DEV)
        call.append((xt, codes[:, : cols // 2], scales[:, : cols // g], R, pos_d if R else None,
                     tab_d if R else None, fmt))
        refs.append((oracle.rope_quant(f32(bits), pos, tab, R, "nvfp4" if g == 16 else "mxfp4"),
                     codes, scales, cols, g))
    csa2.csa2_rope_quant_fp4(call, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for (c_ref, s_ref), codes, scales, cols, g in refs:
        assert np.array_equal(codes[:, : cols // 2].cpu().numpy(), c_ref)
        assert np.array_equal(scales[:, : cols // g].cpu().numpy(), s_ref)
        assert torch.all(codes[:, cols // 2:] == 0xAB) and torch.all(scales[:, cols // g:] == 0xAB)
    # a position past the table: flagged, and that row is quantised without rotation
    xt, codes, scales, R, pos_d, _, fmt = call[0]
    pos_bad = pos_d.clone()
    pos_bad[5] = n_pos
    st2 = status()
    csa2.csa2_rope_quant_fp4([(xt, codes, scales, R, pos_bad, tab_d, fmt)], st2)
    torch.cuda.synchronize()
    assert int(st2.item()) & csa2.DEV_BAD_INDEX
    c_plain, s_plain = oracle.quant_mxfp4(f32(xt[5:6].view(torch.int16).cpu().numpy().view(np.uint16)))
    assert np.array_equal(codes[5:6].cpu().numpy(), c_plain) and np.array_equal(scales[5:6].cpu().numpy(), s_plain)


@pytest.mark.parametrize("aligned", [True, False])
def test_quant_batch_parity(aligned):
    # one launch for several jobs (bf16 and f32, different widths, a row-strided cache view);
    # aligned=False gives one job rows that are not 16-byte aligned (one launch per job)
    specs = [(577, 576, True), (33, 128, False), (5, 64, True), (40, 32, False)]
    st = status()
    triples, refs = [], []
    for i, (rows, cols, bf16) in enumerate(specs):
        raw, x = _codec_inputs(rows, cols, 7000 + i, bf16)
        xt = workload.bf16_tensor(raw, DEV) if bf16 else torch.from_numpy(raw).to(DEV)
        if not aligned and i == 1:            # rows of 128 + 1 floats: 4-byte aligned only
            wide = torch.zeros((rows, cols + 1), dtype=xt.dtype, device=DEV)
            wide[:, :cols] = xt
            xt = wide[:, :cols]
        cache_c = torch.full((rows, cols // 2 + 16), 0xAB, dtype=torch.uint8, device=DEV)   # strided rows
        cache_s = torch.full((rows, cols // 32 + 4), 0xAB, dtype=torch.uint8, device=DEV)
        triples.append((xt, cache_c[:, : cols // 2], cache_s[:, : cols // 32]))
        refs.append((oracle.quant_mxfp4(x), cache_c, cache_s, cols))
    csa2.csa2_quant_fp4_batch(triples, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for (c_ref, s_ref), cache_c, cache_s, cols in refs:
        assert np.array_equal(cache_c[:, : cols // 2].cpu().numpy(), c_ref)
        assert np.array_equal(cache_s[:, : cols // 32].cpu().numpy(), s_ref)
        assert torch.all(cache_c[:, cols // 2:] == 0xAB) and torch.all(cache_s[:, cols // 32:] == 0xAB)


def test_quant_flags_nonfinite():
    x = torch.zeros((3, 64), dtype=torch.float32, device=DEV)
    x[1, 40] = float("inf")
    st = status()
    codes, scales = csa2.quant_fp4(x, st)
    torch.cuda.synchronize()
    assert int(st.item()) & csa2.DEV_NONFINITE
    assert torch.all(codes[0] == 0) and torch.all(codes[2] == 0)


# ------------------------------------------------------------------ indexer scores
W = synth.WORKLOADS
SCORE_CASES = {
    "tiny": W["tiny_full_decode"],
    "ragged_planted": W["full_decode_64k"].scaled(batch=3, n_q=2, n_keys=5003, q_pos0=4000),
    "ratio2": W["prefill_chunk_m2"].scaled(batch=2, n_q=3, n_keys=3001, q_pos0=5000, seed=9),
    # a chunk of 11 queries (groups of 4 queries, the last one ragged) whose visible
    # lengths cross a tile boundary (2,048) inside a group
    "chunk_groups": W["prefill_chunk_m2"].scaled(batch=2, n_q=11, n_keys=2100, q_pos0=4090, seed=11),
    "d32_h1": W["tiny_full_decode"].scaled(batch=2, n_keys=777, q_pos0=776, idx_heads=1, idx_dim=32),
    "ties": W["hier_indexer_1m"].scaled(batch=2, n_keys=20000, q_pos0=19999, palette=64),
    # decode stages are loaded through a view of the key rows in groups of four; a whole
    # stage that reaches into the last (B * n_keys) mod 4 rows is loaded plain instead
    "tensor_end": W["full_decode_64k"].scaled(batch=2, n_q=1, n_keys=257, q_pos0=256, seed=5),
}


def sel_key(s):
    """Selection key of float32 scores as include/csa2.h defines it (NaN 0, -0 as +0)."""
    s = np.asarray(s, np.float32)
    u = s.view(np.uint32).copy()
    u[u == 0x80000000] = 0
    key = np.where(u & np.uint32(0x80000000), ~u, u | np.uint32(0x80000000)).astype(np.uint32)
    key[np.isnan(s)] = 0
    return key


def group_keys(s_valid):
    """Largest selection key of each group of 32 consecutive valid candidates."""
    k = sel_key(s_valid)
    ng = (k.size + 31) // 32
    pad = np.zeros(ng * 32, np.uint32)
    pad[:k.size] = k
    return pad.reshape(ng, 32).max(axis=1)


def _with_group_max(dw, w, pool=None, st=None):
    """The indexer again with its group-maximum output, then Top-K (exact order) fed from it."""
    n_cand = w.n_keys if pool is None else pool.shape[-1] * w.block
    gm = torch.full((w.batch, w.n_q, (n_cand + 31) // 32), -1, dtype=torch.int32, device=DEV)
    scores, row_len, args = csa2.index_score(dw["q_idx"], dw["w_idx"], dw["k_codes"], dw["k_scales"],
                                             dw["q_pos"], w.ratio_m, pool, w.block, st, group_max=gm,
                                             want_args=True)
    idx = csa2.topk(scores, w.topk, row_len, pool, w.block, d_status=st, group_max=gm, exact=args)
    return scores, gm, idx


def score_order(n_q, idx_dim, idx_heads, pool=False):
    """Summation order of the float32 scores the indexer writes (include/csa2.h): the
    chunk kernel (Full mode, >= 8 queries a sequence, head dim 128, <= 32 heads) adds the
    heads in eight partial chains, every other kernel in one chain."""
    return "split8" if (not pool and n_q >= 8 and idx_dim == 128 and idx_heads <= 32) else "chain"


def _oracle_row_scores(w, b, t, qi, ww, kc, ks, pos, pool=False):
    qc, qs = oracle.quant_mxfp4(f32(qi[t]))
    return oracle.index_scores(qc, qs, ww[t], kc, ks, pos,
                               order=score_order(w.n_q, w.idx_dim, w.idx_heads, pool))


def _oracle_row_exact(w, b, t, qi, ww, kc, ks, pos):
    qc, qs = oracle.quant_mxfp4(f32(qi[t]))
    return oracle.index_scores_exact(qc, qs, ww[t], kc, ks, pos)


@pytest.mark.parametrize("name", list(SCORE_CASES))
def test_full_scores_topk_blocks(name):
    w = SCORE_CASES[name]
    st = status()
    dw = workload.build(w, kv=False, device=DEV, d_status=st)
    scores, row_len, args = csa2.index_score(dw["q_idx"], dw["w_idx"], dw["k_codes"], dw["k_scales"],
                                             dw["q_pos"], w.ratio_m, None, w.block, st, want_args=True)
    idx = csa2.topk(scores, w.topk, row_len, d_status=st, exact=args)
    idx_f = csa2.topk(scores, w.topk, row_len, d_status=st)          # float order of the scores
    nb = min(w.n_blocks, 300)
    blocks = csa2.block_candidates(scores, nb, row_len, w.block, st, exact=args)
    blocks_f = csa2.block_candidates(scores, nb, row_len, w.block, st)
    scores_g, gm, idx_g = _with_group_max(dw, w, None, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    qi_all, ww_all, _ = synth.gen_queries(w)
    qpos = synth.q_positions(w)
    for b in range(w.batch):
        kc, ks = oracle.quant_mxfp4(f32(synth.gen_index_keys(w, b, qi_all[b], ww_all[b])))
        assert np.array_equal(dw["k_codes"][b].cpu().numpy(), kc)
        for t in range(w.n_q):
            nvis = oracle.n_visible(int(qpos[b, t]), w.ratio_m, w.n_keys)
            assert int(row_len[b, t]) == nvis
            pos = np.arange(nvis)
            s_ref = _oracle_row_scores(w, b, t, qi_all[b], ww_all[b], kc, ks, pos)
            ex_ref = _oracle_row_exact(w, b, t, qi_all[b], ww_all[b], kc, ks, pos)
            s_gpu = scores[b, t, :nvis].cpu().numpy()
            assert same_f32(s_gpu, s_ref), f"{name} b={b} t={t}"
            assert np.array_equal(idx[b, t].cpu().numpy(), oracle.topk_exact(ex_ref, pos, w.topk))
            assert np.array_equal(blocks[b, t].cpu().numpy(),
                                  oracle.block_candidates_exact(ex_ref, nvis, w.block, nb))
            assert np.array_equal(idx_f[b, t].cpu().numpy(), oracle.topk(s_ref, pos, w.topk))
            assert np.array_equal(blocks_f[b, t].cpu().numpy(),
                                  oracle.block_candidates(s_ref, nvis, w.block, nb))
            # group-maximum output and Top-K fed from it
            assert same_f32(scores_g[b, t, :nvis].cpu().numpy(), s_ref)
            ng = (nvis + 31) // 32
            assert np.array_equal(gm[b, t, :ng].cpu().numpy().view(np.uint32), group_keys(s_ref))
            assert np.array_equal(idx_g[b, t].cpu().numpy(), idx[b, t].cpu().numpy())


@pytest.mark.parametrize("T,sparse,N", [(2, False, 3000), (2, True, 3001), (9, False, 3000), (9, True, 3000)])
def test_scores_wide_exponents(T, sparse, N):
    # random FP4 codes with scale bytes over the whole E8M0 range and queries spanning
    # 2^-60 .. 2^60 per block: the kernels' wide-sum and overflow paths.  T = 9 takes the
    # four-queries-per-CTA kernel (stages flagged and re-checked after its main loop);
    # `sparse` keeps ordinary scales except at 1% of the positions, so only some stages
    # are flagged and only some positions of those need re-scoring.  N = 3,001 puts the
    # second sequence's rows and scale words off the 4-row grid.
    rng = np.random.default_rng(17 + T + int(sparse))
    B, H, d = 2, 8, 128
    kc = rng.integers(0, 256, size=(B, N, d // 2), dtype=np.uint8)
    ks = rng.integers(0, 255, size=(B, N, d // 32)).astype(np.uint8)
    if sparse:
        wide = rng.random((B, N)) < 0.01
        ks = np.where(wide[..., None], ks, rng.integers(125, 130, size=ks.shape)).astype(np.uint8)
    q = rng.standard_normal((B, T, H, d)).astype(np.float32)
    qe = rng.integers(-60, 60, size=(B, T, H, d // 32, 1)) if not sparse else rng.integers(-2, 3, size=(B, T, H, d // 32, 1))
    q *= np.exp2(qe).astype(np.float32).reshape(B, T, H, d // 32, 1).repeat(32, -1).reshape(B, T, H, d)
    qbits = synth.f32_to_bf16_bits(q)
    wv = rng.standard_normal((B, T, H)).astype(np.float32)
    qt = workload.bf16_tensor(qbits, DEV)
    gm = torch.full((B, T, (N + 31) // 32), -1, dtype=torch.int32, device=DEV)
    scores, row_len = csa2.index_score(qt, torch.from_numpy(wv).to(DEV), torch.from_numpy(kc).to(DEV),
                                       torch.from_numpy(ks).to(DEV), group_max=gm)
    torch.cuda.synchronize()
    for b in range(B):
        for t in range(T):
            qc, qs = oracle.quant_mxfp4(f32(qbits[b, t]))
            s_ref = oracle.index_scores(qc, qs, wv[b, t], kc[b], ks[b], np.arange(N),
                                        order=score_order(T, d, H))
            assert same_f32(scores[b, t].cpu().numpy(), s_ref)
            # groups re-scored by the exact pass carry the exact scores' maxima
            assert np.array_equal(gm[b, t].cpu().numpy().view(np.uint32), group_keys(s_ref))


@pytest.mark.parametrize("n_keys,q_pos0", [(40000, 30000), (40003, 40001)])
def test_pool_scores_and_topk(n_keys, q_pos0):
    # 40,003 rows a sequence put the second and third sequences' scale words off the
    # 16-byte grid (their blocks' words are copied one by one) and end in a partial block
    w = W["reuse_reindex_decode_128k"].scaled(batch=3, n_q=2, n_keys=n_keys, q_pos0=q_pos0,
                                              n_blocks=700)
    st = status()
    dw = workload.build(w, kv=False, device=DEV, d_status=st)
    pool = dw["pool"].clone()
    pool[1, 0, 650:] = -1                              # -1 padding
    scores, row_len, args = csa2.index_score(dw["q_idx"], dw["w_idx"], dw["k_codes"], dw["k_scales"],
                                             dw["q_pos"], 1, pool, w.block, st, want_args=True)
    idx = csa2.topk(scores, w.topk, row_len, pool, w.block, d_status=st, exact=args)
    idx_f = csa2.topk(scores, w.topk, row_len, pool, w.block, d_status=st)
    _, gm, idx_g = _with_group_max(dw, w, pool, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    qi_all, ww_all, _ = synth.gen_queries(w)
    qpos = synth.q_positions(w)
    pool_np = pool.cpu().numpy()
    for b in range(w.batch):
        kc, ks = oracle.quant_mxfp4(f32(synth.gen_index_keys(w, b, qi_all[b], ww_all[b])))
        for t in range(w.n_q):
            nvis = oracle.n_visible(int(qpos[b, t]), 1, w.n_keys)
            pos = oracle.pool_positions(pool_np[b, t], w.block, nvis)
            assert int(row_len[b, t]) == pos.size
            s_ref = _oracle_row_scores(w, b, t, qi_all[b], ww_all[b], kc, ks, pos, pool=True)
            assert same_f32(scores[b, t, :pos.size].cpu().numpy(), s_ref)
            ng = (pos.size + 31) // 32
            assert np.array_equal(gm[b, t, :ng].cpu().numpy().view(np.uint32), group_keys(s_ref))
            assert np.array_equal(idx_g[b, t].cpu().numpy(), idx[b, t].cpu().numpy())
            idx_ref, _, _ = oracle.reindex_indexer(f32(qi_all[b, t]), ww_all[b, t], kc, ks,
                                                   int(qpos[b, t]), 1, pool_np[b, t], w.topk, w.block,
                                                   want_f32=False)
            assert np.array_equal(idx[b, t].cpu().numpy(), idx_ref)
            assert np.array_equal(idx_f[b, t].cpu().numpy(), oracle.topk(s_ref, pos, w.topk))


def _near_tie_case(N, seed, neg=False, tiny_exp=-30):
    """Keys whose float32 scores tie while their exact scores differ: two heads with
    w = (1, 2^tiny_exp) (negative: (1, -2^tiny_exp)).  Every key has the same block-0 dot with head 0;
    head 1 reads a block whose dot is a different small integer per key.  The float32
    chain rounds 2^-30 * d_1 away, so the float order is the position order; the exact
    order follows d_1."""
    rng = np.random.default_rng(seed)
    d = 128
    q = np.zeros((1, 1, 2, d), np.float32)
    q[0, 0, 0, :32] = 1.0                              # head 0: block 0
    q[0, 0, 1, 32:64] = 1.0                            # head 1: block 1
    k = np.zeros((1, N, d), np.float32)
    k[0, :, :32] = 0.5                                 # d_0 = 16 for every key
    k[0, :, 32:64] = rng.integers(0, 7, size=(N, 32)) * 0.5 * (rng.random((N, 32)) < 0.3)
    k[0, :, 36] = 3.0                                  # block amax 3: scale 2^-1, values exact
    wv = np.array([[[1.0, (-1.0 if neg else 1.0) * 2.0 ** tiny_exp]]], np.float32)
    return q, k, wv


@pytest.mark.parametrize("N,neg,tiny_exp", [(1500, False, -30), (2000, True, -30), (700, False, -100),
                                            (900, True, -100)])
def test_exact_order_resolves_float32_ties(N, neg, tiny_exp):
    # the whole row is one float32 tie group within the error bound: the band holds every
    # position (<= 2,048) and the exact pass orders them by their low-order bits
    q, k, wv = _near_tie_case(N, N + neg, neg, tiny_exp)
    qb, kb = synth.f32_to_bf16_bits(q), synth.f32_to_bf16_bits(k)
    assert np.array_equal(f32(qb), q) and np.array_equal(f32(kb), k)
    st = status()
    kt = workload.bf16_tensor(kb, DEV)
    kc, ks = csa2.quant_fp4(kt, st)
    wt = torch.from_numpy(wv).to(DEV)
    scores, row_len, args = csa2.index_score(workload.bf16_tensor(qb, DEV), wt, kc, ks, d_status=st,
                                             want_args=True)
    K = 512
    idx = csa2.topk(scores, K, row_len, d_status=st, exact=args)
    blocks = csa2.block_candidates(scores, 40, row_len, 8, st, exact=args)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    kc_o, ks_o = oracle.quant_mxfp4(k[0])
    qc_o, qs_o = oracle.quant_mxfp4(q[0, 0])
    pos = np.arange(N)
    s_ref = oracle.index_scores(qc_o, qs_o, wv[0, 0], kc_o, ks_o, pos)
    ex = oracle.index_scores_exact(qc_o, qs_o, wv[0, 0], kc_o, ks_o, pos)
    assert np.all(s_ref == s_ref[0])                     # one float32 value for the whole row
    ref = oracle.topk_exact(ex, pos, K)
    assert not np.array_equal(ref, oracle.topk(s_ref, pos, K))
    assert np.array_equal(idx[0, 0].cpu().numpy(), ref)
    assert np.array_equal(blocks[0, 0].cpu().numpy(), oracle.block_candidates_exact(ex, N, 8, 40))


FUSED_CASES = dict(SCORE_CASES)
FUSED_CASES.update({
    # more candidates than the 32 stages x 256 positions one CTA keeps: the row takes
    # at least 9 CTAs whatever the SM count
    "decode_70k": W["full_decode_64k"].scaled(batch=2, n_q=1, n_keys=70001, q_pos0=70000, seed=31),
    # fewer visible positions than K: every list holds all of its positions
    "short_rows": W["full_decode_64k"].scaled(batch=3, n_q=1, n_keys=900, q_pos0=300, seed=32),
    "ties_decode": W["hier_indexer_1m"].scaled(batch=2, n_keys=30000, q_pos0=29999, palette=32),
})


@pytest.mark.parametrize("name", list(FUSED_CASES))
def test_index_topk_equals_scores_then_topk(name):
    # csa2_index_topk (no score matrix where the indexer takes one query per CTA) gives
    # exactly what csa2_index_score + exact csa2_topk give
    w = FUSED_CASES[name]
    st = status()
    dw = workload.build(w, kv=False, device=DEV, d_status=st)
    scores, row_len, args = csa2.index_score(dw["q_idx"], dw["w_idx"], dw["k_codes"], dw["k_scales"],
                                             dw["q_pos"], w.ratio_m, None, w.block, st, want_args=True)
    ref, ref_s = csa2.topk(scores, w.topk, row_len, d_status=st, exact=args, want_scores=True)
    idx, rl, out_s = csa2.index_topk(dw["q_idx"], dw["w_idx"], dw["k_codes"], dw["k_scales"], w.topk,
                                     dw["q_pos"], w.ratio_m, d_status=st, want_scores=True)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(rl, row_len)
    assert torch.equal(idx, ref)
    # scores of the selected entries (the fused call returns -0 as +0)
    assert torch.equal(out_s, ref_s + 0.0)


def test_index_after_cache_write_with_fresh_from():
    # the cache write of the decoded token (csa2_rope_quant_fp4, which lets the next kernel
    # start early) directly followed by the indexer with fresh_from = that token's
    # position: the indexer streams the older positions before its dependency wait and must
    # still see the new row.  Each round writes a different row; the scores equal those of
    # a call made after a full synchronisation.
    w = W["full_decode_64k"].scaled(batch=4, n_q=1, n_keys=20000, q_pos0=19999, seed=43)
    st = status()
    dw = workload.build(w, kv=False, device=DEV, d_status=st)
    last = w.n_keys - 1
    kc, ks = dw["k_codes"], dw["k_scales"]
    gen = torch.Generator().manual_seed(44)
    scores = torch.empty((w.batch, 1, w.n_keys), dtype=torch.float32, device=DEV)
    row_len = torch.empty((w.batch, 1), dtype=torch.int32, device=DEV)
    args = csa2.make_index_args(dw["q_idx"], dw["w_idx"], kc, ks, dw["q_pos"], 1)
    args.fresh_from = last
    ref_args = csa2.make_index_args(dw["q_idx"], dw["w_idx"], kc, ks, dw["q_pos"], 1)
    ws = torch.zeros(max(1, csa2.load().csa2_index_score_workspace_size(ctypes.byref(args))), dtype=torch.uint8,
                     device=DEV)
    idx = torch.empty((w.batch, 1, w.topk), dtype=torch.int32, device=DEV)
    wsf = torch.zeros(csa2.load().csa2_index_topk_workspace_size(ctypes.byref(args), w.topk), dtype=torch.uint8,
                      device=DEV)
    for r in range(4):
        new_k = (torch.randn((w.batch, w.idx_dim), generator=gen) * (2.0 + 10 * r)).to(torch.bfloat16).to(DEV)
        jobs = [(new_k, kc[:, last], ks[:, last], 0, None, None, csa2.FMT_MXFP4)]
        csa2.csa2_rope_quant_fp4(jobs, st)
        csa2.csa2_index_score(args, scores, row_len, st, workspace=ws)
        csa2.csa2_rope_quant_fp4(jobs, st)                 # the same row again, then the fused call
        csa2.csa2_index_topk(args, w.topk, idx, None, None, st, workspace=wsf)
        torch.cuda.synchronize()
        ref_s, ref_l = csa2.index_score(dw["q_idx"], dw["w_idx"], kc, ks, dw["q_pos"], 1)
        ref_idx = csa2.topk(ref_s, w.topk, ref_l, d_status=st, exact=ref_args)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert torch.equal(row_len, ref_l)
        assert np.array_equal(scores.cpu().numpy().view(np.uint32), ref_s.cpu().numpy().view(np.uint32)), r
        assert torch.equal(idx, ref_idx), r


def test_index_topk_negative_weights_and_near_ties():
    # head weights of both signs (the CTAs keep every position: the bound needs the whole
    # sequence) and a float32 tie group resolved by the exact order
    w = W["full_decode_64k"].scaled(batch=2, n_q=3, n_keys=9000, q_pos0=8999, plant_frac=0.0, seed=23)
    st = status()
    dw = workload.build(w, kv=False, device=DEV, d_status=st)
    wn = torch.randn(dw["w_idx"].shape, generator=torch.Generator().manual_seed(5)).to(DEV)
    scores, row_len, args = csa2.index_score(dw["q_idx"], wn, dw["k_codes"], dw["k_scales"],
                                             dw["q_pos"], 1, None, w.block, st, want_args=True)
    ref = csa2.topk(scores, w.topk, row_len, d_status=st, exact=args)
    idx, rl = csa2.index_topk(dw["q_idx"], wn, dw["k_codes"], dw["k_scales"], w.topk, dw["q_pos"], 1,
                              d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(idx, ref) and torch.equal(rl, row_len)
    q, k, wv = _near_tie_case(1500, 41)
    qb, kb = synth.f32_to_bf16_bits(q), synth.f32_to_bf16_bits(k)
    kc, ks = csa2.quant_fp4(workload.bf16_tensor(kb, DEV), st)
    qt, wt = workload.bf16_tensor(qb, DEV), torch.from_numpy(wv).to(DEV)
    scores, row_len, args = csa2.index_score(qt, wt, kc, ks, d_status=st, want_args=True)
    ref = csa2.topk(scores, 512, row_len, d_status=st, exact=args)
    idx, _ = csa2.index_topk(qt, wt, kc, ks, 512, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert torch.equal(idx, ref)


def test_exact_order_long_row_spread_tie_group():
    # a row of 70,001 positions: a float32 tie group of 1,000 positions spread over the
    # whole row holds the top 512, whose exact order comes from the tiny second head; the
    # filler keys (one float32 value too) score lower
    N = 70001
    q, k, wv = _near_tie_case(N, 77)
    rng = np.random.default_rng(78)
    tie = np.zeros(N, bool)
    tie[rng.choice(N, 1000, replace=False)] = True
    k[0, ~tie, :32] = 0.25                             # d_0 = 8 for the filler keys
    qb, kb = synth.f32_to_bf16_bits(q), synth.f32_to_bf16_bits(k)
    assert np.array_equal(f32(kb), k)
    st = status()
    kc, ks = csa2.quant_fp4(workload.bf16_tensor(kb, DEV), st)
    wt = torch.from_numpy(wv).to(DEV)
    scores, row_len, args = csa2.index_score(workload.bf16_tensor(qb, DEV), wt, kc, ks, d_status=st,
                                             want_args=True)
    K = 512
    idx = csa2.topk(scores, K, row_len, d_status=st, exact=args)
    idx_f = csa2.topk(scores, K, row_len, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    kc_o, ks_o = oracle.quant_mxfp4(k[0])
    qc_o, qs_o = oracle.quant_mxfp4(q[0, 0])
    pos = np.arange(N)
    s_ref = oracle.index_scores(qc_o, qs_o, wv[0, 0], kc_o, ks_o, pos)
    ex = oracle.index_scores_exact(qc_o, qs_o, wv[0, 0], kc_o, ks_o, pos)
    assert np.all(s_ref[tie] == s_ref[tie][0]) and s_ref[~tie].max() < s_ref[tie][0]
    ref = oracle.topk_exact(ex, pos, K)
    assert not np.array_equal(ref, oracle.topk(s_ref, pos, K))
    assert np.array_equal(idx[0, 0].cpu().numpy(), ref)
    assert np.array_equal(idx_f[0, 0].cpu().numpy(), oracle.topk(s_ref, pos, K))


def test_exact_order_long_rows_negative_weights():
    # three rows of 100,003 positions with head weights of both signs, one row shortened to
    # 40,000 positions and one to K + 1
    w = W["full_decode_64k"].scaled(batch=3, n_q=1, n_keys=100003, q_pos0=100002, plant_frac=0.01, seed=29)
    st = status()
    dw = workload.build(w, kv=False, device=DEV, d_status=st)
    wn = torch.randn(dw["w_idx"].shape, generator=torch.Generator().manual_seed(6)).to(DEV)
    scores, row_len, args = csa2.index_score(dw["q_idx"], wn, dw["k_codes"], dw["k_scales"],
                                             dw["q_pos"], 1, None, w.block, st, want_args=True)
    lens = torch.tensor([[100003], [40000], [w.topk + 1]], dtype=torch.int32, device=DEV)
    row_len = torch.minimum(row_len, lens)
    idx = csa2.topk(scores, w.topk, row_len, d_status=st, exact=args)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    qi_all, ww_all, _ = synth.gen_queries(w)
    wn_np = wn.cpu().numpy()
    for b in range(w.batch):
        kc, ks = oracle.quant_mxfp4(f32(synth.gen_index_keys(w, b, qi_all[b], ww_all[b])))
        L = int(row_len[b, 0])
        pos = np.arange(L)
        ex = _oracle_row_exact(w, b, 0, qi_all[b], wn_np[b], kc, ks, pos)
        assert np.array_equal(idx[b, 0].cpu().numpy(), oracle.topk_exact(ex, pos, w.topk)), b


def test_exact_order_negative_weights():
    # realistic scales with head weights of both signs: the row bound comes from the key
    # scale maxima; the selections equal the exact ones
    w = W["full_decode_64k"].scaled(batch=2, n_q=3, n_keys=9000, q_pos0=8999, plant_frac=0.0, seed=23)
    st = status()
    dw = workload.build(w, kv=False, device=DEV, d_status=st)
    wn = torch.randn(dw["w_idx"].shape, generator=torch.Generator().manual_seed(5)).to(DEV)
    scores, row_len, args = csa2.index_score(dw["q_idx"], wn, dw["k_codes"], dw["k_scales"],
                                             dw["q_pos"], 1, None, w.block, st, want_args=True)
    idx = csa2.topk(scores, w.topk, row_len, d_status=st, exact=args)
    blocks = csa2.block_candidates(scores, 300, row_len, w.block, st, exact=args)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    qi_all, ww_all, _ = synth.gen_queries(w)
    wn_np = wn.cpu().numpy()
    for b in range(w.batch):
        kc, ks = oracle.quant_mxfp4(f32(synth.gen_index_keys(w, b, qi_all[b], ww_all[b])))
        for t in range(w.n_q):
            pos = np.arange(w.n_keys)
            ex = _oracle_row_exact(w, b, t, qi_all[b], wn_np[b], kc, ks, pos)
            assert np.array_equal(idx[b, t].cpu().numpy(), oracle.topk_exact(ex, pos, w.topk))
            assert np.array_equal(blocks[b, t].cpu().numpy(),
                                  oracle.block_candidates_exact(ex, w.n_keys, w.block, 300))


def test_index_workspace_left_zeroed():
    """The indexer's workspace (per-row tile counters) must be zero-filled before its first
    use and is left zero-filled by every call: three calls on one workspace agree bit for
    bit, and the workspace reads all zero after each."""
    w = SCORE_CASES["ragged_planted"]
    dw = workload.build(w, kv=False, device=DEV)
    args = csa2.make_index_args(dw["q_idx"], dw["w_idx"], dw["k_codes"], dw["k_scales"], dw["q_pos"],
                                w.ratio_m)
    need = csa2.load().csa2_index_score_workspace_size(ctypes.byref(args))
    assert need > 0
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    outs = []
    for _ in range(3):
        sc = torch.empty((w.batch, w.n_q, w.n_keys), dtype=torch.float32, device=DEV)
        rl = torch.empty((w.batch, w.n_q), dtype=torch.int32, device=DEV)
        csa2.csa2_index_score(args, sc, rl, workspace=ws)
        torch.cuda.synchronize()
        assert int(ws.count_nonzero()) == 0
        outs.append((sc, rl))
    for sc, rl in outs[1:]:
        assert torch.equal(rl, outs[0][1])
        for b in range(w.batch):
            for t in range(w.n_q):
                L = int(rl[b, t])
                assert np.array_equal(sc[b, t, :L].cpu().numpy().view(np.uint32),
                                      outs[0][0][b, t, :L].cpu().numpy().view(np.uint32))


def test_pool_flags_bad_order():
    w = W["reuse_reindex_decode_128k"].scaled(batch=1, n_keys=4096, q_pos0=4095, n_blocks=64)
    dw = workload.build(w, kv=False, device=DEV)
    pool = dw["pool"].clone()
    pool[0, 0, 5], pool[0, 0, 6] = pool[0, 0, 6].item(), pool[0, 0, 5].item()
    st = status()
    csa2.index_score(dw["q_idx"], dw["w_idx"], dw["k_codes"], dw["k_scales"], dw["q_pos"], 1,
                     pool, 8, st)
    torch.cuda.synchronize()
    assert int(st.item()) & csa2.DEV_BAD_POOL


# ------------------------------------------------------------------ selection on given scores
@pytest.mark.parametrize("rows,n,k,levels", [(3, 300000, 512, 7), (5, 1000, 512, 3), (2, 70000, 2048, 100000),
                                             (4, 4097, 1, 2), (1, 1 << 20, 512, 1 << 20),
                                             (2, 600000, 2048, 50000)])
def test_topk_on_given_scores(rows, n, k, levels):
    rng = np.random.default_rng(rows * n + k)
    s = (rng.integers(0, levels, size=(rows, n)).astype(np.float32) - levels // 2) * np.float32(0.5)
    s[0, ::97] = np.nan
    s[0, 1::89] = -0.0
    s[-1, ::5] = -np.inf
    row_len = rng.integers(0, n + 1, size=rows).astype(np.int32)
    row_len[0] = n
    idx = csa2.topk(torch.from_numpy(s).to(DEV), k, torch.from_numpy(row_len).to(DEV))
    bl = csa2.block_candidates(torch.from_numpy(s).to(DEV), min(k, 2048),
                               torch.from_numpy(row_len).to(DEV), 8)
    torch.cuda.synchronize()
    for r in range(rows):
        L = int(row_len[r])
        assert np.array_equal(idx[r].cpu().numpy(), oracle.topk(s[r, :L], np.arange(L), k))
        assert np.array_equal(bl[r].cpu().numpy(), oracle.block_candidates(s[r], L, 8, min(k, 2048)))


# ------------------------------------------------------------------ attention
def _attn_check(o_gpu, lse_gpu, o_ref, lse_ref):
    o_gpu = o_gpu.astype(np.float64)
    den = np.maximum(np.abs(o_ref).max(axis=-1), 1e-6)
    err = np.abs(o_gpu - o_ref).max(axis=-1) / den
    assert err.max() <= ATTN_TOL, f"max row-relative error {err.max():.3e}"
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse_gpu), fin)
    assert np.abs(lse_gpu[fin] - lse_ref[fin]).max(initial=0) <= LSE_TOL
    return err.max()


def _oracle_attention(w, dw_rows, idx_np, t_range, swa_start=None, kv_fmt="mxfp4", swa8=False):
    """fp64 oracle attention for rows (b, t) with the given idx (swa8: the SWA rows as their
    MXFP8 values)."""
    qpos = synth.q_positions(w)
    n_slots, pos0 = synth.swa_layout(w)
    _, _, qa = synth.gen_queries(w)
    outs, lses = {}, {}
    for b in dw_rows:
        kvc, kvs = oracle.quant_main_kv(f32(synth.gen_main_kv(w, b)), kv_fmt)
        swa = f32(synth.gen_swa(w, b)).astype(np.float64)
        if swa8:
            swa = oracle.dequant_mxfp8(*oracle.quant_mxfp8(swa))
        s0 = 0 if swa_start is None else int(swa_start[b])
        for t in t_range:
            keys = oracle.gather_keys(idx_np[b, t], kvc, kvs, swa, int(qpos[b, t]), pos0, w.window, s0)
            o, l = oracle.attention_rows(f32(qa[b, t])[None].astype(np.float64), [keys],
                                         1.0 / math.sqrt(w.d_qk), w.d_v)
            outs[(b, t)], lses[(b, t)] = o[0], l[0]
    return outs, lses


ATTN_CASES = {
    "tiny": (W["tiny_full_decode"], None),
    "prod_dims_T3": (W["full_decode_64k"].scaled(batch=2, n_q=3, n_keys=3000, q_pos0=2000), None),
    "replay_start": (W["full_decode_64k"].scaled(batch=2, n_q=2, n_keys=1500, q_pos0=1400, heads=20), [1350, 0]),
    "d_v_odd_heads": (W["tiny_full_decode"].scaled(batch=1, n_q=2, heads=5, d_qk=96, d_v=40, n_keys=900, q_pos0=899, topk=100, window=17), None),
}


@pytest.mark.parametrize("name,kv_fmt,swa8", [(n, "mxfp4", False) for n in ATTN_CASES] +
                         [("prod_dims_T3", "nvfp4", False), ("replay_start", "nvfp4", False),
                          ("tiny", "nvfp4", False), ("d_v_odd_heads", "nvfp4", False),
                          ("prod_dims_T3", "nvfp4", True), ("replay_start", "mxfp4", True),
                          ("tiny", "mxfp4", True), ("d_v_odd_heads", "nvfp4", True)])
def test_attention_parity(name, kv_fmt, swa8):
    # kv_fmt "nvfp4": the main KV in the report's E2M1 + E4M3/16 format (tensor-core kernel
    # for the production dims, CUDA-core kernel for the others); swa8: the SWA window in
    # MXFP8, the report's FP8 SWA cache (with nvfp4: the pages' whole cache configuration)
    w, swa_start = ATTN_CASES[name]
    st = status()
    fmt = csa2.FMT_NVFP4_E4M3_16 if kv_fmt == "nvfp4" else csa2.FMT_MXFP4
    dw = workload.build(w, kidx=False, device=DEV, d_status=st, kv_fmt=fmt, swa_fp8=swa8)
    rng = np.random.default_rng(3)
    idx = np.stack([np.stack([np.sort(rng.choice(w.n_keys, w.topk, replace=False)) for _ in range(w.n_q)])
                    for _ in range(w.batch)]).astype(np.int32)
    idx[0, 0, -7:] = -1                                  # padding
    idx[-1, -1, :3] = idx[-1, -1, 3]                     # duplicates are kept
    ss = None if swa_start is None else torch.tensor(swa_start, dtype=torch.int32, device=DEV)
    swa = dw["swa8"] if swa8 else dw["swa"]
    out, lse = csa2.sparse_attn(dw["q_attn"], dw["kv_codes"], dw["kv_scales"],
                                torch.from_numpy(idx).to(DEV), swa, dw["swa_pos0"], dw["q_pos"],
                                ss, w.window, dw.sm_scale, w.d_v, d_status=st,
                                swa_scales=dw["swa8_scales"] if swa8 else None)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    o_ref, l_ref = _oracle_attention(w, range(w.batch), idx, range(w.n_q), swa_start, kv_fmt, swa8)
    for (b, t), o in o_ref.items():
        _attn_check(out[b, t].float().cpu().numpy(), lse[b, t].cpu().numpy(), o, l_ref[(b, t)])


def test_attention_bad_index_and_empty():
    w = W["tiny_full_decode"].scaled(batch=2, n_keys=600, q_pos0=599, topk=16)
    dw = workload.build(w, kidx=False, device=DEV)
    idx = np.full((2, 1, 16), -1, np.int32)
    idx[0, 0, :4] = [5, 700, -3, 9]                       # 700 and -3 are out of range
    st = status()
    out, lse = csa2.sparse_attn(dw["q_attn"], dw["kv_codes"], dw["kv_scales"],
                                torch.from_numpy(idx).to(DEV), None, None, None, None, w.window,
                                dw.sm_scale, w.d_v, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & csa2.DEV_BAD_INDEX
    # row 1 has no keys at all: zeros and -inf
    assert torch.all(out[1] == 0) and torch.all(torch.isneginf(lse[1]))
    o_ref, l_ref = _oracle_attention(w.scaled(window=0), [0], np.where(idx >= 600, -1, idx), [0])
    _attn_check(out[0, 0].float().cpu().numpy(), lse[0, 0].cpu().numpy(), o_ref[(0, 0)], l_ref[(0, 0)])


# ------------------------------------------------------------------ failure detection
def test_bounded_wait_gives_up_and_context_survives():
    # no fault involved: one CTA waits, through the kernels' own bounded-wait routine, on an
    # mbarrier that nothing completes; the wait must end after its poll limit with
    # CSA2_DEV_TIMEOUT, and the next call on the stream must run normally
    st = status()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    csa2.csa2_selftest_bounded_wait(1024, st)
    e1.record()
    torch.cuda.synchronize()
    assert int(st.item()) & csa2.DEV_TIMEOUT
    ms = e0.elapsed_time(e1)
    print(f"1,024 polls of an mbarrier that never completes: {ms:.3f} ms")
    assert ms < 5000.0
    raw, x = _codec_inputs(64, 64, 5, True)
    st2 = status()
    codes, scales = csa2.quant_fp4(workload.bf16_tensor(raw, DEV), st2)
    c_ref, s_ref = oracle.quant_mxfp4(x)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    assert np.array_equal(codes.cpu().numpy(), c_ref) and np.array_equal(scales.cpu().numpy(), s_ref)
