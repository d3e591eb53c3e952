"""CPU oracle for the CSA2 decode/prefill path -- TEST INFRASTRUCTURE.

Only the tests, the package's smoke check and the benchmark's CPU-baseline leg may
import this package.  The product library never loads it, and it shares no code
with the CUDA sources: the arithmetic lives in ``csa2_oracle.c`` (plain loops,
exact integers, fp64), selection here uses a library sort.

What it computes, step by step (DeepSeek-V4.1-Flash report, aipaper.jasonlin.tech):
  1. MXFP4 codec for indexer q/k and the main KV (report §2.4.4; OCP MX v1.0 rule);
     the report's own main-KV format, E2M1 + E4M3 per 16 (report §2.4.4), as an option.
  2. Indexer score of every candidate position, s = sum_h w_h ReLU(q_h . k), exact:
     the dots of the MXFP4 vectors and the weighted head sum are carried out in wide
     integers with nothing rounded (``index_scores_exact``).  The float32 scores the
     library writes out beside its selection (each head dot rounded once to float32,
     the head sum a float32 fma chain) are reproduced by ``index_scores``.
  3. Top-K (K = 512, report §4.2.1): full sort by (-exact score, position); emitted in
     ascending position order, padded with -1.
  4. Hierarchical pool (report §2.3.2): block score = max exact score of the block's
     visible positions (8 per block); top 2,048 blocks by (-score, block id);
     ascending, -1 pad.
  5. Reindex (report §2.3.2; review page, notes on the official code: scores over the
     full range, then a candidate mask): only pool positions compete.
  6. Core attention in fp64 over the selected main-KV entries (dequantised) followed by
     the SWA keys in [max(s, i-W+1), i] (report §2.3.1, §3.2.2).

Parity of the attention values at scale is pinned only by closed forms, library
special cases and invariants (see tests); the pages print no attention outputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa2_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libcsa2_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11 + OpenMP)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off",
                               "-fno-fast-math", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            I = ctypes.c_int
            lib.orc_quant_mxfp4.argtypes = [P, I64, I64, P, P]
            lib.orc_dequant_mxfp4.argtypes = [P, P, I64, I64, P]
            lib.orc_quant_nvfp4.argtypes = [P, I64, I64, P, P]
            lib.orc_dequant_nvfp4.argtypes = [P, P, I64, I64, P]
            lib.orc_quant_mxfp8.argtypes = [P, I64, I64, P, P]
            lib.orc_dequant_mxfp8.argtypes = [P, P, I64, I64, P]
            lib.orc_head_dots.argtypes = [I, I, P, P, P, P, P, I64, P]
            lib.orc_index_scores.argtypes = [I, I, P, P, P, P, P, P, I64, P, I]
            lib.orc_index_scores_exact.argtypes = [I, I, P, P, P, P, P, P, I64, P]
            lib.orc_exact_limbs.restype = I
            lib.orc_exact_e0.restype = I
            lib.orc_attention.argtypes = [I64, I, I, I, P, P, P, ctypes.c_double, P, P]
            lib.orc_num_threads.restype = I
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_L().orc_num_threads())


# ---------------------------------------------------------------- MXFP4 codec
def quant_mxfp4(x: np.ndarray):
    """x [..., D] (float32/float64 holding exact values), D % 32 == 0 ->
    (codes uint8 [..., D/2], scales uint8 [..., D/32])."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    D = x.shape[-1]
    assert D % 32 == 0
    rows = x.size // D
    codes = np.empty(x.shape[:-1] + (D // 2,), np.uint8)
    scales = np.empty(x.shape[:-1] + (D // 32,), np.uint8)
    _L().orc_quant_mxfp4(_p(x), rows, D, _p(codes), _p(scales))
    return codes, scales


def dequant_mxfp4(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    D = codes.shape[-1] * 2
    rows = codes.size // (D // 2)
    y = np.empty(codes.shape[:-1] + (D,), np.float64)
    _L().orc_dequant_mxfp4(_p(codes), _p(scales), rows, D, _p(y))
    return y


# ---------------------------------------------------------------- E2M1 + E4M3/16 codec
def quant_nvfp4(x: np.ndarray):
    """Main-KV format of the report (§2.4.4): E2M1 codes with one E4M3 scale per 16
    values, no global scale.  x [..., D] (exact values), D % 16 == 0 ->
    (codes uint8 [..., D/2], scales uint8 [..., D/16]).  Scale = amax/6 rounded to the
    nearest E4M3 value (ties to even, clamped to 448); a zero scale zeroes the block."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    D = x.shape[-1]
    assert D % 16 == 0
    rows = x.size // D
    codes = np.empty(x.shape[:-1] + (D // 2,), np.uint8)
    scales = np.empty(x.shape[:-1] + (D // 16,), np.uint8)
    _L().orc_quant_nvfp4(_p(x), rows, D, _p(codes), _p(scales))
    return codes, scales


def dequant_nvfp4(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    D = codes.shape[-1] * 2
    rows = codes.size // (D // 2)
    y = np.empty(codes.shape[:-1] + (D,), np.float64)
    _L().orc_dequant_nvfp4(_p(codes), _p(scales), rows, D, _p(y))
    return y


# ---------------------------------------------------------------- MXFP8 (E4M3) SWA codec
def quant_mxfp8(x: np.ndarray):
    """SWA KV in FP8 (report §2.4.4), read as OCP MXFP8 with E4M3 elements: one E8M0 scale
    per 32 values, X = floor(log2 amax) - 8, elements rounded to nearest E4M3 (ties to even)
    and saturated at 448.  x [..., D] (exact values), D % 32 == 0 ->
    (codes uint8 [..., D], scales uint8 [..., D/32])."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    D = x.shape[-1]
    assert D % 32 == 0
    rows = x.size // D if D else 0
    codes = np.empty(x.shape, np.uint8)
    scales = np.empty(x.shape[:-1] + (D // 32,), np.uint8)
    _L().orc_quant_mxfp8(_p(x), rows, D, _p(codes), _p(scales))
    return codes, scales


def dequant_mxfp8(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.uint8)
    D = codes.shape[-1]
    rows = codes.size // D if D else 0
    y = np.empty(codes.shape, np.float64)
    _L().orc_dequant_mxfp8(_p(codes), _p(scales), rows, D, _p(y))
    return y


def quant_main_kv(x: np.ndarray, fmt: str = "mxfp4"):
    """Main-KV cache rows in format ``fmt`` ("mxfp4" or "nvfp4")."""
    return quant_nvfp4(x) if fmt == "nvfp4" else quant_mxfp4(x)


def dequant_main_kv(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Dequantise main-KV rows; the format follows from the scale count (D/16 scales:
    E2M1 + E4M3/16, D/32: MXFP4)."""
    D = codes.shape[-1] * 2
    return dequant_nvfp4(codes, scales) if scales.shape[-1] == D // 16 else dequant_mxfp4(codes, scales)


# ---------------------------------------------------------------- RoPE before the cache write
def rope_rotate(x: np.ndarray, pos: np.ndarray, cos_sin: np.ndarray, rope_dim: int) -> np.ndarray:
    """Rotary embedding of the trailing ``rope_dim`` channels of each row, the step the
    report (§2.4.4) places before the main-KV cache is quantised.

    The pages give no formula; the reading used: channel pairs (c0 + 2i, c0 + 2i + 1),
    c0 = cols - rope_dim, rotated by the caller's table row p = pos[r] (rope_dim/2 cosines
    then rope_dim/2 sines):  (a, b) -> (a c - b s, a s + b c).  The rotated values decide
    the integer codes, so they are computed in the kernel's float32 precision: one rounding
    per product and per sum, no fused multiply-add.  x [rows, cols] (float32 values) ->
    float32 [rows, cols]."""
    y = np.array(x, dtype=np.float32, copy=True)
    if rope_dim == 0 or y.shape[0] == 0:
        return y
    c0, h = y.shape[1] - rope_dim, rope_dim // 2
    tab = np.asarray(cos_sin, np.float32)[np.asarray(pos, np.int64)]
    c, s = tab[:, :h], tab[:, h:]
    a, b = y[:, c0::2].copy(), y[:, c0 + 1::2].copy()
    y[:, c0::2] = np.subtract(np.multiply(a, c), np.multiply(b, s))
    y[:, c0 + 1::2] = np.add(np.multiply(a, s), np.multiply(b, c))
    return y


def rope_quant(x: np.ndarray, pos, cos_sin, rope_dim: int, fmt: str = "mxfp4"):
    """Cache write of one main-KV (or key) row block: RoPE, then the 4-bit codec."""
    return quant_main_kv(rope_rotate(x, pos, cos_sin, rope_dim).astype(np.float64), fmt)


# ---------------------------------------------------------------- scoring
def head_dots(qc, qs, kc, ks, pos) -> np.ndarray:
    """Per-head float32 dots D [npos, H] of one quantised query ([H, d/2], [H, d/32])
    against key rows ``pos`` of a cache (kc [N, d/2], ks [N, d/32])."""
    qc = np.ascontiguousarray(qc, np.uint8); qs = np.ascontiguousarray(qs, np.uint8)
    kc = np.ascontiguousarray(kc, np.uint8); ks = np.ascontiguousarray(ks, np.uint8)
    pos = np.ascontiguousarray(pos, np.int64)
    H, d = qc.shape[0], qc.shape[1] * 2
    out = np.empty((pos.size, H), np.float32)
    _L().orc_head_dots(H, d, _p(qc), _p(qs), _p(kc), _p(ks), _p(pos), pos.size, _p(out))
    return out


def index_scores(qc, qs, w, kc, ks, pos, order: str = "chain") -> np.ndarray:
    """float32 indexer scores of one quantised query at key rows ``pos``, the head terms
    summed in the library's order: "chain" (one fma chain in head order) or "split8" (the
    prefill-chunk kernel's eight partial chains over heads h = j mod 8, then
    ((p0 + p1) + (p2 + p3)) + ((p4 + p5) + (p6 + p7)))."""
    qc = np.ascontiguousarray(qc, np.uint8); qs = np.ascontiguousarray(qs, np.uint8)
    kc = np.ascontiguousarray(kc, np.uint8); ks = np.ascontiguousarray(ks, np.uint8)
    w = np.ascontiguousarray(w, np.float32)
    pos = np.ascontiguousarray(pos, np.int64)
    H, d = qc.shape[0], qc.shape[1] * 2
    out = np.empty(pos.size, np.float32)
    _L().orc_index_scores(H, d, _p(qc), _p(qs), _p(w), _p(kc), _p(ks), _p(pos), pos.size,
                          _p(out), {"chain": 0, "split8": 1}[order])
    return out


def exact_format():
    """(limbs, e0): an exact score is a two's-complement integer of ``limbs`` 32-bit
    limbs (least significant first) in units of 2^e0."""
    lib = _L()
    return int(lib.orc_exact_limbs()), int(lib.orc_exact_e0())


def index_scores_exact(qc, qs, w, kc, ks, pos) -> np.ndarray:
    """Exact indexer scores of one quantised query at key rows ``pos``:
    s = sum_h w_h * max(0, q_hat_h . k_hat), nothing rounded.  Returns uint32 limbs
    [npos, limbs] (see ``exact_format``)."""
    qc = np.ascontiguousarray(qc, np.uint8); qs = np.ascontiguousarray(qs, np.uint8)
    kc = np.ascontiguousarray(kc, np.uint8); ks = np.ascontiguousarray(ks, np.uint8)
    w = np.ascontiguousarray(w, np.float32)
    pos = np.ascontiguousarray(pos, np.int64)
    H, d = qc.shape[0], qc.shape[1] * 2
    L, _ = exact_format()
    out = np.empty((pos.size, L), np.uint32)
    _L().orc_index_scores_exact(H, d, _p(qc), _p(qs), _p(w), _p(kc), _p(ks), _p(pos), pos.size,
                                _p(out))
    return out


def exact_int(limbs_row) -> int:
    """The integer S of one exact score (value = S * 2^e0)."""
    v = int.from_bytes(np.ascontiguousarray(limbs_row, np.uint32).astype("<u4").tobytes(), "little",
                       signed=True)
    return v


def exact_fraction(limbs_row):
    """One exact score as a fractions.Fraction."""
    from fractions import Fraction
    _, e0 = exact_format()
    return Fraction(exact_int(limbs_row)) * Fraction(2) ** e0


def _exact_desc_keys(limbs: np.ndarray):
    """numpy.lexsort keys (least significant first) that sort exact scores in
    descending order: limbs complemented, the top limb's sign bit flipped first so
    that unsigned limb order is numeric order.  Limbs equal in every row are left out
    (they cannot change the order)."""
    lim = np.array(limbs, dtype=np.uint32, copy=True)
    if lim.shape[0] == 0:
        return []
    lim[:, -1] ^= np.uint32(0x80000000)
    keys = []
    for j in range(lim.shape[1]):
        col = lim[:, j]
        if np.all(col == col[0]):
            continue
        keys.append(~col)
    return keys


def order_exact_desc(limbs: np.ndarray, ids: np.ndarray) -> np.ndarray:
    """Permutation sorting by (exact score descending, id ascending)."""
    return np.lexsort(tuple([np.asarray(ids)] + _exact_desc_keys(limbs)))


def topk_exact(limbs: np.ndarray, pos: np.ndarray, k: int) -> np.ndarray:
    """The k best positions by (exact score descending, position ascending); returned
    ascending, -1 padded."""
    out = np.full(k, -1, np.int32)
    if pos.size:
        sel = np.sort(np.asarray(pos)[order_exact_desc(limbs, pos)[:k]])
        out[: sel.size] = sel
    return out


def block_max_exact(limbs: np.ndarray, n_vis: int, block: int) -> np.ndarray:
    """Exact block scores: for block b the largest exact score among its visible
    positions 8b .. (positions 0..n_vis-1, limbs [n_vis, L]).  Returns limbs [nblk, L]."""
    nblk = (n_vis + block - 1) // block
    if nblk == 0:
        return np.zeros((0, limbs.shape[1]), np.uint32)
    p = np.arange(n_vis)
    blk = p // block
    # within each block, its best position first: sort by (block, exact desc)
    order = np.lexsort(tuple([p] + _exact_desc_keys(limbs[:n_vis]) + [blk]))
    first = np.ones(n_vis, bool)
    first[1:] = blk[order][1:] != blk[order][:-1]
    return limbs[order[first]]


def block_candidates_exact(limbs: np.ndarray, n_vis: int, block: int, nb: int) -> np.ndarray:
    """Top-nb blocks by (exact block score descending, block id ascending); returned
    ascending, -1 padded."""
    out = np.full(nb, -1, np.int32)
    bl = block_max_exact(limbs, n_vis, block)
    if bl.shape[0]:
        ids = np.arange(bl.shape[0])
        sel = np.sort(ids[order_exact_desc(bl, ids)[:nb]])
        out[: sel.size] = sel
    return out


def n_visible(q_pos: int, ratio_m: int, n_keys: int) -> int:
    """Entries a query at token position q_pos can see: entry j covers tokens
    [j*m, j*m + m - 1] with no overlap (report §2.3), and only complete entries are
    visible: (j + 1) * m - 1 <= q_pos."""
    return int(min(n_keys, max(0, (q_pos + 1) // ratio_m)))


# ---------------------------------------------------------------- selection
def _order_desc(scores: np.ndarray, pos: np.ndarray) -> np.ndarray:
    """Permutation sorting by (score descending, position ascending).

    Floats compare by value (-0 == +0); a NaN score ranks below every number."""
    s = scores.astype(np.float64)
    key = np.where(np.isnan(s), np.inf, -s)
    return np.lexsort((pos, key))


def topk(scores: np.ndarray, pos: np.ndarray, k: int) -> np.ndarray:
    """The k best (score, position) pairs; positions returned ascending, -1 padded."""
    out = np.full(k, -1, np.int32)
    if pos.size:
        sel = pos[_order_desc(scores, pos)[:k]]
        sel = np.sort(sel)
        out[: sel.size] = sel
    return out


def block_candidates(scores: np.ndarray, n_vis: int, block: int, nb: int) -> np.ndarray:
    """Top-nb blocks of ``block`` positions by max visible position score.

    ``scores`` holds the scores of positions 0..n_vis-1; a partial last block uses its
    visible positions only.  Block ids returned ascending, -1 padded."""
    out = np.full(nb, -1, np.int32)
    nblk = (n_vis + block - 1) // block
    if nblk == 0:
        return out
    pad = np.full(nblk * block, -np.inf, np.float64)
    s = scores[:n_vis].astype(np.float64)
    pad[:n_vis] = np.where(np.isnan(s), -np.inf, s)
    bscore = pad.reshape(nblk, block).max(axis=1)
    # a block whose visible scores are all NaN ranks lowest, like a NaN position
    allnan = np.zeros(nblk * block, bool)
    allnan[:n_vis] = np.isnan(s)
    allnan[n_vis:] = True
    bscore = np.where(allnan.reshape(nblk, block).all(axis=1), np.nan, bscore)
    sel = np.arange(nblk)[_order_desc(bscore.astype(np.float32), np.arange(nblk))[:nb]]
    sel = np.sort(sel)
    out[: sel.size] = sel
    return out


def pool_positions(block_ids: np.ndarray, block: int, n_vis: int) -> np.ndarray:
    """Positions covered by the pool's blocks, restricted to the visible range."""
    b = block_ids[block_ids >= 0].astype(np.int64)
    p = (b[:, None] * block + np.arange(block)[None, :]).reshape(-1)
    return np.sort(p[p < n_vis])


# ---------------------------------------------------------------- layer flows
def quant_query(q_f32: np.ndarray):
    """Indexer q [H, d] (exact bf16 values) -> MXFP4 (codes [H, d/2], scales [H, d/32])."""
    return quant_mxfp4(q_f32)


def full_indexer(q_f32, w, kc, ks, q_pos, ratio_m, k=512, block=8, nb=2048,
                 want_blocks=False, want_f32=True):
    """Full-mode indexer for one query: exact score of every visible position, Top-K,
    and (for the decoder's first Full layer) the block pool.  Returns (idx, blocks,
    float32 scores or None)."""
    qc, qs = quant_query(q_f32)
    nvis = n_visible(q_pos, ratio_m, kc.shape[0])
    pos = np.arange(nvis, dtype=np.int64)
    ex = index_scores_exact(qc, qs, w, kc, ks, pos)
    idx = topk_exact(ex, pos, k)
    blocks = block_candidates_exact(ex, nvis, block, nb) if want_blocks else None
    s = index_scores(qc, qs, w, kc, ks, pos) if want_f32 else None
    return idx, blocks, s


def reindex_indexer(q_f32, w, kc, ks, q_pos, ratio_m, pool_blocks, k=512, block=8,
                    want_f32=True):
    """Reindex-mode indexer for one query: only positions of the pool compete, ranked
    by their exact scores.  Returns (idx, float32 scores or None, positions)."""
    qc, qs = quant_query(q_f32)
    nvis = n_visible(q_pos, ratio_m, kc.shape[0])
    pos = pool_positions(np.asarray(pool_blocks), block, nvis)
    ex = index_scores_exact(qc, qs, w, kc, ks, pos)
    s = index_scores(qc, qs, w, kc, ks, pos) if want_f32 else None
    return topk_exact(ex, pos, k), s, pos


def swa_keys_range(q_pos: int, swa_pos0: int, n_slots: int, window: int, swa_start: int):
    """Slots of an SWA buffer (slot j holds token swa_pos0 + j) that a query at q_pos
    attends: tokens in [max(s, i - W + 1, 0), i] (report §3.2.2)."""
    lo = max(swa_start, q_pos - window + 1, 0)
    j0 = max(lo - swa_pos0, 0)
    j1 = min(q_pos - swa_pos0, n_slots - 1)
    return j0, j1          # inclusive; empty when j1 < j0


def attention_rows(q_rows, key_lists, sm_scale, d_v):
    """fp64 attention: q_rows [R, H, d_qk] float64, key_lists: list of [n_j, d_qk]
    float64 arrays -> (out [R, H, d_v], lse [R, H])."""
    q_rows = np.ascontiguousarray(q_rows, np.float64)
    R, H, dqk = q_rows.shape
    off = np.zeros(R + 1, np.int64)
    for r, kl in enumerate(key_lists):
        off[r + 1] = off[r] + kl.shape[0]
    keys = (np.concatenate(key_lists, axis=0) if off[-1] > 0
            else np.zeros((1, dqk), np.float64))
    keys = np.ascontiguousarray(keys, np.float64)
    out = np.empty((R, H, d_v), np.float64)
    lse = np.empty((R, H), np.float64)
    _L().orc_attention(R, H, dqk, d_v, _p(q_rows), _p(off), _p(keys), float(sm_scale),
                       _p(out), _p(lse))
    return out, lse


def gather_keys(idx, kv_codes, kv_scales, swa_f64, q_pos, swa_pos0, window, swa_start):
    """Key list of one query: dequantised main-KV rows for idx >= 0 (in idx order,
    duplicates kept, out-of-range indices dropped), then its SWA slots in order.  The
    main KV may be MXFP4 or E2M1 + E4M3/16 (told apart by the scale count)."""
    n = kv_codes.shape[0]
    sel = [int(i) for i in np.asarray(idx).reshape(-1) if 0 <= int(i) < n]
    parts = []
    if sel:
        parts.append(dequant_main_kv(kv_codes[sel], kv_scales[sel]))
    if swa_f64 is not None:
        j0, j1 = swa_keys_range(q_pos, swa_pos0, swa_f64.shape[0], window, swa_start)
        if j1 >= j0:
            parts.append(swa_f64[j0:j1 + 1])
    d = kv_codes.shape[1] * 2
    return np.concatenate(parts, 0) if parts else np.zeros((0, d), np.float64)
