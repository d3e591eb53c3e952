"""Seeded synthetic inputs for the CSA2 decode/prefill path.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no FP4 coding, no scoring, no selection, no attention).
Both the CUDA path and the CPU oracle take their inputs from here, and each
side quantises the float inputs with its own codec.

Shapes follow the workloads the DeepSeek-V4.1-Flash report describes for CSA2
(report §2.3, §2.3.2 and §4.2.1 on aipaper.jasonlin.tech): 32 indexer heads of
dim 128, Top-512, a 128-token SWA window, 64 attention heads over a shared
latent, blocks of 8 positions and at most 2,048 blocks.  Every array is drawn
per batch row from ``numpy.random.default_rng([seed, stream, row])`` so a
subset of rows can be regenerated on its own, identically on x86 and Arm.

bf16 tensors are returned as ``uint16`` bit patterns (round-to-nearest-even
from the float32 draw); ``bf16_to_f32`` widens them exactly.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

# stream ids: one independent random stream per kind of tensor
_S_QIDX, _S_W, _S_KIDX, _S_KV, _S_QATTN, _S_SWA, _S_PLANT, _S_IDX, _S_POOL, _S_PAL = range(10)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern, round to nearest even (inputs are finite)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & 1) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit pattern -> float32 (exact)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclass(frozen=True)
class Workload:
    """One CSA2 workload.  All sizes are per call of the path."""
    name: str
    batch: int                 # B: independent sequences
    n_q: int                   # T: query tokens per sequence
    n_keys: int                # N: global (main KV / indexer K) entries per sequence
    ratio_m: int               # compression ratio m: entry j covers tokens [j*m, j*m+m-1]
    q_pos0: int                # absolute token position of the first query
    idx_heads: int             # H_i indexer heads
    idx_dim: int               # d_i indexer head dim
    heads: int                 # H attention heads
    d_qk: int                  # latent dim used for q.k
    d_v: int                   # leading latent dims used as V
    topk: int = 512
    window: int = 128          # SWA window W
    block: int = 8             # positions per block of the hierarchical pool
    n_blocks: int = 2048       # blocks kept in the pool
    seed: int = 0
    plant_frac: float = 0.0    # fraction of positions given a planted signal
    plant_sigma: float = 3.0
    palette: int = 0           # >0: K rows drawn from this many distinct rows (ties)
    palette_zero: int = 0      # how many palette rows are all-zero (score exactly 0)
    pool_blocks: int = 0       # >0: a given Reindex pool of this many blocks
    reuse_idx: bool = False    # draw given Top-K indices for a Reuse layer
    swa_start: int = 0         # replay start s of the SWA window
    extra: dict = field(default_factory=dict)

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads (sizes as the report's configuration and the scope table state).
WORKLOADS = {
    # tiny Full decode: batch 1, 1 query, 4,096 positions, latent 128, 16 heads, indexer 4x64
    "tiny_full_decode": Workload("tiny_full_decode", batch=1, n_q=1, n_keys=4096, ratio_m=1,
                                 q_pos0=4095, idx_heads=4, idx_dim=64, heads=16, d_qk=128,
                                 d_v=128, seed=0),
    # Full decode at 64K context, 1% planted positions
    "full_decode_64k": Workload("full_decode_64k", batch=32, n_q=1, n_keys=65536, ratio_m=1,
                                q_pos0=65535, idx_heads=32, idx_dim=128, heads=64, d_qk=576,
                                d_v=512, seed=1, plant_frac=0.01),
    # Reuse + Reindex decode at 128K context (production dims)
    "reuse_reindex_decode_128k": Workload("reuse_reindex_decode_128k", batch=64, n_q=1,
                                          n_keys=131072, ratio_m=1, q_pos0=131071,
                                          idx_heads=32, idx_dim=128, heads=64, d_qk=576,
                                          d_v=512, seed=2, pool_blocks=2048, reuse_idx=True),
    # decoder hierarchical indexer (first Full layer of the decoder) at 1M context, with ties
    "hier_indexer_1m": Workload("hier_indexer_1m", batch=4, n_q=1, n_keys=1048576, ratio_m=1,
                                q_pos0=1048575, idx_heads=32, idx_dim=128, heads=64, d_qk=576,
                                d_v=512, seed=3, palette=1024, palette_zero=16),
    # encoder Full layer prefill chunk at ratio 2: 4,096 queries after a 131,072-token prefix
    "prefill_chunk_m2": Workload("prefill_chunk_m2", batch=1, n_q=4096, n_keys=67584, ratio_m=2,
                                 q_pos0=131072, idx_heads=32, idx_dim=128, heads=64, d_qk=576,
                                 d_v=512, seed=4),
    # decoder SWA bounded replay (report §3.2.2): the last 128 tokens of a 131,072-token
    # context replayed from s = 131,072 through attention; query i attends its given
    # Top-512 entries and the SWA keys [max(s, i - W + 1), i] (1 to 128 of them)
    "swa_replay_prefill": Workload("swa_replay_prefill", batch=8, n_q=128, n_keys=131072, ratio_m=1,
                                   q_pos0=131072, idx_heads=32, idx_dim=128, heads=64, d_qk=576,
                                   d_v=512, seed=5, reuse_idx=True, swa_start=131072),
}


def _rng(w: Workload, stream: int, row: int) -> np.random.Generator:
    return np.random.default_rng([w.seed, stream, row])


def q_positions(w: Workload) -> np.ndarray:
    """Absolute token position of every query: [B, T] int32."""
    t = np.arange(w.n_q, dtype=np.int64) + w.q_pos0
    return np.broadcast_to(t, (w.batch, w.n_q)).astype(np.int32).copy()


def swa_layout(w: Workload):
    """SWA buffer layout: slots, and the absolute token position of slot 0.

    The buffer holds tokens [q_pos0 - W + 1, q_pos_last] (W + T - 1 slots), so each
    query finds its whole window in it."""
    n_slots = w.window + w.n_q - 1
    pos0 = w.q_pos0 - w.window + 1
    return n_slots, pos0


def gen_queries(w: Workload, rows=None):
    """Indexer q (bf16 bits [B,T,Hi,di]), head weights w (f32 U(0,1) [B,T,Hi]),
    attention q (bf16 bits [B,T,H,d_qk])."""
    rows = range(w.batch) if rows is None else rows
    qi, ww, qa = [], [], []
    for b in rows:
        qi.append(f32_to_bf16_bits(_rng(w, _S_QIDX, b).standard_normal(
            (w.n_q, w.idx_heads, w.idx_dim), dtype=np.float32)))
        ww.append(_rng(w, _S_W, b).random((w.n_q, w.idx_heads), dtype=np.float32))
        qa.append(f32_to_bf16_bits(_rng(w, _S_QATTN, b).standard_normal(
            (w.n_q, w.heads, w.d_qk), dtype=np.float32)))
    return np.stack(qi), np.stack(ww), np.stack(qa)


def gen_index_keys(w: Workload, b: int, q_idx_bits: Optional[np.ndarray] = None,
                   head_w: Optional[np.ndarray] = None) -> np.ndarray:
    """Float indexer-K rows of sequence b as bf16 bits [N, di].

    N(0,1) by default.  With ``palette`` > 0 each row is one of ``palette`` distinct
    rows (the first ``palette_zero`` of them all zero), so equal scores repeat.  With
    ``plant_frac`` > 0 that fraction of rows gets ``plant_sigma`` added along the unit
    vector of sum_h w_h q_h of the sequence's first query (a planted signal)."""
    r = _rng(w, _S_KIDX, b)
    if w.palette > 0:
        pal = _rng(w, _S_PAL, 0).standard_normal((w.palette, w.idx_dim), dtype=np.float32)
        pal[: w.palette_zero] = 0.0
        which = r.integers(0, w.palette, size=w.n_keys)
        k = pal[which]
    else:
        k = r.standard_normal((w.n_keys, w.idx_dim), dtype=np.float32)
    if w.plant_frac > 0:
        assert q_idx_bits is not None and head_w is not None
        q = bf16_to_f32(q_idx_bits[0]).astype(np.float64)          # [Hi, di] of query 0
        g = (head_w[0].astype(np.float64)[:, None] * q).sum(0)
        g /= np.linalg.norm(g)
        n_plant = int(round(w.plant_frac * w.n_keys))
        pr = _rng(w, _S_PLANT, b)
        pos = pr.choice(w.n_keys, size=n_plant, replace=False)
        k[pos] += (w.plant_sigma * g).astype(np.float32)
    return f32_to_bf16_bits(k)


def gen_main_kv(w: Workload, b: int) -> np.ndarray:
    """Float main-KV latent rows of sequence b as bf16 bits [N, d_qk], N(0,1)."""
    return f32_to_bf16_bits(_rng(w, _S_KV, b).standard_normal((w.n_keys, w.d_qk),
                                                              dtype=np.float32))


def gen_swa(w: Workload, b: int) -> np.ndarray:
    """SWA KV of sequence b as bf16 bits [W + T - 1, d_qk], N(0,1)."""
    n_slots, _ = swa_layout(w)
    return f32_to_bf16_bits(_rng(w, _S_SWA, b).standard_normal((n_slots, w.d_qk),
                                                               dtype=np.float32))


def gen_reuse_idx(w: Workload, b: int) -> np.ndarray:
    """Given Top-K indices for a Reuse layer: [T, K] int32, uniform, unique, ascending."""
    r = _rng(w, _S_IDX, b)
    out = np.empty((w.n_q, w.topk), dtype=np.int32)
    for t in range(w.n_q):
        out[t] = np.sort(r.choice(w.n_keys, size=w.topk, replace=False))
    return out


def gen_pool_blocks(w: Workload, b: int) -> np.ndarray:
    """A given Reindex pool: [T, n_blocks] int32 block ids, unique, ascending."""
    r = _rng(w, _S_POOL, b)
    nb_all = (w.n_keys + w.block - 1) // w.block
    out = np.empty((w.n_q, w.n_blocks), dtype=np.int32)
    for t in range(w.n_q):
        out[t] = np.sort(r.choice(nb_all, size=w.n_blocks, replace=False))
    return out
