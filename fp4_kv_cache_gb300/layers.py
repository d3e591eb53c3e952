"""CSA2 layer flows: Full, Reindex and Reuse (pure data flow over the C entry points).

DeepSeek-V4.1-Flash report (aipaper.jasonlin.tech) §2.3.1: each CSA2 layer is statically
Full, Reindex or Reuse; every mode computes its own query and SWA KV and attends them with
the selected main-KV entries.  Full runs the indexer over all visible entries; Reindex
re-scores the shared indexer K with the layer's own indexer query (inside the block pool,
§2.3.2); Reuse takes the latest Top-K indices and only attends.  Sharing a cache across
layers is passing the same tensors.

Each function enqueues its kernels on the current (or given) CUDA stream and returns
device tensors; nothing here computes on the host.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from . import csa2


@dataclass
class Cache:
    """One source layer's shared global cache: the main KV (MXFP4, or the report's E2M1 +
    E4M3/16 -- told apart by the width of kv_scales) and the MXFP4 indexer K."""
    kv_codes: torch.Tensor      # uint8 [B, N, d_qk/2]
    kv_scales: torch.Tensor     # uint8 [B, N, d_qk/32] (MXFP4) or [B, N, d_qk/16] (E2M1 + E4M3/16)
    k_codes: torch.Tensor       # uint8 [B, N, d_i/2]
    k_scales: torch.Tensor      # uint8 [B, N, d_i/32]
    ratio_m: int = 1


@dataclass
class LayerInput:
    """What a layer computes for itself in every mode: its query and SWA KV."""
    q_attn: torch.Tensor                    # bf16 [B, T, H, d_qk]
    swa: Optional[torch.Tensor]             # bf16 [B, S, d_qk]
    swa_pos0: Optional[torch.Tensor]        # int32 [B]
    q_pos: torch.Tensor                     # int32 [B, T]
    q_idx: Optional[torch.Tensor] = None    # bf16 [B, T, H_i, d_i] (Full / Reindex)
    w_idx: Optional[torch.Tensor] = None    # f32 [B, T, H_i]       (Full / Reindex)
    swa_start: Optional[torch.Tensor] = None


@dataclass
class LayerOutput:
    out: torch.Tensor                       # bf16 [B, T, H, d_v]
    lse: Optional[torch.Tensor]
    idx: torch.Tensor                       # int32 [B, T, K] selection used
    pool_blocks: Optional[torch.Tensor] = None
    scores: Optional[torch.Tensor] = None


def _attend(cache: Cache, x: LayerInput, idx, window, d_v, sm_scale, d_status, stream):
    return csa2.sparse_attn(x.q_attn, cache.kv_codes, cache.kv_scales, idx, x.swa, x.swa_pos0,
                            x.q_pos, x.swa_start, window, sm_scale, d_v, True, d_status, stream)


def full_layer(cache: Cache, x: LayerInput, k: int = 512, window: int = 128, d_v: int = 512,
               build_pool: bool = False, n_blocks: int = 2048, block: int = 8,
               sm_scale: Optional[float] = None, d_status=None, stream=None) -> LayerOutput:
    """Full mode: score every visible entry, Top-K by the exact score (and, for the
    decoder's first Full layer, the block pool of report §2.3.2), then attend."""
    n = cache.k_codes.shape[1]
    gmax = torch.empty(x.q_idx.shape[:2] + ((n + 31) // 32,), dtype=torch.int32, device=x.q_idx.device)
    scores, row_len, args = csa2.index_score(x.q_idx, x.w_idx, cache.k_codes, cache.k_scales, x.q_pos,
                                             cache.ratio_m, None, block, d_status, stream, group_max=gmax,
                                             want_args=True)
    idx = csa2.topk(scores, k, row_len, None, block, False, d_status, stream, group_max=gmax,
                    exact=args)
    pool = csa2.block_candidates(scores, n_blocks, row_len, block, d_status, stream, exact=args) \
        if build_pool else None
    out, lse = _attend(cache, x, idx, window, d_v, sm_scale, d_status, stream)
    return LayerOutput(out, lse, idx, pool, scores)


def reindex_layer(cache: Cache, x: LayerInput, pool_blocks: torch.Tensor, k: int = 512,
                  window: int = 128, d_v: int = 512, block: int = 8,
                  sm_scale: Optional[float] = None, d_status=None, stream=None) -> LayerOutput:
    """Reindex mode: the layer's own indexer query re-scores the shared indexer K, but only
    at the positions of the pool; its own Top-K inside the pool; then attend."""
    n = pool_blocks.shape[-1] * block
    gmax = torch.empty(x.q_idx.shape[:2] + ((n + 31) // 32,), dtype=torch.int32, device=x.q_idx.device)
    scores, row_len, args = csa2.index_score(x.q_idx, x.w_idx, cache.k_codes, cache.k_scales, x.q_pos,
                                             cache.ratio_m, pool_blocks, block, d_status, stream,
                                             group_max=gmax, want_args=True)
    idx = csa2.topk(scores, k, row_len, pool_blocks, block, False, d_status, stream, group_max=gmax,
                    exact=args)
    out, lse = _attend(cache, x, idx, window, d_v, sm_scale, d_status, stream)
    return LayerOutput(out, lse, idx, pool_blocks, scores)


def reuse_layer(cache: Cache, x: LayerInput, idx: torch.Tensor, window: int = 128,
                d_v: int = 512, sm_scale: Optional[float] = None, d_status=None,
                stream=None) -> LayerOutput:
    """Reuse mode: attention over the latest Top-K indices; no indexer work."""
    out, lse = _attend(cache, x, idx, window, d_v, sm_scale, d_status, stream)
    return LayerOutput(out, lse, idx)


# The report's schedule (§4.2.1; the review page's zero-based table): layers 0-1 SWA only;
# encoder layers 2-19 at ratio 2 in groups of Full + 5 Reuse; decoder layers 20-39 at
# ratio 1, Full at 20, Reindex at 24/28/32/36, Reuse elsewhere.
def layer_mode(layer: int) -> str:
    if layer < 2:
        return "swa"
    if layer < 20:
        return "full" if (layer - 2) % 6 == 0 else "reuse"
    if layer == 20:
        return "full"
    return "reindex" if (layer - 20) % 4 == 0 else "reuse"
