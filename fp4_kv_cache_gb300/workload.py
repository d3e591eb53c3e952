"""Device-resident inputs of a CSA2 workload, built from the seeded generator.

Float inputs are drawn on the host (``synth``), copied to the device one sequence at a
time and quantised there by csa2_quant_fp4, so a 1M-position cache never needs a
full float copy on the host.  Used by the benchmark and the GPU tests.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Dict, Optional

import numpy as np
import torch

from . import csa2, synth


def bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


@dataclass
class DeviceWorkload:
    w: synth.Workload
    rows: list
    t: Dict[str, torch.Tensor] = field(default_factory=dict)
    sm_scale: float = 0.0

    def __getitem__(self, k):
        return self.t[k]


def build(w: synth.Workload, rows=None, device="cuda:0", kv: bool = True, kidx: bool = True,
          d_status: Optional[torch.Tensor] = None, kv_fmt: int = csa2.FMT_MXFP4,
          also_nvfp4: bool = False, swa_fp8: bool = False) -> DeviceWorkload:
    """kv_fmt: main-KV cache format (MXFP4, or E2M1 + E4M3/16 as the report stores it);
    the indexer keys are MXFP4 either way.  also_nvfp4: quantise the same main-KV rows a
    second time into E2M1 + E4M3/16 ("kv_codes_nv", "kv_scales_nv").  swa_fp8: also the SWA
    rows in MXFP8 ("swa8" codes, "swa8_scales"), the report's FP8 SWA cache."""
    rows = list(range(w.batch)) if rows is None else list(rows)
    B = len(rows)
    dev = torch.device(device)
    out = DeviceWorkload(w, rows)
    qi, ww, qa = synth.gen_queries(w, rows)
    out.t["q_idx"] = bf16_tensor(qi, dev)
    out.t["w_idx"] = torch.from_numpy(ww).to(dev)
    out.t["q_attn"] = bf16_tensor(qa, dev)
    out.t["q_pos"] = torch.from_numpy(synth.q_positions(w)[: B]).to(dev)
    n_slots, pos0 = synth.swa_layout(w)
    out.t["swa_pos0"] = torch.full((B,), pos0, dtype=torch.int32, device=dev)
    N = w.n_keys
    if kidx:
        kc = torch.empty((B, N, w.idx_dim // 2), dtype=torch.uint8, device=dev)
        ks = torch.empty((B, N, w.idx_dim // 32), dtype=torch.uint8, device=dev)
        for i, b in enumerate(rows):
            x = bf16_tensor(synth.gen_index_keys(w, b, qi[i], ww[i]), dev)
            csa2.csa2_quant_fp4(x, kc[i], ks[i], d_status)
            del x
        out.t["k_codes"], out.t["k_scales"] = kc, ks
    if kv:
        vc = torch.empty((B, N, w.d_qk // 2), dtype=torch.uint8, device=dev)
        vs = torch.empty((B, N, w.d_qk // csa2.FMT_BLOCK[kv_fmt]), dtype=torch.uint8, device=dev)
        swa = torch.empty((B, n_slots, w.d_qk), dtype=torch.bfloat16, device=dev)
        if also_nvfp4:
            nvc = torch.empty((B, N, w.d_qk // 2), dtype=torch.uint8, device=dev)
            nvs = torch.empty((B, N, w.d_qk // 16), dtype=torch.uint8, device=dev)
            out.t["kv_codes_nv"], out.t["kv_scales_nv"] = nvc, nvs
        for i, b in enumerate(rows):
            x = bf16_tensor(synth.gen_main_kv(w, b), dev)
            csa2.csa2_quant_fp4(x, vc[i], vs[i], d_status, fmt=kv_fmt)
            if also_nvfp4:
                csa2.csa2_quant_fp4(x, nvc[i], nvs[i], d_status, fmt=csa2.FMT_NVFP4_E4M3_16)
            del x
            swa[i] = bf16_tensor(synth.gen_swa(w, b), dev)
        out.t["kv_codes"], out.t["kv_scales"], out.t["swa"] = vc, vs, swa
        if swa_fp8:
            out.t["swa8"], out.t["swa8_scales"] = csa2.quant_fp8(swa, d_status)
    if w.pool_blocks:
        out.t["pool"] = torch.from_numpy(np.stack([synth.gen_pool_blocks(w, b) for b in rows])).to(dev)
    if w.reuse_idx:
        out.t["reuse_idx"] = torch.from_numpy(np.stack([synth.gen_reuse_idx(w, b) for b in rows])).to(dev)
    if w.swa_start:
        out.t["swa_start"] = torch.full((B,), w.swa_start, dtype=torch.int32, device=dev)
    out.sm_scale = 1.0 / math.sqrt(w.d_qk)
    torch.cuda.synchronize(dev)
    return out
