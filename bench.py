"""Benchmark of the CSA2 decode hot path on one GB300 (or N independent replicas).

Default workload: Full-mode decode layer, batch 32, 65,536 global positions per sequence,
indexer 32 heads x 128 (MXFP4 K), main KV 512 + 64 dims (MXFP4), 64 heads, Top-512,
SWA 128 (bf16).  One step = the whole path for one new token per sequence:
  csa2_rope_quant_fp4 (write the token's main-KV row, after RoPE on its 64 trailing channels,
                       and its indexer-K row into the caches: one launch)
  csa2_index_score (indexer query quantised inside; every visible position scored)
  csa2_topk        (Top-512, ascending)
  csa2_sparse_attn (gather + dequantise 512 entries, + 128 SWA keys, 64-head attention)
metric: decode tokens/s per layer (batch / step time); roofline of the dominant kernel
(the indexer scan) in achieved HBM GB/s.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--no-prefill]
Under torchrun each rank runs its own replica (the path has no exchange step).
Rank 0 also times the prefill indexer on an encoder chunk (4,096 queries after 65,536
entries at ratio 2) and the whole chunk (indexer, Top-512, attention), reported beside the
decode line as "prefill_indexer"; one decoder group (the Full layer's step, then 3 Reuse
layers attending its Top-K) as "decoder_group"; the step over the report's E2M1 +
E4M3/16 main-KV cache as "main_kv_e4m3_16"; and the indexer steps the decode step does not
exercise -- the Reindex layer's pool scoring at 128K and the decoder's hierarchical indexer
at 1M (scores, Top-512, Top-2,048 blocks) -- as "indexer_rows".  Every kernel's own roofline
is in "kernels_roofline".
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from fp4_kv_cache_gb300 import synth  # noqa: E402

METRIC = "CSA2 decode tokens/s per layer (Full mode, 64K ctx)"
WORKLOAD = "full_decode_64k"
L2_FLUSH_BYTES = 256 << 20


class L2Flush:
    """Evicts L2 between timed runs: writes one buffer larger than L2, then reads a second
    one, so the dirty lines the write leaves are written back before the timed region
    instead of competing with its reads.  Untimed."""

    def __init__(self, dev):
        import torch
        self.a = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.b = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def __call__(self):
        self.a.fill_(1)
        self.b.max()


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _kernel_bytes(w):
    """Algorithmic bytes of the indexer scan per launch: MXFP4 K codes + scales of every
    visible position (68 B at d_i = 128), the bf16 indexer query and the head weights.
    Score materialisation is overhead and not counted."""
    per_pos = w.idx_dim // 2 + w.idx_dim // 32
    return w.batch * w.n_keys * per_pos + w.batch * w.n_q * w.idx_heads * (w.idx_dim * 2 + 4)


def _step_bytes(w):
    """Algorithmic bytes of a whole step (what the method must move)."""
    kv_row = w.d_qk // 2 + w.d_qk // 32
    idx_bytes = _kernel_bytes(w)
    attn = w.batch * w.n_q * (w.topk * (kv_row + 4) + w.window * w.d_qk * 2
                              + w.heads * w.d_qk * 2 + w.heads * w.d_v * 2)
    # cache write: both bf16 rows in, their codes and scales out, and the RoPE table row
    # (64 cosines and sines) of the new token
    write = w.batch * (w.d_qk * 2 + kv_row + w.idx_dim * 2 + w.idx_dim // 2 + w.idx_dim // 32 + 64 * 4)
    return idx_bytes + attn + write


def _bf16_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        return float(json.load(open(p)).get("bf16_tflops", 1900.0))
    return 1900.0


def kernel_rooflines(w, per_kernel_ms, peak_gbs, bf16_tflops):
    """Per-call roofline of each kernel of the step: its algorithmic bytes per call (and,
    for attention, its MMA flops) over its event-timed duration.  Cache write: both bf16 rows
    in, codes and scales out, the RoPE table row; indexer: _kernel_bytes; Top-K: the group
    keys in and the indices out (the few surviving groups' scores it also reads depend on
    the data and are left out); attention: as in _step_bytes."""
    kv_row = w.d_qk // 2 + w.d_qk // 32
    rows = w.batch * w.n_q
    algo = {
        "cache_write": w.batch * (w.d_qk * 2 + kv_row + w.idx_dim * 2 + w.idx_dim // 2
                                  + w.idx_dim // 32 + 64 * 4),
        "index_score": _kernel_bytes(w),
        "topk": rows * (((w.n_keys + 31) // 32) * 4 + w.topk * 4),
        "sparse_attn": rows * (w.topk * (kv_row + 4) + w.window * w.d_qk * 2
                               + w.heads * w.d_qk * 2 + w.heads * w.d_v * 2),
    }
    out = {}
    for name, ms in per_kernel_ms.items():
        if name not in algo or not ms:
            continue
        gbs = algo[name] / (ms * 1e-3) / 1e9
        out[name] = {"bytes": algo[name], "ms": ms, "gbs": gbs, "frac_hbm": gbs / peak_gbs}
    if "sparse_attn" in out:
        flop = 2.0 * rows * w.heads * (w.topk + w.window) * (w.d_qk + w.d_v)
        tf = flop / (per_kernel_ms["sparse_attn"] * 1e-3) / 1e12
        out["sparse_attn"]["tflops"] = tf
        out["sparse_attn"]["frac_bf16"] = tf / bf16_tflops
    return out


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU baseline (oracle)
def oracle_sample(w, rows):
    """Run the CPU oracle over `rows` sequences of the workload: indexer over every
    visible position, Top-512, fp64 attention.  Returns (seconds, tokens)."""
    import oracle
    f32 = synth.bf16_to_f32
    qi, ww, qa = synth.gen_queries(w, rows)
    qpos = synth.q_positions(w)
    n_slots, pos0 = synth.swa_layout(w)
    inputs = []
    for i, b in enumerate(rows):   # inputs prepared outside the timed region
        kc, ks = oracle.quant_mxfp4(f32(synth.gen_index_keys(w, b, qi[i], ww[i])))
        kv = f32(synth.gen_main_kv(w, b))
        swa = f32(synth.gen_swa(w, b)).astype(np.float64)
        inputs.append((kc, ks, kv, swa))
    t0 = time.perf_counter()
    for i, b in enumerate(rows):
        kc, ks, kv, swa = inputs[i]
        for t in range(w.n_q):
            idx, _, _ = oracle.full_indexer(f32(qi[i, t]), ww[i, t], kc, ks, int(qpos[b, t]),
                                            w.ratio_m, w.topk)
            sel = idx[idx >= 0]
            vc, vs = oracle.quant_mxfp4(kv[sel])
            keys = oracle.gather_keys(np.arange(sel.size), vc, vs, swa, int(qpos[b, t]), pos0,
                                      w.window, 0)
            oracle.attention_rows(f32(qa[i, t])[None].astype(np.float64), [keys],
                                  1.0 / math.sqrt(w.d_qk), w.d_v)
    return time.perf_counter() - t0, len(rows) * w.n_q


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    w = synth.WORKLOADS[WORKLOAD]
    for _ in range(args.warmup):
        oracle_sample(w, [0])
    times = []
    for s in range(args.steps):
        dt, tok = oracle_sample(w, [s % w.batch])
        times.append(dt)
    tps = args.steps / sum(times)
    cores = oracle.num_threads()
    sample = "1 of 32 sequences per step: oracle indexer over 65,536 positions, Top-512, fp64 attention"
    line = {"impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000 * sum(times) / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": w.batch, "seq_len": w.n_keys,
                       "parallelism": "cpu-oracle (one sampled sequence per step)",
                       "topk": w.topk, "window": w.window, "indexer": f"{w.idx_heads}x{w.idx_dim}",
                       "heads": w.heads, "d_qk": w.d_qk, "d_v": w.d_v},
            "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": cores, "cpu_model": cpu_model(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------ ranks
def max_over_ranks(dist, values, device):
    """Each timing's maximum over the ranks (every rank runs its own replica of the step
    between barriers, so the job is as fast as its slowest rank); no reduction alone."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(units_per_rank, world, ms):
    """Whole-job units per second: `world` ranks each process units_per_rank in ms."""
    return units_per_rank * world / (ms * 1e-3)


# ------------------------------------------------------------------ GPU arm
def run_gpu(args):
    import torch
    from fp4_kv_cache_gb300 import csa2, workload

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    w = synth.WORKLOADS[WORKLOAD]
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    want_nv = rank == 0 and not args.no_nvfp4
    dw = workload.build(w, device=dev, d_status=st, also_nvfp4=want_nv, swa_fp8=want_nv)
    B, T = w.batch, w.n_q
    stream = torch.cuda.current_stream(dev)

    # the token being decoded: its main-KV / indexer-K rows (float) to write into the caches
    rng = np.random.default_rng([w.seed, 1000])
    new_kv = workload.bf16_tensor(synth.f32_to_bf16_bits(
        rng.standard_normal((B, w.d_qk), dtype=np.float32)), dev)
    new_k = workload.bf16_tensor(synth.f32_to_bf16_bits(
        rng.standard_normal((B, w.idx_dim), dtype=np.float32)), dev)
    last = w.n_keys - 1        # the decoded token's slot (the query sits at position N - 1)
    new_kvc, new_kvs = dw["kv_codes"][:, last], dw["kv_scales"][:, last]
    new_kc, new_ks = dw["k_codes"][:, last], dw["k_scales"][:, last]
    # preallocated outputs
    scores = torch.empty((B, T, w.n_keys), dtype=torch.float32, device=dev)
    row_len = torch.empty((B, T), dtype=torch.int32, device=dev)
    idx = torch.empty((B, T, w.topk), dtype=torch.int32, device=dev)
    out = torch.empty((B, T, w.heads, w.d_v), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, T, w.heads), dtype=torch.float32, device=dev)
    gmax = csa2.group_max_buffer(scores)     # per-32 group maxima: indexer -> Top-K
    iargs = csa2.make_index_args(dw["q_idx"], dw["w_idx"], dw["k_codes"], dw["k_scales"],
                                 dw["q_pos"], w.ratio_m, group_max=gmax)
    # only the decoded token's row (position N - 1) comes from the cache write just before the
    # indexer: the older positions stream while that write runs
    iargs.fresh_from = w.n_keys - 1
    aargs = csa2.make_attn_args(dw["q_attn"], dw["kv_codes"], dw["kv_scales"], idx, dw["swa"],
                                dw["swa_pos0"], dw["q_pos"], None, w.window, dw.sm_scale, w.d_v)
    lib = csa2.load()
    import ctypes
    ws_index = torch.zeros(max(1, lib.csa2_index_score_workspace_size(ctypes.byref(iargs))),
                           dtype=torch.uint8, device=dev)     # zero before first use
    ws_attn = torch.empty(max(1, lib.csa2_sparse_attn_workspace_size(ctypes.byref(aargs))),
                          dtype=torch.uint8, device=dev)
    ws_topk = torch.empty(max(1, lib.csa2_topk_workspace_size(B * T, w.n_keys, w.topk, ctypes.byref(iargs))),
                          dtype=torch.uint8, device=dev)
    flush = L2Flush(dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    # cache write (report §2.4.4: quantised after RoPE): the new main-KV row's 64 trailing
    # (RoPE) channels are rotated with a synthetic table (base 10,000) at the token's position,
    # then both rows are quantised -- one launch
    R = 64
    ang = np.arange(w.n_keys, dtype=np.float64)[:, None] * \
        10000.0 ** (-2.0 * np.arange(R // 2, dtype=np.float64) / R)[None, :]
    rope_tab = torch.from_numpy(np.concatenate([np.cos(ang), np.sin(ang)], 1).astype(np.float32)).to(dev)
    new_pos = torch.full((B,), last, dtype=torch.int32, device=dev)
    cache_rows = [(new_kv, new_kvc, new_kvs, R, new_pos, rope_tab, csa2.FMT_MXFP4),
                  (new_k, new_kc, new_ks, 0, None, None, csa2.FMT_MXFP4)]
    cache_jobs = csa2.rope_quant_jobs(cache_rows)
    # our kernels per step: the cache write (RoPE + quantisation of both rows), the indexer (it
    # also writes the per-32 group maxima), Top-K select, attention
    launches_per_step = 4

    def step(k_ev=None):
        # k_ev: events bracketing each call of the step.  The calls form one chain on one
        # stream, so each kernel can start its set-up while the one before it drains (a
        # side stream for the main-KV write would join the chain with an event and cut the
        # programmatic overlap of attention with Top-K).
        stream = torch.cuda.current_stream(dev)       # the capture stream while capturing
        if k_ev:
            k_ev[0].record(stream)
        # cache write: the new token's main-KV row (after RoPE) and indexer-K row, quantised
        # in place (one launch for both)
        csa2.csa2_rope_quant_fp4(cache_rows, st, jobs=cache_jobs)
        if k_ev:
            k_ev[1].record(stream)
        csa2.csa2_index_score(iargs, scores, row_len, st, workspace=ws_index)
        if k_ev:
            k_ev[2].record(stream)
        csa2.csa2_topk(scores, w.topk, idx, row_len, d_status=st, workspace=ws_topk, group_max=gmax,
                       exact=iargs)
        if k_ev:
            k_ev[3].record(stream)
        csa2.csa2_sparse_attn(aargs, out, lse, st, workspace=ws_attn)
        if k_ev:
            k_ev[4].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())}")

    # ---- the step as CUDA graphs (no host launch gaps): one plain, timed as the step (its
    #      kernels follow one another directly, so each may start its set-up while the
    #      previous one finishes), and one with timing events between the calls, replayed
    #      separately for the per-call breakdown
    names = ["cache_write", "index_score", "topk", "sparse_attn"]
    graph, graph_ev, g_ev = None, None, None
    try:
        g_ev = tuple(torch.cuda.Event(enable_timing=True, external=True) for _ in range(5))
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        graph_ev = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_ev):
            step(g_ev)
        for _ in range(args.warmup):
            graph.replay()
            graph_ev.replay()
        torch.cuda.synchronize(dev)
    except (TypeError, RuntimeError) as exc:          # no external events / capture: eager
        graph, graph_ev, g_ev = None, None, None
        torch.cuda.synchronize(dev)
        print(f"# CUDA graph capture unavailable ({exc}); timing eager launches", file=sys.stderr)
    stream = torch.cuda.current_stream(dev)

    def run_step(k_ev=None):
        if graph is not None:
            (graph_ev if k_ev is not None else graph).replay()
        else:
            step(k_ev)

    # ---- device-timed steps: inputs resident in HBM, L2 flushed between steps (untimed)
    ms_steps, per_k = [], {n: [] for n in names}
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clocks:
        for _ in range(args.steps):
            flush()
            e0, e1 = ev(), ev()
            e0.record(stream)
            run_step()
            e1.record(stream)
            e1.synchronize()
            ms_steps.append(e0.elapsed_time(e1))
        torch.cuda.synchronize(dev)
    for _ in range(args.steps):                       # per-call breakdown (not the step time)
        flush()
        k_ev = g_ev if graph is not None else tuple(ev() for _ in range(5))
        run_step(k_ev)
        k_ev[4].synchronize()
        for i, n in enumerate(names):
            per_k[n].append(k_ev[i].elapsed_time(k_ev[i + 1]))
    torch.cuda.synchronize(dev)
    per_kernel = {n: sum(v) / len(v) for n, v in per_k.items()}
    ms_step = sum(ms_steps) / len(ms_steps)
    ms_k = per_kernel["index_score"]

    # ---- end to end through the public API from pinned host buffers: every step uploads
    #      its inputs (the indexer query and head weights as one packed copy, the attention
    #      query on a second branch, since only the last call needs it), runs the four calls
    #      and downloads the attention output.  The whole sequence is one CUDA graph (copy
    #      nodes and kernels), so host launch gaps stay out of it; eager calls otherwise.
    n_qi = dw["q_idx"].numel() * 2
    n_w = dw["w_idx"].numel() * 4
    d_in = torch.empty(n_qi + n_w, dtype=torch.uint8, device=dev)      # packed inputs
    e_qi = d_in[:n_qi].view(torch.bfloat16).view(dw["q_idx"].shape)
    e_w = d_in[n_qi:].view(torch.float32).view(dw["w_idx"].shape)
    h_in = torch.empty(n_qi + n_w, dtype=torch.uint8).pin_memory()
    h_in[:n_qi].copy_(dw["q_idx"].cpu().view(torch.uint8).reshape(-1))
    h_in[n_qi:].copy_(dw["w_idx"].cpu().view(torch.uint8).reshape(-1))
    iargs_e2e = csa2.make_index_args(e_qi, e_w, dw["k_codes"], dw["k_scales"], dw["q_pos"], w.ratio_m,
                                     group_max=gmax)
    iargs_e2e.fresh_from = w.n_keys - 1
    h_qa = dw["q_attn"].cpu().pin_memory()
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = h_in.numel() + h_qa.numel() * 2
    d2h = h_out.numel() * 2
    copy_stream = torch.cuda.Stream(dev)

    def e2e_step_calls():
        cs = torch.cuda.current_stream(dev)
        fork = torch.cuda.Event()
        fork.record(cs)
        copy_stream.wait_event(fork)
        with torch.cuda.stream(copy_stream):
            dw["q_attn"].copy_(h_qa, non_blocking=True)
        qa_done = torch.cuda.Event()
        qa_done.record(copy_stream)
        d_in.copy_(h_in, non_blocking=True)
        csa2.csa2_rope_quant_fp4(cache_rows, st, jobs=cache_jobs)
        csa2.csa2_index_score(iargs_e2e, scores, row_len, st, workspace=ws_index)
        csa2.csa2_topk(scores, w.topk, idx, row_len, d_status=st, workspace=ws_topk, group_max=gmax,
                       exact=iargs_e2e)
        cs.wait_event(qa_done)
        csa2.csa2_sparse_attn(aargs, out, lse, st, workspace=ws_attn)
        h_out.copy_(out, non_blocking=True)

    g_e2e = None
    if graph is not None:
        try:
            for _ in range(2):
                e2e_step_calls()
            torch.cuda.synchronize(dev)
            g_e2e = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_e2e):
                e2e_step_calls()
        except (TypeError, RuntimeError) as exc:
            g_e2e = None
            torch.cuda.synchronize(dev)
            print(f"# end-to-end graph capture unavailable ({exc}); eager calls", file=sys.stderr)
    e2e_ms = []
    for it in range(args.steps + 2):
        flush()
        e0, e1 = ev(), ev()
        e0.record(stream)
        if g_e2e is not None:
            g_e2e.replay()
        else:
            e2e_step_calls()
        e1.record(stream)
        e1.synchronize()
        if it >= 2:
            e2e_ms.append(e0.elapsed_time(e1))
    e2e_step = sum(e2e_ms) / len(e2e_ms)
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())}")

    # ---- a decoder group (report §4.2.1 schedule: a Full layer then 3 Reuse layers that
    #      attend its Top-K over the same shared cache, each with its own query and SWA KV),
    #      one CUDA graph, L2 flushed between groups; rank 0 only
    group = None
    if rank == 0 and not args.no_group and graph is not None:
        gen = torch.Generator(device=dev)
        gen.manual_seed(w.seed * 7919 + 3)
        r_q = [torch.randn(dw["q_attn"].shape, generator=gen, device=dev).to(torch.bfloat16) for _ in range(3)]
        r_swa = [torch.randn(dw["swa"].shape, generator=gen, device=dev).to(torch.bfloat16) for _ in range(3)]
        r_out = [torch.empty_like(out) for _ in range(3)]
        r_lse = [torch.empty_like(lse) for _ in range(3)]
        r_args = [csa2.make_attn_args(r_q[l], dw["kv_codes"], dw["kv_scales"], idx, r_swa[l], dw["swa_pos0"],
                                      dw["q_pos"], None, w.window, dw.sm_scale, w.d_v) for l in range(3)]

        def group_step():
            step()
            for l in range(3):
                csa2.csa2_sparse_attn(r_args[l], r_out[l], r_lse[l], st, workspace=ws_attn)

        for _ in range(args.warmup):
            group_step()
        g_group = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_group):
            group_step()
        g_ms = []
        for it in range(args.steps + 2):
            flush()
            e0, e1 = ev(), ev()
            e0.record(stream)
            g_group.replay()
            e1.record(stream)
            e1.synchronize()
            if it >= 2:
                g_ms.append(e0.elapsed_time(e1))
        if int(st.item()) != 0:
            raise RuntimeError(f"device status {int(st.item())}")
        gt = sum(g_ms) / len(g_ms)
        group = {"layers": "Full + 3 Reuse (one decoder group, shared cache, Full layer's Top-K reused)",
                 "ms": gt, "tokens_per_s": B * T / (gt * 1e-3), "ms_per_layer": gt / 4,
                 "launches": launches_per_step + 3}

    # ---- the same step over the report's own main-KV format (E2M1 + E4M3 per 16, report
    #      §2.4.4): cache write (main-KV row after RoPE in that format, indexer-K row in
    #      MXFP4: one launch), indexer, Top-K, attention over the E4M3/16 cache; one CUDA
    #      graph, L2 flushed between steps; the attention call alone is timed for both formats
    nv = None
    pages_cfg = None
    fused_cfg = None
    if want_nv and graph is not None:
        nv_c, nv_s = dw["kv_codes_nv"], dw["kv_scales_nv"]
        aargs_nv = csa2.make_attn_args(dw["q_attn"], nv_c, nv_s, idx, dw["swa"], dw["swa_pos0"],
                                       dw["q_pos"], None, w.window, dw.sm_scale, w.d_v)
        ws_attn_nv = torch.empty(max(1, lib.csa2_sparse_attn_workspace_size(ctypes.byref(aargs_nv))),
                                 dtype=torch.uint8, device=dev)
        out_nv, lse_nv = torch.empty_like(out), torch.empty_like(lse)
        nv_rows = [(new_kv, nv_c[:, last], nv_s[:, last], R, new_pos, rope_tab, csa2.FMT_NVFP4_E4M3_16),
                   cache_rows[1]]
        nv_jobs = csa2.rope_quant_jobs(nv_rows)

        def step_nv():
            csa2.csa2_rope_quant_fp4(nv_rows, st, jobs=nv_jobs)
            csa2.csa2_index_score(iargs, scores, row_len, st, workspace=ws_index)
            csa2.csa2_topk(scores, w.topk, idx, row_len, d_status=st, workspace=ws_topk, group_max=gmax,
                       exact=iargs)
            csa2.csa2_sparse_attn(aargs_nv, out_nv, lse_nv, st, workspace=ws_attn_nv)

        # the pages' whole cache configuration: E2M1 + E4M3/16 main KV and the SWA window in
        # FP8 (MXFP8); the step also writes the new token's SWA row (its last slot)
        swa8, swa8_s = dw["swa8"], dw["swa8_scales"]
        aargs_pc = csa2.make_attn_args(dw["q_attn"], nv_c, nv_s, idx, swa8, dw["swa_pos0"], dw["q_pos"], None,
                                       w.window, dw.sm_scale, w.d_v, swa8_s)
        ws_attn_pc = torch.empty(max(1, lib.csa2_sparse_attn_workspace_size(ctypes.byref(aargs_pc))),
                                 dtype=torch.uint8, device=dev)
        out_pc, lse_pc = torch.empty_like(out), torch.empty_like(lse)
        slot = swa8.shape[1] - 1

        def step_pc():
            csa2.csa2_rope_quant_fp4(nv_rows, st, jobs=nv_jobs)
            csa2.csa2_quant_fp8(new_kv, swa8[:, slot], swa8_s[:, slot], st)
            csa2.csa2_index_score(iargs, scores, row_len, st, workspace=ws_index)
            csa2.csa2_topk(scores, w.topk, idx, row_len, d_status=st, workspace=ws_topk, group_max=gmax,
                           exact=iargs)
            csa2.csa2_sparse_attn(aargs_pc, out_pc, lse_pc, st, workspace=ws_attn_pc)

        for _ in range(args.warmup):
            step_nv()
            step_pc()
        g_pc = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_pc):
            step_pc()
        g_nv, g_a_nv, g_a_mx = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_nv):
            step_nv()
        with torch.cuda.graph(g_a_nv):
            csa2.csa2_sparse_attn(aargs_nv, out_nv, lse_nv, st, workspace=ws_attn_nv)
        with torch.cuda.graph(g_a_mx):
            csa2.csa2_sparse_attn(aargs, out, lse, st, workspace=ws_attn)

        def timed(g):
            ts = []
            for it in range(args.steps + 2):
                flush()
                e0, e1 = ev(), ev()
                e0.record(stream)
                g.replay()
                e1.record(stream)
                e1.synchronize()
                if it >= 2:
                    ts.append(e0.elapsed_time(e1))
            return sum(ts) / len(ts)

        t_nv, t_a_nv, t_a_mx, t_pc = timed(g_nv), timed(g_a_nv), timed(g_a_mx), timed(g_pc)
        if int(st.item()) != 0:
            raise RuntimeError(f"device status {int(st.item())}")
        pages_cfg = {"format": "main KV E2M1 + E4M3 per 16, indexer K MXFP4, SWA MXFP8 (report §2.4.4)",
                     "ms_per_step": t_pc, "tokens_per_s": B * T / (t_pc * 1e-3), "launches": 5,
                     "calls": "RoPE + cache write (main KV, indexer K), SWA row write (MXFP8), indexer, "
                              "exact Top-512, attention"}
        # the same step with the selection fused into the indexer (csa2_index_topk: its CTAs
        # keep their scores on chip and write candidate lists; no score matrix)
        iargs_f = csa2.make_index_args(dw["q_idx"], dw["w_idx"], dw["k_codes"], dw["k_scales"], dw["q_pos"],
                                       w.ratio_m)
        iargs_f.fresh_from = w.n_keys - 1
        ws_f = torch.zeros(max(1, lib.csa2_index_topk_workspace_size(ctypes.byref(iargs_f), w.topk)),
                           dtype=torch.uint8, device=dev)
        idx_f = torch.empty_like(idx)
        aargs_f = csa2.make_attn_args(dw["q_attn"], dw["kv_codes"], dw["kv_scales"], idx_f, dw["swa"],
                                      dw["swa_pos0"], dw["q_pos"], None, w.window, dw.sm_scale, w.d_v)
        out_f, lse_f = torch.empty_like(out), torch.empty_like(lse)

        def step_fused():
            csa2.csa2_rope_quant_fp4(cache_rows, st, jobs=cache_jobs)
            csa2.csa2_index_topk(iargs_f, w.topk, idx_f, None, row_len, st, workspace=ws_f)
            csa2.csa2_sparse_attn(aargs_f, out_f, lse_f, st, workspace=ws_attn)

        for _ in range(args.warmup):
            step_fused()
        g_f = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_f):
            step_fused()
        t_f = timed(g_f)
        if int(st.item()) != 0:
            raise RuntimeError(f"device status {int(st.item())}")
        fused_cfg = {"calls": "RoPE + cache write, csa2_index_topk (indexer CTAs keep their scores on chip "
                              "and write candidate lists; a merge selects), attention",
                     "ms_per_step": t_f, "tokens_per_s": B * T / (t_f * 1e-3), "launches": 4,
                     "score_bytes_written": 0, "same_idx": bool(torch.equal(idx_f, idx))}
        row_nv = w.d_qk // 2 + w.d_qk // 16
        nv = {"format": "E2M1 + E4M3 per 16, no global scale (report §2.4.4)",
              "ms_per_step": t_nv, "tokens_per_s": B * T / (t_nv * 1e-3), "launches": launches_per_step,
              "sparse_attn_ms": t_a_nv, "sparse_attn_ms_mxfp4": t_a_mx,
              "main_kv_bytes_per_position": row_nv,
              "cache_bytes_per_position": lib.csa2_cache_bytes_per_position(csa2.FMT_NVFP4_E4M3_16, w.d_qk,
                                                                            w.idx_dim),
              "cache_bytes_per_position_512ch": lib.csa2_cache_bytes_per_position(csa2.FMT_NVFP4_E4M3_16,
                                                                                  512, w.idx_dim)}

    # ---- max over ranks
    ms_step, ms_k, e2e_step = max_over_ranks(dist, [ms_step, ms_k, e2e_step], dev)
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    peak, peak_kind = _peaks()
    krl = kernel_rooflines(w, per_kernel, peak, _bf16_peak())
    # the roofline object: the kernel with the longest per-call CUDA-event time in the step
    dom = max(krl, key=lambda n: krl[n]["ms"])
    api_name = {"cache_write": "csa2_rope_quant_fp4", "index_score": "csa2_index_score",
                "topk": "csa2_topk", "sparse_attn": "csa2_sparse_attn"}[dom]
    line = {
        "metric": METRIC, "value": job_throughput(B * T, world, ms_step), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp4-e2m1/f32",
        "data": "synthetic (seeded N(0,1) caches quantised to MXFP4, U(0,1) head weights, 1% planted)",
        "config": {"workload": WORKLOAD, "global_batch": B * world, "seq_len": w.n_keys,
                   "parallelism": f"replicas{world}", "topk": w.topk, "window": w.window,
                   "indexer": f"{w.idx_heads}x{w.idx_dim}", "heads": w.heads,
                   "d_qk": w.d_qk, "d_v": w.d_v,
                   "l2": "flushed between timed steps (256 MiB written, then 256 MiB read so the "
                         "write-back drains; untimed)",
                   "launch": "CUDA graph of the step" if graph is not None else "eager"},
        "achieved_gbs_step": _step_bytes(w) / (ms_step * 1e-3) / 1e9,
        "frac_step": _step_bytes(w) / (ms_step * 1e-3) / 1e9 / peak,
        "roofline": {"bound": "hbm", "kernel": api_name, "achieved": krl[dom]["gbs"],
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": krl[dom]["frac_hbm"], "traffic": None,
                     "algorithmic_bytes": krl[dom]["bytes"], "ms": krl[dom]["ms"],
                     "chosen_as": "longest per-call CUDA-event time of the step's calls"},
        "e2e": {"value": job_throughput(B * T, world, e2e_step), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_step,
                "copies": "pinned host buffers; indexer query + head weights in one upload, the "
                          "attention query uploads on a second branch while the cache write, "
                          "indexer and Top-K run; output downloaded; "
                          + ("one CUDA graph per step" if g_e2e is not None else "eager calls")},
        "kernels_ms": per_kernel,
        "kernels_roofline": krl,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks.summary(),
    }
    if group is not None:
        line["decoder_group"] = group
    if nv is not None:
        line["main_kv_e4m3_16"] = nv
    if pages_cfg is not None:
        line["pages_cache_config"] = pages_cfg
    if fused_cfg is not None:
        line["fused_selection"] = fused_cfg
    if not args.no_prefill:
        line["prefill_indexer"] = prefill_indexer(dev, line["clocks"].get("sm_mhz"))
    if not args.no_indexer_rows:
        try:
            line["indexer_rows"] = indexer_rows(dev)
        except Exception as exc:          # reported, not fatal: the decode line stands
            line["indexer_rows"] = {"error": f"{type(exc).__name__}: {exc}"}
        try:
            line["decode_workloads"] = decode_workloads(dev)
        except Exception as exc:          # reported, not fatal
            line["decode_workloads"] = {"error": f"{type(exc).__name__}: {exc}"}
    if not args.no_cpu_baseline:
        import oracle
        dt, tok = oracle_sample(w, [0, 1])
        line["cpu_baseline"] = {"value": tok / dt, "unit": "tokens/s", "cores": oracle.num_threads(),
                                "cpu_model": cpu_model(), "kind": "oracle",
                                "sample": "2 of 32 sequences: oracle indexer over 65,536 positions, "
                                          "Top-512, fp64 attention"}
    print(json.dumps(line))
    if dist:
        dist.destroy_process_group()
    return 0


def indexer_rows(dev):
    """The indexer steps the decode line does not time, on their own workloads: the Reindex
    layer's scoring of its block pool (2,048 blocks of 8 per sequence, batch 64, 128K context)
    with its Top-512 inside the pool, and the decoder's hierarchical indexer at 1M context
    (batch 4: every causal position scored, Top-512, Top-2,048 blocks of 8).  Each call is
    timed alone after an L2 flush (median of 7); the indexer against the HBM copy rate with
    68 B per scored position plus the pool ids, query and head weights."""
    import ctypes
    import torch
    from fp4_kv_cache_gb300 import csa2, workload
    lib = csa2.load()
    peak, _ = _peaks()
    flush = L2Flush(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)

    def timed(fn):
        ts = []
        for it in range(10):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            e1.synchronize()
            if it >= 3:
                ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    res = {}
    # ---- Reindex: pool scoring + Top-512 within the pool
    w = synth.WORKLOADS["reuse_reindex_decode_128k"]
    dw = workload.build(w, device=dev, kv=False, d_status=st)
    B, T = w.batch, w.n_q
    pool = dw["pool"]
    n_cand = pool.shape[-1] * w.block
    scores = torch.empty((B, T, n_cand), dtype=torch.float32, device=dev)
    row_len = torch.empty((B, T), dtype=torch.int32, device=dev)
    gmax = csa2.group_max_buffer(scores)
    idx = torch.empty((B, T, w.topk), dtype=torch.int32, device=dev)
    iargs = csa2.make_index_args(dw["q_idx"], dw["w_idx"], dw["k_codes"], dw["k_scales"], dw["q_pos"],
                                 w.ratio_m, pool, w.block, gmax)
    ws_i = torch.zeros(max(1, lib.csa2_index_score_workspace_size(ctypes.byref(iargs))),
                       dtype=torch.uint8, device=dev)
    ws_t = torch.empty(max(1, lib.csa2_topk_workspace_size(B * T, n_cand, w.topk, ctypes.byref(iargs))),
                       dtype=torch.uint8, device=dev)

    def score():
        csa2.csa2_index_score(iargs, scores, row_len, st, workspace=ws_i)

    def select():
        csa2.csa2_topk(scores, w.topk, idx, row_len, pool, w.block, d_status=st, workspace=ws_t,
                       group_max=gmax, exact=iargs)

    def chain():
        score()
        select()

    chain()
    t_score, t_select, t_chain = timed(score), timed(select), timed(chain)
    torch.cuda.synchronize(dev)
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())}")
    scored = int(row_len.sum().item())
    ib = scored * 68 + B * T * (pool.shape[-1] * 4 + w.idx_heads * (w.idx_dim * 2 + 4))
    res["reindex_pool_128k"] = {
        "workload": w.name, "batch": B, "context": w.n_keys, "pool_positions": n_cand,
        "positions_scored": scored, "index_score_ms": t_score, "index_bytes": ib,
        "index_gbs": ib / (t_score * 1e-3) / 1e9, "index_frac_hbm": ib / (t_score * 1e-3) / 1e9 / peak,
        "topk_ms": t_select, "ms": t_chain, "tokens_per_s": B * T / (t_chain * 1e-3)}
    del dw, scores, row_len, gmax, idx, ws_i, ws_t, iargs
    torch.cuda.empty_cache()

    # ---- decoder's hierarchical indexer at 1M: scores, Top-512, Top-2,048 blocks
    w = synth.WORKLOADS["hier_indexer_1m"]
    dw = workload.build(w, device=dev, kv=False, d_status=st)
    B, T = w.batch, w.n_q
    scores = torch.empty((B, T, w.n_keys), dtype=torch.float32, device=dev)
    row_len = torch.empty((B, T), dtype=torch.int32, device=dev)
    gmax = csa2.group_max_buffer(scores)
    idx = torch.empty((B, T, w.topk), dtype=torch.int32, device=dev)
    blocks = torch.empty((B, T, w.n_blocks), dtype=torch.int32, device=dev)
    iargs = csa2.make_index_args(dw["q_idx"], dw["w_idx"], dw["k_codes"], dw["k_scales"], dw["q_pos"],
                                 w.ratio_m, None, w.block, gmax)
    ws_i = torch.zeros(max(1, lib.csa2_index_score_workspace_size(ctypes.byref(iargs))),
                       dtype=torch.uint8, device=dev)
    ws_t = torch.empty(max(1, lib.csa2_topk_workspace_size(B * T, w.n_keys, w.topk, ctypes.byref(iargs))), dtype=torch.uint8,
                       device=dev)
    ws_b = torch.empty(max(1, lib.csa2_block_candidates_workspace_size(B * T, w.n_keys, w.block, w.n_blocks,
                                                                        ctypes.byref(iargs))),
                       dtype=torch.uint8, device=dev)

    def score1m():
        csa2.csa2_index_score(iargs, scores, row_len, st, workspace=ws_i)

    def select1m():
        csa2.csa2_topk(scores, w.topk, idx, row_len, d_status=st, workspace=ws_t, group_max=gmax,
                       exact=iargs)

    def blocks1m():
        csa2.csa2_block_candidates(scores, w.n_blocks, blocks, row_len, w.block, st, workspace=ws_b,
                                   exact=iargs)

    def chain1m():
        score1m()
        select1m()
        blocks1m()

    chain1m()
    t_score, t_select, t_blocks, t_chain = timed(score1m), timed(select1m), timed(blocks1m), timed(chain1m)
    torch.cuda.synchronize(dev)
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())}")
    ib = _kernel_bytes(w)
    res["hier_indexer_1m"] = {
        "workload": w.name, "batch": B, "context": w.n_keys, "index_score_ms": t_score,
        "index_bytes": ib, "index_gbs": ib / (t_score * 1e-3) / 1e9,
        "index_frac_hbm": ib / (t_score * 1e-3) / 1e9 / peak, "topk_ms": t_select,
        "block_candidates_ms": t_blocks, "ms": t_chain, "tokens_per_s": B * T / (t_chain * 1e-3)}
    return res


def decode_workloads(dev):
    """The attention workloads the default line does not time, each on its own sizes: the
    tiny Full decode layer (batch 1, 4,096 positions, indexer 4 x 64, 16 heads over a
    128-dim latent; index score, exact Top-512, attention) as a latency; the Reuse layer at
    batch 64 x 131,072 (attention over the given Top-512 + SWA 128; no indexer work); and
    the decoder's SWA bounded replay (8 x 128 tokens from s = 131,072, SWA keys truncated at
    s).  The last two against the HBM copy rate with their algorithmic bytes (gathered
    main-KV rows, indices, SWA rows, query, output).  Each is one CUDA graph, replayed after
    an L2 flush; median of 20."""
    import ctypes
    import torch
    from fp4_kv_cache_gb300 import csa2, workload
    lib = csa2.load()
    peak, _ = _peaks()
    flush = L2Flush(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)

    def graph_ms(fn, reps=20):
        fn()
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        ts = []
        for it in range(reps + 3):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            e1.synchronize()
            if it >= 3:
                ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    res = {}
    # ---- tiny Full decode layer (latency)
    w = synth.WORKLOADS["tiny_full_decode"]
    dw = workload.build(w, device=dev, d_status=st)
    B, T = w.batch, w.n_q
    scores = torch.empty((B, T, w.n_keys), dtype=torch.float32, device=dev)
    row_len = torch.empty((B, T), dtype=torch.int32, device=dev)
    idx = torch.empty((B, T, w.topk), dtype=torch.int32, device=dev)
    out = torch.empty((B, T, w.heads, w.d_v), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, T, w.heads), dtype=torch.float32, device=dev)
    iargs = csa2.make_index_args(dw["q_idx"], dw["w_idx"], dw["k_codes"], dw["k_scales"], dw["q_pos"],
                                 w.ratio_m)
    aargs = csa2.make_attn_args(dw["q_attn"], dw["kv_codes"], dw["kv_scales"], idx, dw["swa"],
                                dw["swa_pos0"], dw["q_pos"], None, w.window, dw.sm_scale, w.d_v)
    ws_i = torch.zeros(max(1, lib.csa2_index_score_workspace_size(ctypes.byref(iargs))), dtype=torch.uint8,
                       device=dev)
    ws_t = torch.empty(max(1, lib.csa2_topk_workspace_size(B * T, w.n_keys, w.topk, ctypes.byref(iargs))),
                       dtype=torch.uint8, device=dev)
    ws_a = torch.empty(max(1, lib.csa2_sparse_attn_workspace_size(ctypes.byref(aargs))), dtype=torch.uint8,
                       device=dev)

    def tiny_layer():
        csa2.csa2_index_score(iargs, scores, row_len, st, workspace=ws_i)
        csa2.csa2_topk(scores, w.topk, idx, row_len, d_status=st, workspace=ws_t, exact=iargs)
        csa2.csa2_sparse_attn(aargs, out, lse, st, workspace=ws_a)

    t = graph_ms(tiny_layer)
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())}")
    res["tiny_full_decode"] = {"workload": w.name, "batch": B, "context": w.n_keys, "latency_ms": t,
                               "launches": 3, "calls": "index score, exact Top-512, attention"}
    del dw, scores, row_len, idx, out, lse, ws_i, ws_t, ws_a
    torch.cuda.empty_cache()

    # ---- Reuse layer at batch 64 x 131,072 (given Top-512)
    w = synth.WORKLOADS["reuse_reindex_decode_128k"]
    dw = workload.build(w, device=dev, kidx=False, d_status=st)
    B, T = w.batch, w.n_q
    out = torch.empty((B, T, w.heads, w.d_v), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, T, w.heads), dtype=torch.float32, device=dev)
    aargs = csa2.make_attn_args(dw["q_attn"], dw["kv_codes"], dw["kv_scales"], dw["reuse_idx"], dw["swa"],
                                dw["swa_pos0"], dw["q_pos"], None, w.window, dw.sm_scale, w.d_v)
    ws_a = torch.empty(max(1, lib.csa2_sparse_attn_workspace_size(ctypes.byref(aargs))), dtype=torch.uint8,
                       device=dev)

    def reuse():
        csa2.csa2_sparse_attn(aargs, out, lse, st, workspace=ws_a)

    t = graph_ms(reuse)
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())}")
    kv_row = w.d_qk // 2 + w.d_qk // 32
    ab = B * T * (w.topk * (kv_row + 4) + w.window * w.d_qk * 2 + w.heads * w.d_qk * 2 + w.heads * w.d_v * 2)
    flop = 2.0 * B * T * w.heads * (w.topk + w.window) * (w.d_qk + w.d_v)
    res["reuse_decode_128k"] = {
        "workload": w.name, "batch": B, "context": w.n_keys, "sparse_attn_ms": t,
        "tokens_per_s": B * T / (t * 1e-3), "bytes": ab, "gbs": ab / (t * 1e-3) / 1e9,
        "frac_hbm": ab / (t * 1e-3) / 1e9 / peak, "tflops": flop / (t * 1e-3) / 1e12,
        "frac_bf16": flop / (t * 1e-3) / 1e12 / _bf16_peak()}
    del dw, out, lse, ws_a
    torch.cuda.empty_cache()

    # ---- SWA bounded replay: 128 tokens from s through attention (given Top-512 each)
    w = synth.WORKLOADS["swa_replay_prefill"]
    dw = workload.build(w, device=dev, kidx=False, d_status=st)
    B, T = w.batch, w.n_q
    out = torch.empty((B, T, w.heads, w.d_v), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, T, w.heads), dtype=torch.float32, device=dev)
    aargs = csa2.make_attn_args(dw["q_attn"], dw["kv_codes"], dw["kv_scales"], dw["reuse_idx"], dw["swa"],
                                dw["swa_pos0"], dw["q_pos"], dw["swa_start"], w.window, dw.sm_scale, w.d_v)
    ws_a = torch.empty(max(1, lib.csa2_sparse_attn_workspace_size(ctypes.byref(aargs))), dtype=torch.uint8,
                       device=dev)

    def replay():
        csa2.csa2_sparse_attn(aargs, out, lse, st, workspace=ws_a)

    t = graph_ms(replay)
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {int(st.item())}")
    n_swa_keys = sum(min(w.window, j + 1) for j in range(T))          # query s + j sees j + 1
    # per sequence: every query's gathered rows, indices, query and output, and the T
    # replayed SWA rows (tokens s .. s + T - 1), each needed once
    ab = B * (T * (w.topk * (kv_row + 4) + w.heads * w.d_qk * 2 + w.heads * w.d_v * 2) + T * w.d_qk * 2)
    flop = 2.0 * B * w.heads * (T * w.topk + n_swa_keys) * (w.d_qk + w.d_v)
    res["swa_replay_prefill"] = {
        "workload": w.name, "batch": B, "queries": T, "replay_start": w.swa_start, "sparse_attn_ms": t,
        "tokens_per_s": B * T / (t * 1e-3), "bytes": ab, "gbs": ab / (t * 1e-3) / 1e9,
        "frac_hbm": ab / (t * 1e-3) / 1e9 / peak, "tflops": flop / (t * 1e-3) / 1e12,
        "frac_bf16": flop / (t * 1e-3) / 1e12 / _bf16_peak()}
    return res


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or None."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for ln in open("/proc/cpuinfo"):
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


PREFILL_WORKLOAD = "prefill_chunk_m2"


def prefill_indexer(dev, sm_mhz, with_chunk=True):
    """Tensor-core indexer over one prefill chunk: FP4 dot TFLOP/s (2 x heads x d_i per
    visible (query, position) pair) against the FP4 tensor peak (the measured bf16 GEMM
    peak x 6, the nominal fp4/bf16 ratio) and against the CUDA-core bound of its epilogue
    (one max and one fma in fp32 per pair and head)."""
    import torch
    from fp4_kv_cache_gb300 import csa2, workload
    w = synth.WORKLOADS[PREFILL_WORKLOAD]
    dw = workload.build(w, device=dev, kv=with_chunk)
    B, T = w.batch, w.n_q
    scores = torch.empty((B, T, w.n_keys), dtype=torch.float32, device=dev)
    row_len = torch.empty((B, T), dtype=torch.int32, device=dev)
    gmax = csa2.group_max_buffer(scores)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    iargs = csa2.make_index_args(dw["q_idx"], dw["w_idx"], dw["k_codes"], dw["k_scales"], dw["q_pos"],
                                 w.ratio_m, group_max=gmax)
    import ctypes
    lib = csa2.load()
    ws_index = torch.zeros(max(1, lib.csa2_index_score_workspace_size(ctypes.byref(iargs))),
                           dtype=torch.uint8, device=dev)     # zero before first use; calls keep it so
    flush = L2Flush(dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    ms = []
    for it in range(8):
        flush()
        e0, e1 = ev(), ev()
        e0.record()
        csa2.csa2_index_score(iargs, scores, row_len, st, workspace=ws_index)
        e1.record()
        e1.synchronize()
        if it >= 3:
            ms.append(e0.elapsed_time(e1))
    t = statistics.median(ms)
    chunk = None
    if with_chunk:
        # the whole chunk (encoder Full layer): indexer, per-query Top-512 (fed the indexer's
        # group maxima), then attention over the 512 selected entries + the SWA window
        idx = torch.empty((B, T, w.topk), dtype=torch.int32, device=dev)
        out = torch.empty((B, T, w.heads, w.d_v), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((B, T, w.heads), dtype=torch.float32, device=dev)
        aargs = csa2.make_attn_args(dw["q_attn"], dw["kv_codes"], dw["kv_scales"], idx, dw["swa"],
                                    dw["swa_pos0"], dw["q_pos"], None, w.window, dw.sm_scale, w.d_v)
        ws_topk = torch.empty(max(1, lib.csa2_topk_workspace_size(B * T, w.n_keys, w.topk, ctypes.byref(iargs))),
                              dtype=torch.uint8, device=dev)
        ws_attn = torch.empty(max(1, lib.csa2_sparse_attn_workspace_size(ctypes.byref(aargs))),
                              dtype=torch.uint8, device=dev)
        per = {"index_score": [], "topk": [], "sparse_attn": [], "chunk": []}
        for it in range(7):
            flush()
            e = [ev() for _ in range(4)]
            e[0].record()
            csa2.csa2_index_score(iargs, scores, row_len, st, workspace=ws_index)
            e[1].record()
            csa2.csa2_topk(scores, w.topk, idx, row_len, d_status=st, workspace=ws_topk, group_max=gmax,
                       exact=iargs)
            e[2].record()
            csa2.csa2_sparse_attn(aargs, out, lse, st, workspace=ws_attn)
            e[3].record()
            e[3].synchronize()
            if it >= 2:
                for k, (a, b) in zip(["index_score", "topk", "sparse_attn", "chunk"],
                                     [(0, 1), (1, 2), (2, 3), (0, 3)]):
                    per[k].append(e[a].elapsed_time(e[b]))
        if int(st.item()) != 0:
            raise RuntimeError(f"device status {int(st.item())}")
        med = {k: statistics.median(v) for k, v in per.items()}
        attn_flop = 2.0 * B * T * w.heads * (w.topk + w.window) * (w.d_qk + w.d_v)
        chunk = {"layer": "encoder Full layer at ratio 2: indexer, Top-512, attention (512 + SWA 128)",
                 "ms": med["chunk"], "tokens_per_s": B * T / (med["chunk"] * 1e-3),
                 "ms_per_call": {k: med[k] for k in ("index_score", "topk", "sparse_attn")},
                 "attn_tflops": attn_flop / (med["sparse_attn"] * 1e-3) / 1e12,
                 "launches": 3}
    pairs = int(row_len.sum().item())
    flop = 2.0 * pairs * w.idx_heads * w.idx_dim
    tf = flop / (t * 1e-3) / 1e12
    d = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if os.path.exists(
        os.path.join(ROOT, "MEASURED_PEAKS.json")) else {}
    bf16 = float(d.get("bf16_tflops", 1900.0))
    fp4_peak = 6.0 * bf16
    mhz = sm_mhz or 2070.0
    alu_tf = 152 * 128 * mhz * 1e6 / 2 * (2 * w.idx_dim) / 1e12
    res = {"workload": PREFILL_WORKLOAD, "queries": B * T, "positions": w.n_keys,
           "visible_pairs": pairs, "ms": t, "achieved": tf, "unit": "TFLOP/s",
            "fp4_peak": fp4_peak,
            "fp4_peak_kind": ("measured bf16 x 6" if "bf16_tflops" in d else "fallback bf16 x 6"),
           "frac_fp4": tf / fp4_peak, "alu_peak": alu_tf, "frac_alu": tf / alu_tf,
           "l2": "flushed between timed launches (write + read of 256 MiB)"}
    if chunk is not None:
        res["chunk"] = chunk
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-group", action="store_true")
    ap.add_argument("--no-indexer-rows", action="store_true",
                    help="skip timing the Reindex pool scoring (128K) and the 1M hierarchical indexer")
    ap.add_argument("--indexer-rows-only", action="store_true",
                    help="time only those and print their object")
    ap.add_argument("--no-nvfp4", action="store_true",
                    help="skip the step over the E2M1 + E4M3/16 main-KV cache")
    ap.add_argument("--prefill-only", action="store_true",
                    help="time only the prefill indexer (for profiling it) and print its object")
    ap.add_argument("--workloads-only", action="store_true",
                    help="time only the tiny decode, Reuse and SWA-replay workloads and print their object")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.prefill_only:
        import torch
        torch.cuda.set_device(0)
        print(json.dumps({"prefill_indexer": prefill_indexer(torch.device("cuda", 0), None, with_chunk=False)}))
        return 0
    if args.workloads_only:
        import torch
        torch.cuda.set_device(0)
        print(json.dumps({"decode_workloads": decode_workloads(torch.device("cuda", 0))}))
        return 0
    if args.indexer_rows_only:
        import torch
        torch.cuda.set_device(0)
        print(json.dumps({"indexer_rows": indexer_rows(torch.device("cuda", 0))}))
        return 0
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
