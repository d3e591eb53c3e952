"""Host-side arithmetic of bench.py (CPU only): the algorithmic byte counts behind the
roofline numbers, checked against each other and against the workload's shapes."""
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from fp4_kv_cache_gb300 import synth  # noqa: E402


def test_indexer_bytes_are_the_scan():
    w = synth.WORKLOADS["full_decode_64k"]
    # 68 B per position (64 B of codes + 4 scale bytes) over 32 x 65,536 positions, plus
    # the bf16 query and the fp32 head weights of 32 queries x 32 heads
    assert bench._kernel_bytes(w) == 32 * 65536 * 68 + 32 * 32 * (128 * 2 + 4)


def test_kernel_rooflines_add_up_to_the_step():
    w = synth.WORKLOADS["full_decode_64k"]
    ms = {"cache_write": 0.0078, "index_score": 0.0369, "topk": 0.0205, "sparse_attn": 0.0389}
    r = bench.kernel_rooflines(w, ms, 6684.5, 1928.5)
    assert set(r) == set(ms)
    # the step's bytes are the cache write, the scan and the attention's
    assert r["cache_write"]["bytes"] + r["index_score"]["bytes"] + r["sparse_attn"]["bytes"] == \
        bench._step_bytes(w)
    assert r["index_score"]["frac_hbm"] == pytest.approx(bench._kernel_bytes(w) / 36.9e-6 / 6684.5e9)
    # attention: 32 queries x 64 heads x 640 keys x (576 + 512) x 2 flops
    assert r["sparse_attn"]["tflops"] == pytest.approx(2.0 * 32 * 64 * 640 * 1088 / 38.9e-6 / 1e12)
    assert 0 < r["sparse_attn"]["frac_bf16"] < 1 and 0 < r["topk"]["frac_hbm"] < 1
    json.dumps(r)                          # it goes into the JSON line as it is
    assert bench.kernel_rooflines(w, {"other": 1.0, "topk": 0.0}, 6684.5, 1928.5) == {}
