"""The C-ABI library on the host: it builds, loads, exports every entry point the header
declares, computes the cache byte ledger, and rejects bad arguments before launching
anything (none of these calls reach the GPU)."""
import ctypes
import os
import re
import subprocess

import pytest

from fp4_kv_cache_gb300 import build as libbuild
from fp4_kv_cache_gb300 import csa2
from fp4_kv_cache_gb300.layers import layer_mode

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "csa2.h")).read()
    return sorted(set(re.findall(r"CSA2_API[^;(]*?\b(csa2_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return csa2.load(build_if_missing=False)


def test_exports_every_declared_symbol(lib):
    syms = _declared_symbols()
    assert len(syms) == 21
    for s in syms:
        assert hasattr(lib, s), s
    out = os.popen(f"nm -D --defined-only {libbuild.LIB}").read()
    exported = set(re.findall(r" T (csa2_\w+)", out))
    assert exported == set(syms)


def _ledger():
    vals = {}
    for line in open(os.path.join(GOLDEN, "cache_ledger.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            vals[k] = int(v)
    return vals


def test_cache_byte_ledger(lib):
    g = _ledger()
    per_pos = csa2.cache_bytes_per_position(csa2.FMT_NVFP4_E4M3_16, 512, 128)
    assert per_pos == g["per_position_total"] == (g["main_kv_codes_512ch"] + g["main_kv_scales_e4m3_per16"]
                                                  + g["indexer_k_codes_128ch"]
                                                  + g["indexer_k_scales_e8m0_per32"])
    # three encoder source layers at ratio 2 + one decoder source layer at ratio 1
    assert per_pos * 3 // 2 + per_pos == g["per_token_total"]
    assert 448 * 6 == g["nvfp4_no_global_scale_max"]
    assert 2048 * 8 == g["pool_max_positions"]
    # the default MXFP4 main KV at 512 + 64 dims: 288 + 18 bytes, plus the 68-byte key
    assert csa2.cache_bytes_per_position(csa2.FMT_MXFP4, 576, 128) == 288 + 18 + 64 + 4
    assert csa2.cache_bytes_per_position(csa2.FMT_MXFP4, 500, 128) == 0
    # the report's main-KV format at 512 + 64 dims: 288 + 36 bytes, plus the key
    assert csa2.cache_bytes_per_position(csa2.FMT_NVFP4_E4M3_16, 576, 128) == 288 + 36 + 64 + 4
    assert csa2.cache_bytes_per_position(csa2.FMT_NVFP4_E4M3_16, 40, 128) == 0


def test_status_strings(lib):
    assert csa2.status_string(0) == "ok"
    assert "invalid" in csa2.status_string(1)
    assert lib.csa2_version() >= 100


FAKE = ctypes.c_void_p(256)   # never dereferenced: every call below fails validation first


def test_quant_rejects_bad_shapes(lib):
    assert lib.csa2_quant_fp4(FAKE, 0, 4, 33, 33, FAKE, 17, FAKE, 2, 0, None, None) == 1
    assert lib.csa2_quant_fp4(FAKE, 5, 4, 32, 32, FAKE, 16, FAKE, 1, 0, None, None) == 1
    assert lib.csa2_quant_fp4(FAKE, 0, 4, 32, 16, FAKE, 16, FAKE, 1, 0, None, None) == 1
    # E2M1 + E4M3/16: one scale per 16 values, so 32 columns need 2 scale bytes per row
    assert lib.csa2_quant_fp4(FAKE, 0, 4, 32, 32, FAKE, 16, FAKE, 1, 1, None, None) == 1
    assert lib.csa2_quant_fp4(FAKE, 0, 4, 40, 40, FAKE, 20, FAKE, 3, 1, None, None) == 1  # 40 % 16
    assert lib.csa2_quant_fp4(FAKE, 0, 4, 32, 32, FAKE, 16, FAKE, 2, 2, None, None) == 1  # no format 2
    assert lib.csa2_dequant_fp4(FAKE, 16, FAKE, 1, 4, 32, 1, FAKE, 0, 32, None) == 1
    assert lib.csa2_quant_fp4(None, 0, 0, 32, 32, None, 16, None, 1, 0, None, None) == 0


def test_quant_batch_rejects_bad_args(lib):
    def jobs(*specs):
        arr = (csa2.QuantJob * max(1, len(specs)))()
        for i, (xt, rows, cols, ldx, ldc, lds) in enumerate(specs):
            arr[i] = csa2.QuantJob(FAKE, xt, rows, cols, ldx, FAKE, ldc, FAKE, lds)
        return arr
    ok = (0, 4, 32, 32, 16, 1)
    assert lib.csa2_quant_fp4_batch(jobs(ok), 5, 0, None, None) == 1          # more than 4 jobs
    assert lib.csa2_quant_fp4_batch(jobs(ok), -1, 0, None, None) == 1
    assert lib.csa2_quant_fp4_batch(jobs(ok), 1, 1, None, None) == 1          # NVFP4: 2 scales per row
    assert lib.csa2_quant_fp4_batch(jobs(ok), 1, 2, None, None) == 1          # no format 2
    assert lib.csa2_quant_fp4_batch(None, 1, 0, None, None) == 1
    assert lib.csa2_quant_fp4_batch(jobs(ok, (0, 4, 33, 33, 17, 2)), 2, 0, None, None) == 1
    assert lib.csa2_quant_fp4_batch(jobs(ok, (5, 4, 32, 32, 16, 1)), 2, 0, None, None) == 1
    assert lib.csa2_quant_fp4_batch(jobs(ok, (0, 4, 32, 16, 16, 1)), 2, 0, None, None) == 1
    assert lib.csa2_quant_fp4_batch(None, 0, 0, None, None) == 0              # nothing to do
    empty = (csa2.QuantJob * 1)()
    empty[0] = csa2.QuantJob(None, 0, 0, 32, 32, None, 16, None, 1)
    assert lib.csa2_quant_fp4_batch(empty, 1, 0, None, None) == 0             # zero rows: no launch


def test_rope_quant_rejects_bad_args(lib):
    def job(rows=4, cols=64, ldx=64, rope=32, pos=FAKE, cs=FAKE, n_pos=10, ldc=32, lds=2, fmt=0,
            x=FAKE, codes=FAKE):
        j = (csa2.RopeQuantJob * 1)()
        j[0] = csa2.RopeQuantJob(x.value if x else None, rows, cols, ldx, rope, pos.value if pos else None,
                                 cs.value if cs else None, n_pos, codes.value if codes else None, ldc,
                                 FAKE.value, lds, fmt)
        return j
    f = lib.csa2_rope_quant_fp4
    assert f(job(rope=31), 1, None, None) == 1                     # odd rotated width
    assert f(job(rope=66), 1, None, None) == 1                     # wider than the row
    assert f(job(pos=None), 1, None, None) == 1                    # rotation without positions
    assert f(job(n_pos=0), 1, None, None) == 1
    assert f(job(ldx=68), 1, None, None) == 1                      # rows not 16-byte aligned
    assert f(job(x=ctypes.c_void_p(264)), 1, None, None) == 1
    assert f(job(ldc=34), 1, None, None) == 1                      # code rows not 4-byte aligned
    assert f(job(cols=48, ldx=48, ldc=24, lds=1), 1, None, None) == 1    # 48 % 32
    assert f(job(fmt=1, lds=2), 1, None, None) == 1                # E4M3/16: 4 scales per row
    assert f(job(fmt=2), 1, None, None) == 1
    assert f(job(), 5, None, None) == 1                            # more than 4 jobs
    assert f(None, 1, None, None) == 1
    assert f(None, 0, None, None) == 0                             # nothing to do
    assert f(job(rows=0), 1, None, None) == 0                      # zero rows: no launch


def test_selftest_rejects_bad_args(lib):
    assert lib.csa2_selftest_bounded_wait(0, FAKE, None) == 1                  # no polls
    assert lib.csa2_selftest_bounded_wait((1 << 20) + 1, FAKE, None) == 1      # too many
    assert lib.csa2_selftest_bounded_wait(16, None, None) == 1                 # status required


def test_index_rejects_bad_args(lib):
    a = csa2.IndexArgs()
    a.batch, a.n_q, a.n_heads, a.head_dim, a.ratio_m, a.n_keys = 1, 1, 4, 48, 1, 100
    a.q = a.w = a.k_codes = a.k_scales = FAKE
    a.mode, a.block = 0, 8
    f = lib.csa2_index_score
    assert f(ctypes.byref(a), FAKE, FAKE, None, 0, None, None) == 1        # head_dim 48
    a.head_dim = 128
    a.n_heads = 65
    assert f(ctypes.byref(a), FAKE, FAKE, None, 0, None, None) == 1        # too many heads
    a.n_heads = 4
    a.ratio_m = 0
    assert f(ctypes.byref(a), FAKE, FAKE, None, 0, None, None) == 1
    a.ratio_m = 1
    a.k_codes = ctypes.c_void_p(257)                                       # misaligned
    assert f(ctypes.byref(a), FAKE, FAKE, None, 0, None, None) == 1
    a.k_codes = FAKE
    a.fresh_from = -1                                                      # no such position
    assert f(ctypes.byref(a), FAKE, FAKE, None, 0, None, None) == 1
    a.fresh_from = 0
    g = lib.csa2_index_topk                                                # (args, k, idx, out_scores, row_len, ws, bytes, status, stream)
    assert g(ctypes.byref(a), -1, FAKE, None, None, FAKE, 1 << 20, None, None) == 1      # k < 0
    assert g(ctypes.byref(a), 512, None, None, None, FAKE, 1 << 20, None, None) == 1     # idx missing
    a.q = ctypes.c_void_p(4104)                                            # q not 16-byte aligned
    assert g(ctypes.byref(a), 512, FAKE, None, None, FAKE, 1 << 20, None, None) == 1
    a.q = FAKE
    a.mode, a.n_pool_blocks, a.pool_blocks = 1, 16, None                   # pool missing
    assert f(ctypes.byref(a), FAKE, FAKE, None, 0, None, None) == 1
    a.batch = 0
    assert f(ctypes.byref(a), None, None, None, 0, None, None) == 0        # empty: nothing to do


def test_select_and_attn_reject_bad_args(lib):
    T, B = lib.csa2_topk, lib.csa2_block_candidates
    assert T(FAKE, -1, 10, None, None, None, 8, None, 4, FAKE, None, None, 0, None, None) == 1
    assert T(FAKE, 2, 10, None, None, FAKE, 8, None, 4, FAKE, None, None, 0, None, None) == 1
    assert T(FAKE, 0, 10, None, None, None, 8, None, 4, FAKE, None, None, 0, None, None) == 0
    need = lib.csa2_topk_workspace_size(2, 64, 4, None)
    assert T(FAKE, 2, 64, None, ctypes.c_void_p(258), None, 8, None, 4, FAKE, None, FAKE,
             need, None, None) == 1                                             # misaligned
    need = lib.csa2_block_candidates_workspace_size(4, 1 << 20, 8, 2048, None)
    assert need >= 4 * (1 << 17) * 4
    assert B(FAKE, 4, 1 << 20, None, 8, 2048, None, FAKE, FAKE, need - 1, None, None) == 4
    # exact order: the context must describe these scores (rows, candidates, pool), and
    # row_len is required; its band slots make the workspace larger
    a = csa2.IndexArgs()
    a.batch, a.n_q, a.n_heads, a.head_dim, a.ratio_m, a.n_keys = 2, 3, 32, 128, 1, 1000
    a.q = a.w = a.k_codes = a.k_scales = FAKE
    a.mode, a.block = 0, 8
    ra = ctypes.byref(a)
    ne = lib.csa2_topk_workspace_size(6, 1000, 512, ra)
    assert ne > lib.csa2_topk_workspace_size(6, 1000, 512, None) + 6 * 26 * 2048 * 4 - 1
    assert T(FAKE, 5, 1000, FAKE, None, None, 8, ra, 512, FAKE, None, FAKE, ne, None, None) == 1   # rows
    assert T(FAKE, 6, 999, FAKE, None, None, 8, ra, 512, FAKE, None, FAKE, ne, None, None) == 1    # n
    assert T(FAKE, 6, 1000, None, None, None, 8, ra, 512, FAKE, None, FAKE, ne, None, None) == 1   # row_len
    assert T(FAKE, 6, 1000, FAKE, None, FAKE, 8, ra, 512, FAKE, None, FAKE, ne, None, None) == 1   # pool in FULL
    assert T(FAKE, 6, 1000, FAKE, None, None, 8, ra, 512, FAKE, None, FAKE, ne - 1, None, None) == 4
    a.mode, a.pool_blocks, a.n_pool_blocks = 1, FAKE, 100                           # POOL: 800 candidates
    other = ctypes.c_void_p(4096)
    assert T(FAKE, 6, 800, FAKE, None, other, 8, ra, 512, FAKE, None, FAKE, ne, None, None) == 1   # other pool
    nb_ws = lib.csa2_block_candidates_workspace_size(6, 800, 8, 64, ra)
    assert B(FAKE, 6, 800, FAKE, 8, 64, ra, FAKE, FAKE, nb_ws, None, None) == 1     # blocks need FULL
    a = csa2.AttnArgs()
    a.batch, a.n_q, a.n_heads, a.d_qk, a.d_v, a.topk, a.window = 1, 1, 64, 576, 600, 512, 128
    a.q = a.idx = a.kv_codes = a.kv_scales = FAKE
    a.n_kv = 10
    assert lib.csa2_sparse_attn(ctypes.byref(a), FAKE, None, None, 0, None, None) == 1   # d_v > d_qk
    a.d_v = 512
    a.kv_fmt = 2                                                                         # no format 2
    assert lib.csa2_sparse_attn(ctypes.byref(a), FAKE, None, None, 0, None, None) == 1
    a.kv_fmt = csa2.FMT_NVFP4_E4M3_16
    a.swa, a.n_swa, a.swa_pos0, a.q_pos = FAKE, 128, None, FAKE                          # no pos0
    assert lib.csa2_sparse_attn(ctypes.byref(a), FAKE, None, None, 0, None, None) == 1


def test_layer_schedule_counts():
    # review page (papers.chlience.com), zero-based schedule table: 4 source layers, 8
    # indexing layers, 30 Reuse layers, 38 layers with global attention
    modes = [layer_mode(i) for i in range(40)]
    assert modes[:2] == ["swa", "swa"]
    assert [i for i, m in enumerate(modes) if m == "full"] == [2, 8, 14, 20]
    assert [i for i, m in enumerate(modes) if m == "reindex"] == [24, 28, 32, 36]
    assert modes.count("reuse") == 30
    assert sum(m != "swa" for m in modes) == 38


def test_header_is_plain_c(tmp_path):
    # the boundary is a C ABI: the header compiles as strict C11 (no C++ or CUDA types), and
    # its argument structs can be zero-initialised and sized from C
    src = tmp_path / "use_header.c"
    src.write_text('#include "csa2.h"\n'
                   'int main(void) {\n'
                   '    csa2_index_args i = {0}; csa2_attn_args a = {0};\n'
                   '    csa2_quant_job q = {0}; csa2_rope_quant_job r = {0};\n'
                   '    return (int)(sizeof i + sizeof a + sizeof q + sizeof r == 0);\n'
                   '}\n')
    out = tmp_path / "use_header.o"
    r = subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-I", os.path.join(ROOT, "include"), "-c", str(src), "-o", str(out)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
