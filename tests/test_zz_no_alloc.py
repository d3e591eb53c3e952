"""csa2_index_score_noalloc against csa2_index_score (needs a GB300).

Some callers cannot allocate device memory when they score -- a server that splits all
device memory into fixed pools at start-up, a plug-in inside a framework that owns the
allocator, a decode loop that must not block on the allocator -- so they cannot pass the
workspace csa2_index_score wants.  csa2_index_score_noalloc takes no workspace and uses
the library's own static device scratch instead.  Its results must be exactly those of
csa2_index_score (scores are compared bit for bit, as in the other indexer tests), on
two calls in a row, since the second call finds the first call's scratch contents.

This file is collected last, so a run that stops at the first failure has already run
every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from fp4_kv_cache_gb300 import csa2, synth, workload

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _bits_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    return np.array_equal(a.cpu().numpy().view(np.uint32), b.cpu().numpy().view(np.uint32))


@pytest.mark.parametrize("name,wl", [
    ("full", synth.WORKLOADS["full_decode_64k"].scaled(batch=3, n_q=2, n_keys=5003, q_pos0=4000)),
    ("pool", synth.WORKLOADS["reuse_reindex_decode_128k"].scaled(batch=2, n_keys=40000,
                                                                q_pos0=39999, n_blocks=700)),
])
def test_noalloc_matches_workspace_entry_point(name, wl):
    dw = workload.build(wl, kv=False, device=DEV)
    pool = dw.t.get("pool")
    args = csa2.make_index_args(dw["q_idx"], dw["w_idx"], dw["k_codes"], dw["k_scales"],
                                dw["q_pos"], wl.ratio_m, pool, wl.block)
    lib = csa2.load()
    need = lib.csa2_index_score_workspace_size(ctypes.byref(args))
    assert 0 < need <= 256 * 1024          # a request that uses scratch, within the limit
    B, T = wl.batch, wl.n_q
    n_cand = wl.n_keys if pool is None else pool.shape[-1] * wl.block
    ref = torch.full((B, T, n_cand), float("nan"), dtype=torch.float32, device=DEV)
    ref_len = torch.full((B, T), -1, dtype=torch.int32, device=DEV)
    csa2.csa2_index_score(args, ref, ref_len)
    torch.cuda.synchronize()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        got = torch.full_like(ref, float("nan"))
        got_len = torch.full_like(ref_len, -1)
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        status = lib.csa2_index_score_noalloc(ctypes.byref(args), ctypes.c_void_p(got.data_ptr()),
                                              ctypes.c_void_p(got_len.data_ptr()),
                                              ctypes.c_void_p(st.data_ptr()), stream)
        assert status == 0, csa2.status_string(status)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, f"call {call}: device status {int(st.item())}"
        assert torch.equal(got_len, ref_len), f"call {call}"
        for b in range(B):
            for t in range(T):
                L = int(ref_len[b, t])
                assert _bits_equal(got[b, t, :L], ref[b, t, :L]), f"{name} call {call} row ({b},{t})"


def test_noalloc_rejects_requests_beyond_its_scratch():
    # 32,769 query rows on tensor-core-eligible arguments need 262,152 bytes of counters,
    # one row more than the 256 KB array holds: CSA2_ERR_WORKSPACE before anything is
    # launched, outputs untouched.  Every buffer is allocated at its full size anyway.
    rows, H, d, N = 32769, 1, 128, 64
    q = torch.zeros((1, rows, H, d), dtype=torch.bfloat16, device=DEV)
    w = torch.ones((1, rows, H), dtype=torch.float32, device=DEV)
    kc = torch.zeros((1, N, d // 2), dtype=torch.uint8, device=DEV)
    ks = torch.full((1, N, d // 32), 127, dtype=torch.uint8, device=DEV)
    args = csa2.make_index_args(q, w, kc, ks)
    lib = csa2.load()
    assert lib.csa2_index_score_workspace_size(ctypes.byref(args)) > 256 * 1024
    scores = torch.full((1, rows, N), float("nan"), dtype=torch.float32, device=DEV)
    row_len = torch.full((1, rows), -7, dtype=torch.int32, device=DEV)
    status = lib.csa2_index_score_noalloc(ctypes.byref(args), ctypes.c_void_p(scores.data_ptr()),
                                          ctypes.c_void_p(row_len.data_ptr()), None,
                                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert status == csa2.ERR_WORKSPACE
    assert bool(torch.isnan(scores).all()) and bool((row_len == -7).all())
