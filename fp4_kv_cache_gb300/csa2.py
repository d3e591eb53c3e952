"""Thin Python binding of libcsa2.so (include/csa2.h) -- argument marshalling only.

Every step of the path runs in the library's CUDA kernels.  PyTorch provides device
memory (tensors) and the stream (the current CUDA stream unless one is given).  The
``csa2_*`` functions mirror the C entry points one to one; the short-named helpers
(``quant_fp4``, ``index_score``, ``topk``, ``block_candidates``, ``sparse_attn``)
allocate the outputs with torch and call them.  There is no CPU fallback: if the
library or a GPU is missing, the first call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional

import torch

from . import build as _build

_lib = None
_lock = threading.Lock()

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_WORKSPACE = 0, 1, 2, 3, 4
DEV_BAD_INDEX, DEV_BAD_POOL, DEV_NONFINITE, DEV_TIMEOUT = 0x1, 0x2, 0x4, 0x8
DEV_SCORE_RANGE, DEV_BAND_LIMIT = 0x10, 0x20
EXACT_BAND_CAP = 2048
BF16, F32 = 0, 1
FMT_MXFP4, FMT_NVFP4_E4M3_16 = 0, 1
SWA_BF16, SWA_MXFP8 = 0, 1
FMT_BLOCK = {FMT_MXFP4: 32, FMT_NVFP4_E4M3_16: 16}     # values per scale byte
INDEX_FULL, INDEX_POOL = 0, 1

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64


class IndexArgs(ctypes.Structure):
    """csa2_index_args"""
    _fields_ = [("batch", _I32), ("n_q", _I32), ("n_heads", _I32), ("head_dim", _I32),
                ("ratio_m", _I32), ("n_keys", _I64), ("q", _P), ("w", _P), ("k_codes", _P),
                ("k_scales", _P), ("q_pos", _P), ("mode", ctypes.c_int), ("pool_blocks", _P),
                ("n_pool_blocks", _I32), ("block", _I32), ("group_max", _P), ("fresh_from", _I64)]


class AttnArgs(ctypes.Structure):
    """csa2_attn_args"""
    _fields_ = [("batch", _I32), ("n_q", _I32), ("n_heads", _I32), ("d_qk", _I32), ("d_v", _I32),
                ("topk", _I32), ("window", _I32), ("sm_scale", ctypes.c_float), ("n_kv", _I64),
                ("q", _P), ("kv_codes", _P), ("kv_scales", _P), ("idx", _P), ("swa", _P),
                ("n_swa", _I32), ("swa_pos0", _P), ("swa_start", _P), ("q_pos", _P),
                ("kv_fmt", ctypes.c_int), ("swa_fmt", ctypes.c_int), ("swa_scales", _P)]


class Csa2Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {status_string(status)} (status {status})")
        self.status = status


def library_path() -> str:
    return _build.LIB


class QuantJob(ctypes.Structure):
    """csa2_quant_job of include/csa2.h."""
    _fields_ = [("x", ctypes.c_void_p), ("xt", ctypes.c_int), ("rows", ctypes.c_int64),
                ("cols", ctypes.c_int64), ("ldx", ctypes.c_int64), ("codes", ctypes.c_void_p),
                ("ldc", ctypes.c_int64), ("scales", ctypes.c_void_p), ("lds", ctypes.c_int64)]


QUANT_MAX_JOBS = 4


class RopeQuantJob(ctypes.Structure):
    """csa2_rope_quant_job of include/csa2.h."""
    _fields_ = [("x", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("ldx", ctypes.c_int64), ("rope_dim", ctypes.c_int32), ("pos", ctypes.c_void_p),
                ("cos_sin", ctypes.c_void_p), ("n_pos", ctypes.c_int64), ("codes", ctypes.c_void_p),
                ("ldc", ctypes.c_int64), ("scales", ctypes.c_void_p), ("lds", ctypes.c_int64),
                ("fmt", ctypes.c_int)]


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libcsa2.so (building it in-tree first if it is absent or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if build_if_missing and not _build.up_to_date():
                _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"libcsa2.so not found at {path}; run fp4_kv_cache_gb300.build")
            lib = ctypes.CDLL(path)
            S = ctypes.c_int
            sz = ctypes.c_size_t
            lib.csa2_status_string.restype = ctypes.c_char_p
            lib.csa2_status_string.argtypes = [S]
            lib.csa2_version.restype = S
            lib.csa2_cache_bytes_per_position.restype = sz
            lib.csa2_cache_bytes_per_position.argtypes = [S, _I32, _I32]
            lib.csa2_quant_fp4.restype = S
            lib.csa2_quant_fp4.argtypes = [_P, S, _I64, _I64, _I64, _P, _I64, _P, _I64, S, _P, _P]
            lib.csa2_quant_fp4_batch.restype = S
            lib.csa2_quant_fp4_batch.argtypes = [ctypes.POINTER(QuantJob), _I32, S, _P, _P]
            lib.csa2_rope_quant_fp4.restype = S
            lib.csa2_rope_quant_fp4.argtypes = [ctypes.POINTER(RopeQuantJob), _I32, _P, _P]
            lib.csa2_quant_fp8.restype = S
            lib.csa2_quant_fp8.argtypes = [_P, S, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _P]
            lib.csa2_dequant_fp8.restype = S
            lib.csa2_dequant_fp8.argtypes = [_P, _I64, _P, _I64, _I64, _I64, _P, S, _I64, _P]
            lib.csa2_dequant_fp4.restype = S
            lib.csa2_dequant_fp4.argtypes = [_P, _I64, _P, _I64, _I64, _I64, S, _P, S, _I64, _P]
            lib.csa2_index_score_workspace_size.restype = sz
            lib.csa2_index_score_workspace_size.argtypes = [ctypes.POINTER(IndexArgs)]
            lib.csa2_index_score.restype = S
            lib.csa2_index_score.argtypes = [ctypes.POINTER(IndexArgs), _P, _P, _P, sz, _P, _P]
            IA = ctypes.POINTER(IndexArgs)
            lib.csa2_topk_workspace_size.restype = sz
            lib.csa2_topk_workspace_size.argtypes = [_I64, _I64, _I32, IA]
            lib.csa2_topk.restype = S
            lib.csa2_topk.argtypes = [_P, _I64, _I64, _P, _P, _P, _I32, IA, _I32, _P, _P, _P, sz, _P, _P]
            lib.csa2_index_topk_workspace_size.restype = sz
            lib.csa2_index_topk_workspace_size.argtypes = [ctypes.POINTER(IndexArgs), _I32]
            lib.csa2_index_topk.restype = S
            lib.csa2_index_topk.argtypes = [ctypes.POINTER(IndexArgs), _I32, _P, _P, _P, _P, sz, _P, _P]
            lib.csa2_block_candidates_workspace_size.restype = sz
            lib.csa2_block_candidates_workspace_size.argtypes = [_I64, _I64, _I32, _I32, IA]
            lib.csa2_block_candidates.restype = S
            lib.csa2_block_candidates.argtypes = [_P, _I64, _I64, _P, _I32, _I32, IA, _P, _P, sz, _P, _P]
            lib.csa2_sparse_attn_workspace_size.restype = sz
            lib.csa2_sparse_attn_workspace_size.argtypes = [ctypes.POINTER(AttnArgs)]
            lib.csa2_sparse_attn.restype = S
            lib.csa2_sparse_attn.argtypes = [ctypes.POINTER(AttnArgs), _P, _P, _P, sz, _P, _P]
            lib.csa2_selftest_bounded_wait.restype = S
            lib.csa2_selftest_bounded_wait.argtypes = [ctypes.c_uint32, _P, _P]
            lib.csa2_index_score_noalloc.restype = S
            lib.csa2_index_score_noalloc.argtypes = [ctypes.POINTER(IndexArgs), _P, _P, _P, _P]
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().csa2_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != OK:
        raise Csa2Error(fn, status)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libcsa2 takes device tensors (got a CPU tensor)")
    if not t.is_contiguous():
        raise ValueError("libcsa2 takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ws(nbytes: int, device, workspace: Optional[torch.Tensor], stream=None):
    """Caller workspace, or a torch allocation ordered on the call's stream (the caching
    allocator does not hand the block out again before that stream's work on it)."""
    if nbytes == 0:
        return None, 0
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes:
            raise ValueError("workspace too small")
        return _ptr(workspace), workspace.numel() * workspace.element_size()
    w = torch.zeros(nbytes, dtype=torch.uint8, device=device)     # workspaces start zeroed
    if stream is not None:
        w.record_stream(stream)
    return _ptr(w), nbytes


def _bits(t: torch.Tensor) -> torch.Tensor:
    """bf16 tensor viewed as its uint16 bit patterns (int16 storage)."""
    return t if t.dtype == torch.int16 else t.view(torch.int16)


# ------------------------------------------------------------------ C entry points
def cache_bytes_per_position(main_fmt: int, d_main: int, d_idx: int) -> int:
    return int(load().csa2_cache_bytes_per_position(main_fmt, d_main, d_idx))


def _rows_view(t: torch.Tensor):
    """(pointer, rows, row stride in elements) of a tensor whose last dim is contiguous:
    a contiguous N-D tensor (rows = all leading dims) or a row-strided 2-D view."""
    if not t.is_cuda:
        raise ValueError("libcsa2 takes device tensors (got a CPU tensor)")
    cols = t.shape[-1]
    if t.is_contiguous():
        return ctypes.c_void_p(t.data_ptr()), (t.numel() // cols if cols else 0), cols
    if t.dim() == 2 and t.stride(1) == 1:
        return ctypes.c_void_p(t.data_ptr()), t.shape[0], t.stride(0)
    raise ValueError("expected a contiguous tensor or a 2-D view with contiguous rows")


def csa2_quant_fp4(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor,
                   d_status: Optional[torch.Tensor] = None, stream=None, fmt: int = FMT_MXFP4):
    cols = x.shape[-1]
    xt = BF16 if x.dtype == torch.bfloat16 else F32 if x.dtype == torch.float32 else None
    if xt is None:
        raise ValueError("x must be bf16 or f32")
    px, rows, ldx = _rows_view(x)
    pc, rows_c, ldc = _rows_view(codes)
    ps, rows_s, lds = _rows_view(scales)
    if rows_c != rows or rows_s != rows:
        raise ValueError("x, codes and scales must have the same number of rows")
    _check("csa2_quant_fp4", load().csa2_quant_fp4(
        px, xt, rows, cols, ldx, pc, ldc, ps, lds, fmt, _ptr(d_status), _stream(stream)))


def csa2_quant_fp8(x: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor,
                   d_status: Optional[torch.Tensor] = None, stream=None):
    """MXFP8 (E4M3 + E8M0 per 32) rows: the SWA cache codec (csa2_quant_fp8)."""
    cols = x.shape[-1]
    xt = BF16 if x.dtype == torch.bfloat16 else F32 if x.dtype == torch.float32 else None
    if xt is None:
        raise ValueError("x must be bf16 or f32")
    px, rows, ldx = _rows_view(x)
    pc, rows_c, ldc = _rows_view(codes)
    ps, rows_s, lds = _rows_view(scales)
    if rows_c != rows or rows_s != rows:
        raise ValueError("x, codes and scales must have the same number of rows")
    _check("csa2_quant_fp8", load().csa2_quant_fp8(px, xt, rows, cols, ldx, pc, ldc, ps, lds,
                                                   _ptr(d_status), _stream(stream)))


def quant_fp8(x: torch.Tensor, d_status=None, stream=None):
    """x [..., D] bf16/f32 -> (codes uint8 [..., D], scales uint8 [..., D/32]) in MXFP8."""
    D = x.shape[-1]
    codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    scales = torch.empty(x.shape[:-1] + (D // 32,), dtype=torch.uint8, device=x.device)
    csa2_quant_fp8(x, codes, scales, d_status, stream)
    return codes, scales


def dequant_fp8(codes, scales, dtype=torch.float32, stream=None):
    cols = codes.shape[-1]
    rows = codes.numel() // cols if cols else 0
    y = torch.empty(codes.shape, dtype=dtype, device=codes.device)
    _check("csa2_dequant_fp8", load().csa2_dequant_fp8(
        _ptr(codes), cols, _ptr(scales), cols // 32, rows, cols, _ptr(y),
        BF16 if dtype == torch.bfloat16 else F32, cols, _stream(stream)))
    return y


def quant_jobs(triples) -> ctypes.Array:
    """(x, codes, scales) tensor triples -> a csa2_quant_job array (keep it alive while used)."""
    jobs = (QuantJob * max(1, len(triples)))()
    for i, (x, codes, scales) in enumerate(triples):
        xt = BF16 if x.dtype == torch.bfloat16 else F32 if x.dtype == torch.float32 else None
        if xt is None:
            raise ValueError("x must be bf16 or f32")
        px, rows, ldx = _rows_view(x)
        pc, rows_c, ldc = _rows_view(codes)
        ps, rows_s, lds = _rows_view(scales)
        if rows_c != rows or rows_s != rows:
            raise ValueError("x, codes and scales must have the same number of rows")
        jobs[i] = QuantJob(px.value, xt, rows, x.shape[-1], ldx, pc.value, ldc, ps.value, lds)
    return jobs


def csa2_quant_fp4_batch(triples, d_status: Optional[torch.Tensor] = None, stream=None,
                         fmt: int = FMT_MXFP4, jobs=None):
    """Quantise several (x, codes, scales) triples in one launch (csa2_quant_fp4_batch)."""
    if jobs is None:
        jobs = quant_jobs(triples)
    _check("csa2_quant_fp4_batch", load().csa2_quant_fp4_batch(
        jobs, len(triples), fmt, _ptr(d_status), _stream(stream)))


def rope_quant_jobs(specs) -> ctypes.Array:
    """(x bf16 [rows, cols], codes, scales, rope_dim, pos int32 [rows] or None, cos_sin f32
    [n_pos, rope_dim] or None, fmt) tuples -> a csa2_rope_quant_job array (keep it alive)."""
    jobs = (RopeQuantJob * max(1, len(specs)))()
    for i, (x, codes, scales, rope_dim, pos, cos_sin, fmt) in enumerate(specs):
        if x.dtype != torch.bfloat16:
            raise ValueError("x must be bf16")
        px, rows, ldx = _rows_view(x)
        pc, rows_c, ldc = _rows_view(codes)
        ps, rows_s, lds = _rows_view(scales)
        if rows_c != rows or rows_s != rows:
            raise ValueError("x, codes and scales must have the same number of rows")
        jobs[i] = RopeQuantJob(px.value, rows, x.shape[-1], ldx, rope_dim,
                               pos.data_ptr() if pos is not None else None,
                               cos_sin.data_ptr() if cos_sin is not None else None,
                               cos_sin.shape[0] if cos_sin is not None else 0,
                               pc.value, ldc, ps.value, lds, fmt)
    return jobs


def csa2_rope_quant_fp4(specs, d_status: Optional[torch.Tensor] = None, stream=None, jobs=None):
    """RoPE on the trailing rope_dim channels, then the 4-bit codec, for up to four jobs
    in one launch (csa2_rope_quant_fp4); specs as for rope_quant_jobs."""
    if jobs is None:
        jobs = rope_quant_jobs(specs)
    _check("csa2_rope_quant_fp4", load().csa2_rope_quant_fp4(jobs, len(specs), _ptr(d_status),
                                                             _stream(stream)))


def csa2_dequant_fp4(codes: torch.Tensor, scales: torch.Tensor, y: torch.Tensor, stream=None,
                     fmt: int = FMT_MXFP4):
    cols = codes.shape[-1] * 2
    rows = codes.numel() // (cols // 2) if cols else 0
    yt = BF16 if y.dtype == torch.bfloat16 else F32
    _check("csa2_dequant_fp4", load().csa2_dequant_fp4(
        _ptr(codes), cols // 2, _ptr(scales), cols // FMT_BLOCK[fmt], rows, cols, fmt, _ptr(y), yt,
        cols, _stream(stream)))


def scales_format(cols: int, scales: torch.Tensor) -> int:
    """Format of rows of `cols` values whose scales tensor is `scales` (one scale per 16
    values: E2M1 + E4M3/16, per 32: MXFP4)."""
    return FMT_NVFP4_E4M3_16 if scales.shape[-1] * 16 == cols else FMT_MXFP4


def make_index_args(q, w, k_codes, k_scales, q_pos=None, ratio_m=1, pool_blocks=None, block=8,
                    group_max=None):
    B, T, H, d = q.shape
    a = IndexArgs()
    a.batch, a.n_q, a.n_heads, a.head_dim, a.ratio_m = B, T, H, d, ratio_m
    a.n_keys = k_codes.shape[1]
    a.q, a.w = _ptr(_bits(q)), _ptr(w)
    a.k_codes, a.k_scales = _ptr(k_codes), _ptr(k_scales)
    a.q_pos = _ptr(q_pos)
    if pool_blocks is None:
        a.mode, a.pool_blocks, a.n_pool_blocks = INDEX_FULL, None, 0
    else:
        a.mode, a.pool_blocks, a.n_pool_blocks = INDEX_POOL, _ptr(pool_blocks), pool_blocks.shape[-1]
    a.block = block
    a.group_max = _ptr(group_max)
    return a


def csa2_index_score(args: IndexArgs, scores: torch.Tensor, row_len: torch.Tensor,
                     d_status=None, stream=None, workspace=None):
    lib = load()
    need = lib.csa2_index_score_workspace_size(ctypes.byref(args))
    ws, wsb = _ws(need, scores.device, workspace, stream)
    _check("csa2_index_score", lib.csa2_index_score(ctypes.byref(args), _ptr(scores),
                                                    _ptr(row_len), ws, wsb, _ptr(d_status),
                                                    _stream(stream)))


def csa2_index_score_noalloc(args: IndexArgs, scores: torch.Tensor, row_len: torch.Tensor,
                             d_status=None, stream=None):
    """csa2_index_score without a workspace: scratch comes from the library's own static
    device array (for callers that cannot allocate; see include/csa2.h)."""
    _check("csa2_index_score_noalloc", load().csa2_index_score_noalloc(
        ctypes.byref(args), _ptr(scores), _ptr(row_len), _ptr(d_status), _stream(stream)))


def csa2_selftest_bounded_wait(polls: int, d_status: torch.Tensor, stream=None):
    """One CTA waits `polls` polls on an mbarrier nothing completes; *d_status must then
    hold DEV_TIMEOUT (the bounded-wait check of include/csa2.h)."""
    _check("csa2_selftest_bounded_wait", load().csa2_selftest_bounded_wait(polls, _ptr(d_status),
                                                                           _stream(stream)))


def _exact_ref(exact: Optional[IndexArgs]):
    return ctypes.byref(exact) if exact is not None else None


def csa2_topk(scores: torch.Tensor, k: int, idx: torch.Tensor, row_len=None, pool_blocks=None,
              block: int = 8, out_scores=None, d_status=None, stream=None, workspace=None,
              group_max=None, exact: Optional[IndexArgs] = None):
    """exact: the IndexArgs of the csa2_index_score call that wrote `scores` (rank by the
    exact score) or None (rank the given floats)."""
    lib = load()
    n = scores.shape[-1]
    rows = scores.numel() // n if n else idx.numel() // max(k, 1)
    need = lib.csa2_topk_workspace_size(rows, n, k, _exact_ref(exact))
    ws, wsb = _ws(need, idx.device, workspace, stream)
    _check("csa2_topk", lib.csa2_topk(_ptr(scores), rows, n, _ptr(row_len), _ptr(group_max),
                                      _ptr(pool_blocks), block, _exact_ref(exact), k, _ptr(idx),
                                      _ptr(out_scores), ws, wsb, _ptr(d_status), _stream(stream)))


def csa2_index_topk(args: IndexArgs, k: int, idx: torch.Tensor, out_scores=None, row_len=None,
                    d_status=None, stream=None, workspace=None):
    """The indexer and the exact Top-K in one call (no score matrix on the decode path)."""
    lib = load()
    need = lib.csa2_index_topk_workspace_size(ctypes.byref(args), k)
    ws, wsb = _ws(need, idx.device, workspace, stream)
    _check("csa2_index_topk", lib.csa2_index_topk(ctypes.byref(args), k, _ptr(idx), _ptr(out_scores),
                                                  _ptr(row_len), ws, wsb, _ptr(d_status), _stream(stream)))


def csa2_block_candidates(scores: torch.Tensor, nb: int, block_ids: torch.Tensor, row_len=None,
                          block: int = 8, d_status=None, stream=None, workspace=None,
                          exact: Optional[IndexArgs] = None):
    lib = load()
    n = scores.shape[-1]
    rows = scores.numel() // n if n else block_ids.numel() // max(nb, 1)
    need = lib.csa2_block_candidates_workspace_size(rows, n, block, nb, _exact_ref(exact))
    ws, wsb = _ws(need, block_ids.device, workspace, stream)
    _check("csa2_block_candidates", lib.csa2_block_candidates(
        _ptr(scores), rows, n, _ptr(row_len), block, nb, _exact_ref(exact), _ptr(block_ids), ws, wsb,
        _ptr(d_status), _stream(stream)))


def make_attn_args(q, kv_codes, kv_scales, idx, swa=None, swa_pos0=None, q_pos=None,
                   swa_start=None, window=128, sm_scale=None, d_v=None, swa_scales=None):
    """csa2_attn_args; the main-KV format follows from the width of kv_scales; the SWA is
    bf16, or MXFP8 when swa holds uint8 codes and swa_scales their scales."""
    B, T, H, dqk = q.shape
    a = AttnArgs()
    a.kv_fmt = scales_format(dqk, kv_scales)
    a.batch, a.n_q, a.n_heads, a.d_qk = B, T, H, dqk
    a.d_v = d_v if d_v is not None else dqk
    a.topk = idx.shape[-1] if idx is not None else 0
    a.window = window
    a.sm_scale = (1.0 / math.sqrt(dqk)) if sm_scale is None else sm_scale
    a.n_kv = kv_codes.shape[1]
    a.q, a.kv_codes, a.kv_scales, a.idx = _ptr(_bits(q)), _ptr(kv_codes), _ptr(kv_scales), _ptr(idx)
    if swa is not None and swa.dtype == torch.uint8:
        if swa_scales is None:
            raise ValueError("MXFP8 SWA codes need swa_scales")
        a.swa, a.swa_fmt, a.swa_scales = _ptr(swa), SWA_MXFP8, _ptr(swa_scales)
    else:
        a.swa = _ptr(_bits(swa)) if swa is not None else None
        a.swa_fmt, a.swa_scales = SWA_BF16, None
    a.n_swa = swa.shape[1] if swa is not None else 0
    a.swa_pos0, a.swa_start, a.q_pos = _ptr(swa_pos0), _ptr(swa_start), _ptr(q_pos)
    return a


def csa2_sparse_attn(args: AttnArgs, out: torch.Tensor, lse=None, d_status=None, stream=None,
                     workspace=None):
    lib = load()
    need = lib.csa2_sparse_attn_workspace_size(ctypes.byref(args))
    ws, wsb = _ws(need, out.device, workspace, stream)
    _check("csa2_sparse_attn", lib.csa2_sparse_attn(ctypes.byref(args), _ptr(_bits(out)),
                                                    _ptr(lse), ws, wsb, _ptr(d_status),
                                                    _stream(stream)))


# ------------------------------------------------------------------ allocating helpers
def quant_fp4(x: torch.Tensor, d_status=None, stream=None, fmt: int = FMT_MXFP4):
    """x [..., D] bf16/f32 -> (codes uint8 [..., D/2], scales uint8 [..., D/G]), G = 32
    (MXFP4) or 16 (E2M1 + E4M3/16)."""
    D = x.shape[-1]
    codes = torch.empty(x.shape[:-1] + (D // 2,), dtype=torch.uint8, device=x.device)
    scales = torch.empty(x.shape[:-1] + (D // FMT_BLOCK[fmt],), dtype=torch.uint8, device=x.device)
    csa2_quant_fp4(x, codes, scales, d_status, stream, fmt=fmt)
    return codes, scales


def dequant_fp4(codes, scales, dtype=torch.float32, stream=None):
    """Dequantise MXFP4 or E2M1 + E4M3/16 rows (told apart by the width of scales)."""
    cols = codes.shape[-1] * 2
    y = torch.empty(codes.shape[:-1] + (cols,), dtype=dtype, device=codes.device)
    csa2_dequant_fp4(codes, scales, y, stream, fmt=scales_format(cols, scales))
    return y


def group_max_buffer(scores: torch.Tensor) -> torch.Tensor:
    """Buffer for the indexer's per-32-candidate group maxima of `scores` (32-bit keys)."""
    return torch.empty(scores.shape[:-1] + ((scores.shape[-1] + 31) // 32,), dtype=torch.int32,
                       device=scores.device)


def index_score(q, w, k_codes, k_scales, q_pos=None, ratio_m=1, pool_blocks=None, block=8,
                d_status=None, stream=None, group_max=None, want_args=False):
    """-> (scores f32 [B, T, n_cand], row_len int32 [B, T]) and, with want_args, the
    IndexArgs used (pass them as `exact` to topk / block_candidates to rank by the exact
    score; they point into q, w and the caches, which must stay alive).  group_max:
    optional buffer from group_max_buffer(scores) that receives the group maxima."""
    B, T = q.shape[:2]
    n_cand = k_codes.shape[1] if pool_blocks is None else pool_blocks.shape[-1] * block
    scores = torch.empty((B, T, n_cand), dtype=torch.float32, device=q.device)
    row_len = torch.empty((B, T), dtype=torch.int32, device=q.device)
    args = make_index_args(q, w, k_codes, k_scales, q_pos, ratio_m, pool_blocks, block, group_max)
    csa2_index_score(args, scores, row_len, d_status, stream)
    return (scores, row_len, args) if want_args else (scores, row_len)


def topk(scores, k=512, row_len=None, pool_blocks=None, block=8, want_scores=False,
         d_status=None, stream=None, group_max=None, exact=None):
    shape = scores.shape[:-1]
    idx = torch.empty(shape + (k,), dtype=torch.int32, device=scores.device)
    out_s = torch.empty(shape + (k,), dtype=torch.float32, device=scores.device) if want_scores else None
    csa2_topk(scores, k, idx, row_len, pool_blocks, block, out_s, d_status, stream,
              group_max=group_max, exact=exact)
    return (idx, out_s) if want_scores else idx


def index_topk(q, w, k_codes, k_scales, k=512, q_pos=None, ratio_m=1, pool_blocks=None, block=8,
               d_status=None, stream=None, want_scores=False):
    """-> (idx int32 [B, T, k], row_len int32 [B, T]) [+ their float32 scores]: the exact
    Top-K of the indexer scores from one csa2_index_topk call."""
    B, T = q.shape[:2]
    idx = torch.empty((B, T, k), dtype=torch.int32, device=q.device)
    row_len = torch.empty((B, T), dtype=torch.int32, device=q.device)
    out_s = torch.empty((B, T, k), dtype=torch.float32, device=q.device) if want_scores else None
    args = make_index_args(q, w, k_codes, k_scales, q_pos, ratio_m, pool_blocks, block)
    csa2_index_topk(args, k, idx, out_s, row_len, d_status, stream)
    return (idx, row_len, out_s) if want_scores else (idx, row_len)


def block_candidates(scores, nb=2048, row_len=None, block=8, d_status=None, stream=None, exact=None):
    ids = torch.empty(scores.shape[:-1] + (nb,), dtype=torch.int32, device=scores.device)
    csa2_block_candidates(scores, nb, ids, row_len, block, d_status, stream, exact=exact)
    return ids


def sparse_attn(q, kv_codes, kv_scales, idx, swa=None, swa_pos0=None, q_pos=None, swa_start=None,
                window=128, sm_scale=None, d_v=None, want_lse=True, d_status=None, stream=None,
                swa_scales=None):
    """-> (out bf16 [B, T, H, d_v], lse f32 [B, T, H] or None)."""
    args = make_attn_args(q, kv_codes, kv_scales, idx, swa, swa_pos0, q_pos, swa_start, window,
                          sm_scale, d_v, swa_scales)
    B, T, H = q.shape[:3]
    out = torch.empty((B, T, H, args.d_v), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, T, H), dtype=torch.float32, device=q.device) if want_lse else None
    csa2_sparse_attn(args, out, lse, d_status, stream)
    return out, lse
