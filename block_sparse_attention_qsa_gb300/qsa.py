"""Python binding of libqsa.so (ctypes).

Argument marshalling only: every step of the QSA decode / MTP-verify path runs
in the library's CUDA kernels. Tensors are torch CUDA tensors used as device
memory; the stream is torch's current stream unless one is given. Shapes and
dtypes are checked here because the C ABI receives bare pointers.

Importing this module loads the library and raises ImportError if it is
missing or was built for another ABI: there is no CPU fallback. The
environment variable QSA_LIBRARY names another build to load instead (the
tracing build, libqsa_trace.so, for timeline.py).
"""

from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("QSA_LIBRARY") or os.path.join(_HERE, "libqsa.so")
ABI_VERSION = 1

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_BAD_INDEX, ERR_TIMEOUT, ERR_CUDA = range(7)
KV_BF16, KV_FP8_E4M3 = 0, 1

BLOCK, TOPK, WIDTH = 4, 512, 2051

# every symbol the C ABI exports (include/qsa.h)
EXPORTS = (
    "qsa_abi_version", "qsa_status_str", "qsa_dims_default", "qsa_workspace_size",
    "qsa_workspace_init", "qsa_compress_keys", "qsa_score", "qsa_topk", "qsa_sparse_attn",
    "qsa_decode", "qsa_check_errors", "qsa_sparse_attn_noalloc", "qsa_draft_attn",
    "qsa_compress_keys_paged", "qsa_score_paged", "qsa_decode_paged", "qsa_score_chunk",
    "qsa_resolve", "qsa_sparse_attn_rows", "qsa_test_chunk_timeout", "qsa_trace_read",
)
TRACE_SCORE, TRACE_TOPK, TRACE_ATTN = 0, 1, 2  # qsa_trace_read tables
TRACE_SLOTS, TRACE_CTAS = 8, 4096

MAX_DRAFT_GAP = 64  # QSA_MAX_DRAFT_GAP
MAX_CHUNK = 65536  # QSA_MAX_CHUNK
MAX_SCORE_BATCH = 16384  # QSA_MAX_SCORE_BATCH


class QSAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_str(status)}")


class Dims(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("n_q", ctypes.c_int32), ("n_idx_heads", ctypes.c_int32),
        ("idx_dim", ctypes.c_int32), ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32), ("max_blocks", ctypes.c_int32),
        ("max_pages", ctypes.c_int32), ("num_pages", ctypes.c_int32), ("topk", ctypes.c_int32),
        ("block", ctypes.c_int32), ("width", ctypes.c_int32), ("sm_scale", ctypes.c_float),
        ("kv_dtype", ctypes.c_int32),
    ]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libqsa.so is not built ({LIB_PATH}); run __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    D = ctypes.POINTER(Dims)
    sig = {
        "qsa_abi_version": (ctypes.c_int32, []),
        "qsa_status_str": (ctypes.c_char_p, [I]),
        "qsa_dims_default": (None, [D]),
        "qsa_workspace_size": (I, [D, ctypes.POINTER(SZ)]),
        "qsa_workspace_init": (I, [P, SZ, P]),
        "qsa_compress_keys": (I, [D, P, P, P, P, P, SZ, P]),
        "qsa_score": (I, [D, P, P, P, P, P, SZ, P]),
        "qsa_topk": (I, [D, P, P, P, P, P, SZ, P]),
        "qsa_sparse_attn": (I, [D, P, P, P, P, P, P, P, P, P, P, SZ, P]),
        "qsa_decode": (I, [D, P, P, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P]),
        "qsa_check_errors": (I, [P, P, ctypes.POINTER(ctypes.c_int32)]),
        "qsa_sparse_attn_noalloc": (I, [D, P, P, P, P, P, P, P, P, P, P]),
        "qsa_draft_attn": (I, [D, P, P, P, P, P, P, P, P, ctypes.c_int32, P, P, P, P, SZ, P]),
        "qsa_compress_keys_paged": (I, [D, P, P, P, P, P, P, SZ, P]),
        "qsa_score_paged": (I, [D, P, P, P, P, P, P, SZ, P]),
        "qsa_decode_paged": (I, [D, P, P, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P]),
        "qsa_score_chunk": (I, [D, ctypes.c_int32, P, P, P, P, P, SZ, P]),
        "qsa_test_chunk_timeout": (I, [D, ctypes.c_int32, P, P, P, P, P, SZ, P]),
        "qsa_resolve": (I, [D, P, P, P, P, P, SZ, P]),
        "qsa_sparse_attn_rows": (I, [D, P, P, P, P, P, P, P, P, SZ, P]),
        "qsa_trace_read": (I, [ctypes.c_int32, P, ctypes.c_int32, ctypes.c_int32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if lib.qsa_abi_version() != ABI_VERSION:
        raise ImportError(f"libqsa.so ABI {lib.qsa_abi_version()} != {ABI_VERSION}; rebuild it")
    return lib


lib = _load()


def status_str(status: int) -> str:
    return lib.qsa_status_str(status).decode()


def _check(status: int, where: str):
    if status != OK:
        raise QSAError(status, where)


def make_dims(batch: int, n_q: int, max_blocks: int, max_pages: int, num_pages: int,
              n_idx_heads: int = 1, kv_dtype: str = "bf16", page_size: int = 64,
              n_q_heads: int = 16, n_kv_heads: int = 2, head_dim: int = 128,
              sm_scale: float = 0.0) -> Dims:
    d = Dims()
    lib.qsa_dims_default(ctypes.byref(d))
    d.batch, d.n_q, d.max_blocks, d.max_pages, d.num_pages = batch, n_q, max_blocks, max_pages, num_pages
    d.n_idx_heads, d.page_size = n_idx_heads, page_size
    d.n_q_heads, d.n_kv_heads, d.head_dim, d.idx_dim = n_q_heads, n_kv_heads, head_dim, head_dim
    d.kv_dtype = {"bf16": KV_BF16, "fp8": KV_FP8_E4M3}[kv_dtype]
    d.sm_scale = sm_scale
    return d


def dims_for_spec(spec) -> Dims:
    """Dims of a ``synth.Spec`` workload."""
    return make_dims(spec.batch, spec.n_q, spec.max_blocks(), spec.max_pages(), spec.num_pages(),
                     spec.n_idx_heads, spec.kv_dtype, spec.page_size, spec.n_q_heads,
                     spec.n_kv_heads, spec.head_dim)


def workspace_size(d: Dims) -> int:
    n = ctypes.c_size_t(0)
    _check(lib.qsa_workspace_size(ctypes.byref(d), ctypes.byref(n)), "qsa_workspace_size")
    return n.value


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def make_workspace(d: Dims, device="cuda", stream=None) -> torch.Tensor:
    """Allocate and zero a workspace for ``d`` (torch owns the memory)."""
    n = workspace_size(d)
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    assert ws.data_ptr() % 256 == 0
    _check(lib.qsa_workspace_init(ctypes.c_void_p(ws.data_ptr()), n, _stream(stream)), "qsa_workspace_init")
    return ws


def _ptr(t: Optional[torch.Tensor]) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _want(t: torch.Tensor, name: str, shape, dtype):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the QSA path has no CPU implementation)")
    if t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _kv_dtype(d: Dims):
    return torch.uint8 if d.kv_dtype == KV_FP8_E4M3 else torch.bfloat16


def _ws(d: Dims, ws: torch.Tensor):
    if ws.numel() < workspace_size(d):
        raise ValueError("workspace too small for these dims")
    return ctypes.c_void_p(ws.data_ptr()), ws.numel()


def compress_keys(d: Dims, idx_keys, q_pos, kc, ws, block_lo=None, stream=None):
    _want(idx_keys, "idx_keys", (d.batch, BLOCK * d.max_blocks, d.n_idx_heads, d.idx_dim), torch.bfloat16)
    _want(q_pos, "q_pos", (d.batch, d.n_q), torch.int32)
    _want(kc, "kc", (d.batch, d.max_blocks, d.n_idx_heads, d.idx_dim), torch.bfloat16)
    if block_lo is not None:
        _want(block_lo, "block_lo", (d.batch,), torch.int32)
    w, n = _ws(d, ws)
    _check(lib.qsa_compress_keys(ctypes.byref(d), _ptr(idx_keys), _ptr(q_pos), _ptr(block_lo), _ptr(kc),
                                 w, n, _stream(stream)), "qsa_compress_keys")


def score(d: Dims, q_idx, kc, q_pos, scores, ws, stream=None):
    _want(q_idx, "q_idx", (d.batch, d.n_q, d.n_idx_heads, d.idx_dim), torch.bfloat16)
    _want(kc, "kc", (d.batch, d.max_blocks, d.n_idx_heads, d.idx_dim), torch.bfloat16)
    _want(q_pos, "q_pos", (d.batch, d.n_q), torch.int32)
    _want(scores, "scores", (d.batch, d.n_q, d.max_blocks), torch.float32)
    w, n = _ws(d, ws)
    _check(lib.qsa_score(ctypes.byref(d), _ptr(q_idx), _ptr(kc), _ptr(q_pos), _ptr(scores), w, n,
                         _stream(stream)), "qsa_score")


def topk(d: Dims, scores, q_pos, sel_blk, sel_pos, ws, stream=None):
    _want(scores, "scores", (d.batch, d.n_q, d.max_blocks), torch.float32)
    _want(q_pos, "q_pos", (d.batch, d.n_q), torch.int32)
    _want(sel_blk, "sel_blk", (d.batch, d.n_q, d.topk), torch.int32)
    _want(sel_pos, "sel_pos", (d.batch, d.n_q, d.width), torch.int32)
    w, n = _ws(d, ws)
    _check(lib.qsa_topk(ctypes.byref(d), _ptr(scores), _ptr(q_pos), _ptr(sel_blk), _ptr(sel_pos), w, n,
                        _stream(stream)), "qsa_topk")


def _check_attn_inputs(d: Dims, q, k_cache, v_cache, k_scale, v_scale, page_table, q_pos, out):
    _want(q, "q", (d.batch, d.n_q, d.n_q_heads, d.head_dim), torch.bfloat16)
    kv_shape = (d.num_pages, d.n_kv_heads, d.page_size, d.head_dim)
    _want(k_cache, "k_cache", kv_shape, _kv_dtype(d))
    _want(v_cache, "v_cache", kv_shape, _kv_dtype(d))
    if d.kv_dtype == KV_FP8_E4M3 or k_scale is not None:
        _want(k_scale, "k_scale", (d.n_kv_heads,), torch.float32)
        _want(v_scale, "v_scale", (d.n_kv_heads,), torch.float32)
    _want(page_table, "page_table", (d.batch, d.max_pages), torch.int32)
    _want(q_pos, "q_pos", (d.batch, d.n_q), torch.int32)
    _want(out, "out", (d.batch, d.n_q, d.n_q_heads, d.head_dim), torch.bfloat16)


def sparse_attn(d: Dims, q, k_cache, v_cache, k_scale, v_scale, page_table, sel_pos, q_pos, out, ws,
                stream=None):
    _check_attn_inputs(d, q, k_cache, v_cache, k_scale, v_scale, page_table, q_pos, out)
    _want(sel_pos, "sel_pos", (d.batch, d.n_q, d.width), torch.int32)
    w, n = _ws(d, ws)
    _check(lib.qsa_sparse_attn(ctypes.byref(d), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                               _ptr(v_scale), _ptr(page_table), _ptr(sel_pos), _ptr(q_pos), _ptr(out), w, n,
                               _stream(stream)), "qsa_sparse_attn")


def resolve(d: Dims, sel_pos, q_pos, page_table, sel_row, ws, stream=None):
    """Selected positions -> cache rows of KV head 0 (-1 for none or rejected)."""
    _want(sel_pos, "sel_pos", (d.batch, d.n_q, d.width), torch.int32)
    _want(q_pos, "q_pos", (d.batch, d.n_q), torch.int32)
    _want(page_table, "page_table", (d.batch, d.max_pages), torch.int32)
    _want(sel_row, "sel_row", (d.batch, d.n_q, d.width), torch.int32)
    w, n = _ws(d, ws)
    _check(lib.qsa_resolve(ctypes.byref(d), _ptr(sel_pos), _ptr(q_pos), _ptr(page_table), _ptr(sel_row), w, n,
                           _stream(stream)), "qsa_resolve")


def sparse_attn_rows(d: Dims, q, k_cache, v_cache, k_scale, v_scale, sel_row, out, ws, stream=None):
    """sparse_attn over cache rows written by resolve."""
    _want(q, "q", (d.batch, d.n_q, d.n_q_heads, d.head_dim), torch.bfloat16)
    kv_shape = (d.num_pages, d.n_kv_heads, d.page_size, d.head_dim)
    _want(k_cache, "k_cache", kv_shape, _kv_dtype(d))
    _want(v_cache, "v_cache", kv_shape, _kv_dtype(d))
    if d.kv_dtype == KV_FP8_E4M3 or k_scale is not None:
        _want(k_scale, "k_scale", (d.n_kv_heads,), torch.float32)
        _want(v_scale, "v_scale", (d.n_kv_heads,), torch.float32)
    _want(sel_row, "sel_row", (d.batch, d.n_q, d.width), torch.int32)
    _want(out, "out", (d.batch, d.n_q, d.n_q_heads, d.head_dim), torch.bfloat16)
    w, n = _ws(d, ws)
    _check(lib.qsa_sparse_attn_rows(ctypes.byref(d), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                    _ptr(v_scale), _ptr(sel_row), _ptr(out), w, n, _stream(stream)),
           "qsa_sparse_attn_rows")


def sparse_attn_noalloc(d: Dims, q, k_cache, v_cache, k_scale, v_scale, page_table, sel_pos, q_pos, out,
                        stream=None):
    """sparse_attn without a workspace, for callers that cannot allocate
    device memory: the library's own static device scratch is used instead.
    Calls that overlap on the GPU race on that scratch; keep them on one
    stream."""
    _check_attn_inputs(d, q, k_cache, v_cache, k_scale, v_scale, page_table, q_pos, out)
    _want(sel_pos, "sel_pos", (d.batch, d.n_q, d.width), torch.int32)
    _check(lib.qsa_sparse_attn_noalloc(ctypes.byref(d), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                       _ptr(v_scale), _ptr(page_table), _ptr(sel_pos), _ptr(q_pos), _ptr(out),
                                       _stream(stream)), "qsa_sparse_attn_noalloc")


def score_chunk(d: Dims, q_idx, kc, q_pos, scores, ws, stream=None):
    """Scores of a chunk of many queries per request (q_idx [B][n_chunk][H][128],
    q_pos [B][n_chunk], scores [B][n_chunk][max_blocks])."""
    if q_idx.dim() != 4:
        raise ValueError("q_idx must be [B][n_chunk][H][128]")
    n_chunk = int(q_idx.shape[1])
    _want(q_idx, "q_idx", (d.batch, n_chunk, d.n_idx_heads, d.idx_dim), torch.bfloat16)
    _want(kc, "kc", (d.batch, d.max_blocks, d.n_idx_heads, d.idx_dim), torch.bfloat16)
    _want(q_pos, "q_pos", (d.batch, n_chunk), torch.int32)
    _want(scores, "scores", (d.batch, n_chunk, d.max_blocks), torch.float32)
    w, n = _ws(d, ws)
    _check(lib.qsa_score_chunk(ctypes.byref(d), n_chunk, _ptr(q_idx), _ptr(kc), _ptr(q_pos), _ptr(scores), w, n,
                               _stream(stream)), "qsa_score_chunk")


def test_chunk_timeout(d: Dims, q_idx, kc, q_pos, scores, ws, stream=None):
    """qsa_test_chunk_timeout: score_chunk with one copy withheld, so that one
    CTA's bounded wait runs out (about a second); check_errors then reports
    ERR_TIMEOUT. For failure-detection tests."""
    n_chunk = int(q_idx.shape[1])
    _want(q_idx, "q_idx", (d.batch, n_chunk, d.n_idx_heads, d.idx_dim), torch.bfloat16)
    _want(kc, "kc", (d.batch, d.max_blocks, d.n_idx_heads, d.idx_dim), torch.bfloat16)
    _want(q_pos, "q_pos", (d.batch, n_chunk), torch.int32)
    _want(scores, "scores", (d.batch, n_chunk, d.max_blocks), torch.float32)
    w, n = _ws(d, ws)
    _check(lib.qsa_test_chunk_timeout(ctypes.byref(d), n_chunk, _ptr(q_idx), _ptr(kc), _ptr(q_pos), _ptr(scores), w,
                                      n, _stream(stream)), "qsa_test_chunk_timeout")


def trace_read(kernel: int, n_ctas: int = TRACE_CTAS, clear: bool = False):
    """qsa_trace_read: the per-CTA phase stamps of a kernel's latest launch
    as a numpy uint64 array [n_ctas][TRACE_SLOTS] (tracing build only; the
    product build raises QSAError with ERR_UNSUPPORTED). clear zeroes the
    table afterwards; n_ctas 0 only clears."""
    buf = np.zeros((n_ctas, TRACE_SLOTS), dtype=np.uint64)
    _check(lib.qsa_trace_read(kernel, buf.ctypes.data if n_ctas else None, n_ctas, int(clear)), "qsa_trace_read")
    return buf


def _want_kc_cache(d: Dims, kc_cache):
    _want(kc_cache, "kc_cache", (d.num_pages, d.page_size // d.block, d.n_idx_heads, d.idx_dim), torch.bfloat16)


def compress_keys_paged(d: Dims, idx_keys, q_pos, page_table, kc_cache, ws, block_lo=None, stream=None):
    """compress_keys into the paged layout [num_pages][page_size / 4][H_idx][128]."""
    _want(idx_keys, "idx_keys", (d.batch, d.block * d.max_blocks, d.n_idx_heads, d.idx_dim), torch.bfloat16)
    _want(q_pos, "q_pos", (d.batch, d.n_q), torch.int32)
    _want(page_table, "page_table", (d.batch, d.max_pages), torch.int32)
    _want_kc_cache(d, kc_cache)
    if block_lo is not None:
        _want(block_lo, "block_lo", (d.batch,), torch.int32)
    w, n = _ws(d, ws)
    _check(lib.qsa_compress_keys_paged(ctypes.byref(d), _ptr(idx_keys), _ptr(q_pos), _ptr(block_lo),
                                       _ptr(page_table), _ptr(kc_cache), w, n, _stream(stream)),
           "qsa_compress_keys_paged")


def score_paged(d: Dims, q_idx, kc_cache, page_table, q_pos, scores, ws, stream=None):
    _want(q_idx, "q_idx", (d.batch, d.n_q, d.n_idx_heads, d.idx_dim), torch.bfloat16)
    _want_kc_cache(d, kc_cache)
    _want(page_table, "page_table", (d.batch, d.max_pages), torch.int32)
    _want(q_pos, "q_pos", (d.batch, d.n_q), torch.int32)
    _want(scores, "scores", (d.batch, d.n_q, d.max_blocks), torch.float32)
    w, n = _ws(d, ws)
    _check(lib.qsa_score_paged(ctypes.byref(d), _ptr(q_idx), _ptr(kc_cache), _ptr(page_table), _ptr(q_pos),
                               _ptr(scores), w, n, _stream(stream)), "qsa_score_paged")


def decode_paged(d: Dims, q_idx, kc_cache, q, k_cache, v_cache, k_scale, v_scale, page_table, q_pos, out, ws,
                 scores=None, sel_blk=None, sel_pos=None, stream=None):
    """decode with the compressed keys in the KV cache's pages."""
    _want(q_idx, "q_idx", (d.batch, d.n_q, d.n_idx_heads, d.idx_dim), torch.bfloat16)
    _want_kc_cache(d, kc_cache)
    _check_attn_inputs(d, q, k_cache, v_cache, k_scale, v_scale, page_table, q_pos, out)
    if scores is not None:
        _want(scores, "scores", (d.batch, d.n_q, d.max_blocks), torch.float32)
    if sel_blk is not None:
        _want(sel_blk, "sel_blk", (d.batch, d.n_q, d.topk), torch.int32)
    if sel_pos is not None:
        _want(sel_pos, "sel_pos", (d.batch, d.n_q, d.width), torch.int32)
    w, n = _ws(d, ws)
    _check(lib.qsa_decode_paged(ctypes.byref(d), _ptr(q_idx), _ptr(kc_cache), _ptr(q), _ptr(k_cache),
                                _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(page_table), _ptr(q_pos),
                                _ptr(scores), _ptr(sel_blk), _ptr(sel_pos), _ptr(out), w, n, _stream(stream)),
           "qsa_decode_paged")


def draft_attn(d: Dims, q, k_cache, v_cache, k_scale, v_scale, page_table, sel_pos, sel_q_pos, src, q_pos,
               out, ws, stream=None):
    """MTP draft step reusing an earlier selection: draft query j of request r
    (d.n_q draft queries per request) attends over row src[r][j] of sel_pos
    (made for a query at sel_q_pos[r][src[r][j]]) plus the positions after
    that query up to its own, q_pos[r][j]."""
    _check_attn_inputs(d, q, k_cache, v_cache, k_scale, v_scale, page_table, q_pos, out)
    if sel_pos.dim() != 3 or sel_pos.shape[0] != d.batch or sel_pos.shape[2] != d.width:
        raise ValueError(f"sel_pos: expected [{d.batch}][n_sel][{d.width}], got {tuple(sel_pos.shape)}")
    n_sel = int(sel_pos.shape[1])
    _want(sel_pos, "sel_pos", (d.batch, n_sel, d.width), torch.int32)
    _want(sel_q_pos, "sel_q_pos", (d.batch, n_sel), torch.int32)
    _want(src, "src", (d.batch, d.n_q), torch.int32)
    w, n = _ws(d, ws)
    _check(lib.qsa_draft_attn(ctypes.byref(d), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                              _ptr(page_table), _ptr(sel_pos), _ptr(sel_q_pos), n_sel, _ptr(src), _ptr(q_pos),
                              _ptr(out), w, n, _stream(stream)), "qsa_draft_attn")


def decode(d: Dims, q_idx, kc, q, k_cache, v_cache, k_scale, v_scale, page_table, q_pos, out, ws,
           scores=None, sel_blk=None, sel_pos=None, stream=None):
    """The fused step: scores -> top-k selection -> sparse attention."""
    _want(q_idx, "q_idx", (d.batch, d.n_q, d.n_idx_heads, d.idx_dim), torch.bfloat16)
    _want(kc, "kc", (d.batch, d.max_blocks, d.n_idx_heads, d.idx_dim), torch.bfloat16)
    _check_attn_inputs(d, q, k_cache, v_cache, k_scale, v_scale, page_table, q_pos, out)
    if scores is not None:
        _want(scores, "scores", (d.batch, d.n_q, d.max_blocks), torch.float32)
    if sel_blk is not None:
        _want(sel_blk, "sel_blk", (d.batch, d.n_q, d.topk), torch.int32)
    if sel_pos is not None:
        _want(sel_pos, "sel_pos", (d.batch, d.n_q, d.width), torch.int32)
    w, n = _ws(d, ws)
    _check(lib.qsa_decode(ctypes.byref(d), _ptr(q_idx), _ptr(kc), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                          _ptr(k_scale), _ptr(v_scale), _ptr(page_table), _ptr(q_pos), _ptr(scores),
                          _ptr(sel_blk), _ptr(sel_pos), _ptr(out), w, n, _stream(stream)), "qsa_decode")


def check_errors(ws: torch.Tensor, stream=None) -> Tuple[int, Tuple[int, int, int, int]]:
    """Synchronise, read and clear the device error record of ``ws``."""
    info = (ctypes.c_int32 * 4)()
    st = lib.qsa_check_errors(ctypes.c_void_p(ws.data_ptr()), _stream(stream), info)
    return st, tuple(info)


def default_sm_scale(head_dim: int = 128) -> float:
    return 1.0 / math.sqrt(head_dim)
