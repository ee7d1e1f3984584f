"""The C ABI library: it builds, loads without a GPU, exports every symbol
include/qsa.h declares, and rejects bad arguments before touching the GPU."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def qsa():
    import __graft_entry__

    __graft_entry__.build()
    from block_sparse_attention_qsa_gb300 import qsa as q

    return q


def _declared():
    txt = open(os.path.join(ROOT, "include", "qsa.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(qsa_[a-z_0-9]+)\s*\(", txt)))


def test_exports_every_declared_symbol(qsa):
    names = _declared()
    assert len(names) == 21
    assert set(names) == set(qsa.EXPORTS)
    lib = ctypes.CDLL(qsa.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_draft_gap_matches_the_header(qsa):
    txt = open(os.path.join(ROOT, "include", "qsa.h")).read()
    m = re.search(r"#define QSA_MAX_DRAFT_GAP (\d+)", txt)
    assert m and int(m.group(1)) == qsa.MAX_DRAFT_GAP
    m = re.search(r"#define QSA_MAX_CHUNK (\d+)", txt)
    assert m and int(m.group(1)) == qsa.MAX_CHUNK
    m = re.search(r"#define QSA_MAX_SCORE_BATCH (\d+)", txt)
    assert m and int(m.group(1)) == qsa.MAX_SCORE_BATCH


def test_abi_version_and_status_strings(qsa):
    assert qsa.lib.qsa_abi_version() == qsa.ABI_VERSION
    assert qsa.status_str(qsa.OK) == "QSA_OK"
    assert qsa.status_str(qsa.ERR_BAD_INDEX) == "QSA_ERR_BAD_INDEX"
    assert qsa.status_str(99) == "QSA_UNKNOWN_STATUS"


def test_default_dims_are_the_pages_geometry(qsa):
    d = qsa.Dims()
    qsa.lib.qsa_dims_default(ctypes.byref(d))
    assert (d.n_q_heads, d.n_kv_heads, d.head_dim, d.idx_dim) == (16, 2, 128, 128)
    assert (d.topk, d.block, d.width, d.page_size) == (512, 4, 2051, 64)
    assert d.kv_dtype == qsa.KV_BF16 and d.sm_scale == 0.0


# These pass made-up device pointers, which the calls must refuse before any
# launch; they run only where no CUDA device exists, so that a regression can
# only return an error and never touch memory.
no_device = pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="fake pointers: CPU-only test")


@no_device
def test_workspace_size_and_rejections_need_no_gpu(qsa):
    d = qsa.make_dims(32, 4, 15301, 957, 28352)
    n = ctypes.c_size_t(0)
    assert qsa.lib.qsa_workspace_size(ctypes.byref(d), ctypes.byref(n)) == qsa.OK
    assert n.value >= 32 * 4 * 15301 * 4  # holds the decode step's score buffer
    fake = ctypes.c_void_p(1 << 20)
    # null pointers
    assert qsa.lib.qsa_score(ctypes.byref(d), None, fake, fake, fake, fake, n.value, None) == qsa.ERR_INVALID_ARG
    assert qsa.lib.qsa_decode(ctypes.byref(d), fake, fake, fake, fake, fake, None, None, fake, fake, None,
                              None, None, None, fake, n.value, None) == qsa.ERR_INVALID_ARG
    # FP8 needs its scales
    d8 = qsa.make_dims(1, 4, 100, 10, 10, kv_dtype="fp8")
    assert qsa.lib.qsa_sparse_attn(ctypes.byref(d8), fake, fake, fake, None, None, fake, fake, fake, fake,
                                   fake, 1 << 30, None) == qsa.ERR_INVALID_ARG
    # geometry outside the supported set
    for field, val in [("head_dim", 64), ("n_q", 5), ("topk", 256), ("width", 2052), ("page_size", 48),
                       ("n_q_heads", 12), ("n_idx_heads", 5), ("kv_dtype", 7)]:
        bad = qsa.make_dims(1, 4, 100, 10, 10)
        setattr(bad, field, val)
        assert qsa.lib.qsa_workspace_size(ctypes.byref(bad), ctypes.byref(n)) == qsa.ERR_UNSUPPORTED, field
    bad = qsa.make_dims(0, 4, 100, 10, 10)
    assert qsa.lib.qsa_workspace_size(ctypes.byref(bad), ctypes.byref(n)) == qsa.ERR_INVALID_ARG
    # a misaligned or missing workspace
    assert qsa.lib.qsa_topk(ctypes.byref(d), fake, fake, fake, fake, None, n.value, None) == qsa.ERR_WORKSPACE
    assert qsa.lib.qsa_topk(ctypes.byref(d), fake, fake, fake, fake, ctypes.c_void_p((1 << 20) + 8), n.value,
                            None) == qsa.ERR_WORKSPACE
    # the attention query is copied 16 bytes at a time: a 4-byte-aligned one is refused
    q4 = ctypes.c_void_p((1 << 20) + 4)
    assert qsa.lib.qsa_sparse_attn(ctypes.byref(d), q4, fake, fake, None, None, fake, fake, fake, fake, fake,
                                   n.value, None) == qsa.ERR_INVALID_ARG
    assert qsa.lib.qsa_sparse_attn_rows(ctypes.byref(d), q4, fake, fake, None, None, fake, fake, fake, n.value,
                                        None) == qsa.ERR_INVALID_ARG
    # 4-byte and 2-byte elements need their own alignment
    odd = ctypes.c_void_p((1 << 20) + 2)
    assert qsa.lib.qsa_score(ctypes.byref(d), fake, fake, odd, fake, fake, n.value, None) == qsa.ERR_INVALID_ARG
    assert qsa.lib.qsa_sparse_attn_rows(ctypes.byref(d), fake, fake, fake, None, None, fake,
                                        ctypes.c_void_p((1 << 20) + 1), fake, n.value, None) == qsa.ERR_INVALID_ARG
    # resolve / attention over rows: null pointers
    assert qsa.lib.qsa_resolve(ctypes.byref(d), fake, fake, None, fake, fake, n.value, None) == qsa.ERR_INVALID_ARG
    assert qsa.lib.qsa_sparse_attn_rows(ctypes.byref(d), fake, fake, fake, None, None, None, fake, fake, n.value,
                                        None) == qsa.ERR_INVALID_ARG
    # chunked scoring: chunk length and batch limits
    assert qsa.lib.qsa_score_chunk(ctypes.byref(d), 0, fake, fake, fake, fake, fake, n.value,
                                   None) == qsa.ERR_INVALID_ARG
    assert qsa.lib.qsa_score_chunk(ctypes.byref(d), qsa.MAX_CHUNK + 1, fake, fake, fake, fake, fake, n.value,
                                   None) == qsa.ERR_INVALID_ARG
    # scoring: batch limit
    huge = qsa.make_dims(qsa.MAX_SCORE_BATCH + 1, 1, 4, 1, 1)
    assert qsa.lib.qsa_score(ctypes.byref(huge), fake, fake, fake, fake, fake, 1 << 40, None) == qsa.ERR_UNSUPPORTED
    big = qsa.make_dims(65536, 1, 4, 1, 1)
    assert qsa.lib.qsa_score_chunk(ctypes.byref(big), 1, fake, fake, fake, fake, fake, 1 << 40,
                                   None) == qsa.ERR_UNSUPPORTED


def test_binding_refuses_host_tensors(qsa):
    import torch

    d = qsa.make_dims(1, 1, 8, 1, 1)
    with pytest.raises(ValueError, match="CUDA"):
        qsa.score(d, torch.zeros(1, 1, 1, 128, dtype=torch.bfloat16), torch.zeros(1, 8, 1, 128, dtype=torch.bfloat16),
                  torch.zeros(1, 1, dtype=torch.int32), torch.zeros(1, 1, 8), torch.zeros(4096, dtype=torch.uint8))


@no_device
def test_noalloc_rejects_sizes_beyond_its_scratch(qsa):
    # 300,000 requests x 4 queries: far more resolved cache rows than the
    # 16 MiB static scratch holds
    d = qsa.make_dims(300000, 4, 16, 1, 1)
    fake = ctypes.c_void_p(1 << 20)
    st = qsa.lib.qsa_sparse_attn_noalloc(ctypes.byref(d), fake, fake, fake, None, None, fake, fake, fake, fake,
                                         None)
    assert st == qsa.ERR_WORKSPACE
