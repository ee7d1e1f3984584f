"""CPU oracle for the QSA decode / MTP-verify step.

TEST INFRASTRUCTURE ONLY. Nothing in the library path imports, calls or runs
this module: it is used by ``tests/``, by ``__graft_entry__.smoke()`` and by the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``. It shares no code
with the CUDA path; its inputs are plain numpy arrays.

What it computes follows the pages' statement of the Qwen Sparse Attention
(QSA) selection pipeline (arex-research.com, "稀疏选择、CuTe DSL 内核与 MTP 复用：
四类优化", bullets 1-3; 10100.com, "第一处"):

  * tokens form micro-blocks of 4 and each block has a compressed index key;
  * each query scores every full block (FP32 score buffer);
  * each query keeps at most 512 full blocks (at most 2,048 positions);
  * the current unfilled block is kept without selection;
  * the selection buffer has a fixed width of 2,051 positions;
  * sparse attention runs over the selected positions with a BF16 query and a
    BF16 or FP8-E4M3 KV cache.

Points the pages leave open are taken as follows (each is listed with its
reason in the design notes of the repository):

  * compressed key: FP32 mean of the block's 4 BF16 index keys, summed as
    ((k0 + k1) + k2) + k3, times 0.25, stored BF16 round-to-nearest-even;
  * score: plain dot product of index query and compressed key, summed over
    index heads, computed here in FP64 and rounded once to FP32;
  * full blocks of query position p: b < floor((p + 1) / 4); the partial
    block holds positions 4 * floor((p + 1) / 4) .. p ((p + 1) mod 4 of them);
  * ties in the top-k go to the lower block index; -0.0 equals +0.0; a NaN
    score ranks below every number;
  * selection buffer: selected blocks ascending, each expanded to its 4
    positions, then the partial block's positions, then -1 up to 2,051;
  * attention: query head h reads KV head h // (H_q / H_kv); scale
    1/sqrt(head_dim); plain max-subtracted softmax over the valid selected
    positions; FP8 values are decode(code) * per-head FP32 scale;
  * MTP draft steps (arex, same section, heading "MTP 复用"; 10100.com,
    "第三处": later draft steps reuse the positions selected before): a draft
    query at p reusing the selection row made for a query at p_src <= p
    attends over that row's positions plus p_src + 1 .. p, the positions the
    row cannot hold (at most 64 of them).

All floating point here is FP64 unless a step fixes FP32 (the score buffer,
the compressed-key mean) or BF16 (the compressed key's storage).
"""

from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np

BLOCK = 4
TOPK = 512
WIDTH = TOPK * BLOCK + (BLOCK - 1)  # 2,051
MAX_DRAFT_GAP = 64  # positions a draft query may lie after the selection's query


# ---------------------------------------------------------------------------
# storage formats
# ---------------------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """BF16 bit patterns (uint16) to FP64: BF16 is the top half of an FP32."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round FP32 values to BF16 (round to nearest, ties to even).

    The kept part is the top 16 bits of the FP32 pattern; the dropped low 16
    bits decide the rounding: above half rounds up, below half rounds down,
    exactly half rounds to the even kept pattern. NaN maps to a quiet NaN.
    """
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    keep = u >> np.uint64(16)
    low = u & np.uint64(0xFFFF)
    up = (low > 0x8000) | ((low == 0x8000) & ((keep & np.uint64(1)) == 1))
    r = (keep + up.astype(np.uint64)) & np.uint64(0xFFFF)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    r = np.where(nan, np.uint64(0x7FC0), r)
    return r.astype(np.uint16)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """Decode FP8-E4M3 codes (OCP 8-bit floating point, E4M3 variant).

    Bit layout s.eeee.mmm, exponent bias 7, no infinities. Exponent field 0
    encodes subnormals m/8 * 2^-6; exponent field 15 with mantissa 7 is NaN;
    every other code is (1 + m/8) * 2^(e - 7). The largest finite value is
    0x7E = 448.
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where((c >> 7) & 1 == 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    sub = (m / 8.0) * 2.0 ** -6
    nor = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    v = s * np.where(e == 0, sub, nor)
    return np.where((e == 15) & (m == 7), np.nan, v)


# ---------------------------------------------------------------------------
# micro-blocks
# ---------------------------------------------------------------------------

def n_full(p: int) -> int:
    """Full 4-token blocks visible to a query at position p (tokens 0..p)."""
    return (p + 1) // BLOCK


def n_part(p: int) -> int:
    """Tokens in the query's unfilled block (0..3)."""
    return (p + 1) % BLOCK


def compress_keys(idx_keys_bits: np.ndarray, nblocks: int) -> np.ndarray:
    """Compressed index key of each of the first ``nblocks`` blocks.

    ``idx_keys_bits``: BF16 bits [T][H][D] (per-token index keys of one
    request, T >= 4 * nblocks). Returns BF16 bits [nblocks][H][D]: the FP32
    mean of the block's 4 keys, summed in token order, rounded to BF16.
    """
    k = bf16_to_f64(idx_keys_bits[: BLOCK * nblocks]).astype(np.float32)
    k = k.reshape(nblocks, BLOCK, *k.shape[1:])
    s = k[:, 0] + k[:, 1]
    s = s + k[:, 2]
    s = s + k[:, 3]
    mean = s * np.float32(0.25)
    return f32_to_bf16_bits(mean)


# ---------------------------------------------------------------------------
# the step
# ---------------------------------------------------------------------------

def score_row(q_idx_bits: np.ndarray, kc_bits: np.ndarray, p: int) -> np.ndarray:
    """FP32 block scores of one query at position p.

    ``q_idx_bits``: BF16 bits [H][D]; ``kc_bits``: BF16 bits [>= n_full][H][D].
    Score of block b < n_full(p) = sum over heads h and dims d of
    q[h][d] * kc[b][h][d], in FP64, rounded once to FP32. Blocks at or past
    n_full(p) are not scored.
    """
    nb = n_full(p)
    q = bf16_to_f64(q_idx_bits)
    kc = bf16_to_f64(kc_bits[:nb])
    s = np.einsum("bhd,hd->b", kc, q)
    return s.astype(np.float32)


def topk_blocks(scores: np.ndarray, k: int = TOPK) -> np.ndarray:
    """The k highest-scoring blocks, ties to the lower index, ascending.

    Orders every candidate by (score descending, block index ascending), with
    NaN after every number and -0.0 equal to +0.0, takes the first
    min(k, n), and returns them sorted by block index, padded with -1 to k.
    """
    s = np.asarray(scores, dtype=np.float64)
    n = s.shape[0]
    idx = np.arange(n)
    nan = np.isnan(s)
    key = np.where(nan, 0.0, -s)  # -(-0.0) == -(+0.0) numerically
    order = np.lexsort((idx, key, nan))  # last key is primary
    take = np.sort(order[: min(k, n)])
    out = np.full(k, -1, dtype=np.int32)
    out[: take.shape[0]] = take
    return out


def select_positions(sel_blk: np.ndarray, p: int) -> np.ndarray:
    """Selection buffer of a query at position p (width 2,051).

    Each selected block b (ascending) contributes positions 4b..4b+3; the
    unfilled block's positions 4*n_full(p)..p follow; -1 fills the rest.
    """
    out = np.full(WIDTH, -1, dtype=np.int32)
    pos = []
    for b in sel_blk:
        if b < 0:
            continue
        pos.extend(range(BLOCK * int(b), BLOCK * int(b) + BLOCK))
    pos.extend(range(BLOCK * n_full(p), p + 1))
    out[: len(pos)] = pos
    return out


def gather_kv(cache: np.ndarray, page_table_row: np.ndarray, positions: Sequence[int],
              g: int, kv_dtype: str, scale: float) -> np.ndarray:
    """K or V rows of KV head g at token positions, as FP64 [n][D].

    ``cache``: [num_pages][H_kv][P][D] (BF16 bits or E4M3 codes). Token t lives
    in page ``page_table_row[t // P]`` at slot ``t % P``.
    """
    P = cache.shape[2]
    rows = []
    for t in positions:
        page = int(page_table_row[t // P])
        rows.append(cache[page, g, t % P])
    raw = np.stack(rows) if rows else np.zeros((0, cache.shape[3]), dtype=cache.dtype)
    if kv_dtype == "bf16":
        return bf16_to_f64(raw)
    if kv_dtype == "fp8":
        return e4m3_to_f64(raw) * float(scale)
    raise ValueError(kv_dtype)


def sparse_attn(q_bits: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                page_table_row: np.ndarray, sel_pos: np.ndarray, kv_dtype: str = "bf16",
                k_scale: Optional[Sequence[float]] = None, v_scale: Optional[Sequence[float]] = None,
                sm_scale: Optional[float] = None) -> np.ndarray:
    """Attention of one query token over its selected positions, FP64.

    ``q_bits``: BF16 bits [H_q][D]. ``sel_pos``: positions, -1 = unused.
    Query head h reads KV head h // (H_q / H_kv). Returns [H_q][D] FP64.
    """
    Hq, D = q_bits.shape
    Hkv = k_cache.shape[1]
    group = Hq // Hkv
    scale = 1.0 / math.sqrt(D) if sm_scale is None else sm_scale
    ks = [1.0] * Hkv if k_scale is None else [float(x) for x in k_scale]
    vs = [1.0] * Hkv if v_scale is None else [float(x) for x in v_scale]
    pos = [int(t) for t in sel_pos if t >= 0]
    q = bf16_to_f64(q_bits)
    out = np.zeros((Hq, D))
    for g in range(Hkv):
        K = gather_kv(k_cache, page_table_row, pos, g, kv_dtype, ks[g])
        V = gather_kv(v_cache, page_table_row, pos, g, kv_dtype, vs[g])
        for h in range(g * group, (g + 1) * group):
            s = (K @ q[h]) * scale
            w = np.exp(s - s.max())
            out[h] = (w @ V) / w.sum()
    return out


def draft_positions(sel_row: np.ndarray, p_src: int, p: int) -> np.ndarray:
    """Positions a draft query at p attends to when it reuses the selection
    row ``sel_row`` made for a query at p_src (arex, "四类优化", MTP reuse;
    10100.com, "第三处"): the row's valid positions, then p_src + 1 .. p."""
    if not (0 <= p_src <= p <= p_src + MAX_DRAFT_GAP):
        raise ValueError(f"draft position {p} does not follow its selection's query {p_src}")
    kept = [int(t) for t in sel_row if t >= 0]
    if any(t > p_src for t in kept):
        raise ValueError("selection row holds a position after its own query")
    return np.array(kept + list(range(p_src + 1, p + 1)), dtype=np.int64)


def draft_attn(q_bits: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, page_table_row: np.ndarray,
               sel_row: np.ndarray, p_src: int, p: int, kv_dtype: str = "bf16",
               k_scale: Optional[Sequence[float]] = None, v_scale: Optional[Sequence[float]] = None,
               sm_scale: Optional[float] = None) -> np.ndarray:
    """Attention of a draft query at p over a reused selection row (made for
    p_src) and the positions after p_src, FP64 [H_q][D]."""
    return sparse_attn(q_bits, k_cache, v_cache, page_table_row, draft_positions(sel_row, p_src, p), kv_dtype,
                       k_scale, v_scale, sm_scale)


def dense_attn(q: np.ndarray, K: np.ndarray, V: np.ndarray, allowed: Sequence[int],
               sm_scale: Optional[float] = None) -> np.ndarray:
    """Plain attention over contiguous per-token K/V, written as loops.

    ``q``: FP64 [H_q][D]; ``K``, ``V``: FP64 [T][H_kv][D] indexed by token
    position; ``allowed``: the positions attended to. Independent of the
    paged/selection machinery: it is the textbook softmax(q k^T * scale) v
    evaluated position by position with a running maximum.
    """
    Hq, D = q.shape
    Hkv = K.shape[1]
    scale = 1.0 / math.sqrt(D) if sm_scale is None else sm_scale
    out = np.zeros((Hq, D))
    for h in range(Hq):
        g = h * Hkv // Hq
        logits = [float(np.dot(q[h], K[t, g])) * scale for t in allowed]
        mx = max(logits)
        den = 0.0
        acc = np.zeros(D)
        for t, lg in zip(allowed, logits):
            w = math.exp(lg - mx)
            den += w
            acc += w * V[t, g]
        out[h] = acc / den
    return out


def decode_step(inp: dict, kv_dtype: str = "bf16", rows: Optional[Sequence[tuple]] = None,
                sm_scale: Optional[float] = None) -> dict:
    """The whole step for the (request, query) rows asked for.

    ``inp`` holds numpy arrays: q_idx [B][n_q][H][D] (BF16 bits), kc
    [B][max_blocks][H][D] (BF16 bits), q [B][n_q][H_q][D] (BF16 bits),
    k_cache, v_cache, k_scale, v_scale, page_table [B][max_pages],
    q_pos [B][n_q]. Returns dicts keyed by (r, j) of scores, sel_blk, sel_pos
    and out (FP64 [H_q][D]).
    """
    qp = inp["q_pos"]
    B, nq = qp.shape
    if rows is None:
        rows = [(r, j) for r in range(B) for j in range(nq)]
    res = {"scores": {}, "sel_blk": {}, "sel_pos": {}, "out": {}}
    for r, j in rows:
        p = int(qp[r, j])
        s = score_row(inp["q_idx"][r, j], inp["kc"][r], p)
        sb = topk_blocks(s)
        sp = select_positions(sb, p)
        o = sparse_attn(inp["q"][r, j], inp["k_cache"], inp["v_cache"], inp["page_table"][r], sp,
                        kv_dtype, inp.get("k_scale"), inp.get("v_scale"), sm_scale)
        res["scores"][(r, j)] = s
        res["sel_blk"][(r, j)] = sb
        res["sel_pos"][(r, j)] = sp
        res["out"][(r, j)] = o
    return res
