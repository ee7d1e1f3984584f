"""Pins of the CPU oracle against facts that do not come from the oracle itself:
the pages' printed constants, format definitions checked by library routines,
closed forms, brute force on tiny inputs and invariants of the method.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

from block_sparse_attention_qsa_gb300 import synth
from oracle import qsa_oracle as O
from tests._util import bits, small_spec, to_numpy_inputs, unpage

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# the pages' printed constants
# --------------------------------------------------------------------------

def test_page_constants():
    g = json.load(open(os.path.join(GOLDEN, "page_constants.json")))
    assert O.BLOCK == g["block_tokens"]["value"]
    assert O.TOPK == g["topk_blocks"]["value"]
    assert O.TOPK * O.BLOCK == g["max_full_positions"]["value"]
    # width = all selected positions + the largest unfilled block (3 tokens)
    assert O.WIDTH == g["selection_width"]["value"] == 512 * 4 + 3
    # the shared-memory figures decompose as 256 B per block (128 BF16 dims)
    # plus 1 KiB per query sharing the tile
    sb, sa = g["score_smem_bytes"]["before"], g["score_smem_bytes"]["after"]
    tb, ta = g["score_tile_blocks"]["before"], g["score_tile_blocks"]["after"]
    nq = g["max_queries_sharing_tile"]["value"]
    assert sb == tb * 128 * 2 + 1 * 1024
    assert sa == ta * 128 * 2 + nq * 1024


# --------------------------------------------------------------------------
# storage formats, against torch's own conversions
# --------------------------------------------------------------------------

def test_e4m3_decode_all_codes_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_to_f64(codes)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(ref[~nan], got[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(got[~nan]))


def test_e4m3_landmarks():
    d = O.e4m3_to_f64(np.array([0x7E, 0x08, 0x01, 0x38, 0xB8, 0x00, 0x07, 0x77], dtype=np.uint8))
    assert d.tolist() == [448.0, 2.0 ** -6, 2.0 ** -9, 1.0, -1.0, 0.0, 7 * 2.0 ** -9, 240.0]
    # finite positive codes decode strictly increasing
    pos = O.e4m3_to_f64(np.arange(0, 0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)


def test_bf16_round_vs_torch():
    rng = np.random.default_rng(3)
    x = rng.standard_normal(200000).astype(np.float32) * np.float32(3.0)
    # exact halfway cases between neighbouring BF16 values, both parities
    base = (rng.integers(0, 1 << 15, 5000).astype(np.uint32) << 16) | 0x8000
    x = np.concatenate([x, base.view(np.float32), np.array([0.0, -0.0, 1e-40, -3e38, 3.3e38], np.float32)])
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(O.f32_to_bf16_bits(x), ref)


def test_bf16_decode_landmarks():
    d = O.bf16_to_f64(np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x3E80], dtype=np.uint16))
    assert d.tolist() == [1.0, -2.0, 0.0, -0.0, 0.25]


# --------------------------------------------------------------------------
# compressed key
# --------------------------------------------------------------------------

def _bf(vals):
    return O.f32_to_bf16_bits(np.array(vals, dtype=np.float32))


def test_compress_closed_forms():
    H, D = 2, 128
    rng = np.random.default_rng(5)
    key = _bf(rng.standard_normal((H, D)))
    same = np.stack([key] * 4)  # 4 identical tokens
    assert np.array_equal(O.compress_keys(same, 1)[0], key)
    a = _bf(np.full((H, D), 1.0))
    b = _bf(np.full((H, D), 2.0))
    kc = O.compress_keys(np.stack([a, a, a, b]), 1)
    assert np.all(O.bf16_to_f64(kc) == 1.25)
    x = _bf(rng.standard_normal((H, D)))
    y = _bf(rng.standard_normal((H, D)))
    neg = lambda t: t ^ np.uint16(0x8000)
    kc = O.compress_keys(np.stack([x, neg(x), y, neg(y)]), 1)
    assert np.all(O.bf16_to_f64(kc) == 0.0)


def test_compress_rounding_vs_torch():
    rng = np.random.default_rng(9)
    keys = _bf(rng.standard_normal((64, 1, 128)))
    got = O.compress_keys(keys, 16)
    k = torch.from_numpy(keys.view(np.int16)).view(torch.bfloat16).float().view(16, 4, 1, 128)
    ref = (((k[:, 0] + k[:, 1]) + k[:, 2]) + k[:, 3]) * 0.25
    ref = ref.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


# --------------------------------------------------------------------------
# scores
# --------------------------------------------------------------------------

def test_score_unit_query_reads_one_dim():
    rng = np.random.default_rng(11)
    H, D, nb = 3, 128, 40
    kc = _bf(rng.standard_normal((nb, H, D)))
    for h, d in [(0, 0), (1, 77), (2, 127)]:
        q = np.zeros((H, D), dtype=np.float32)
        q[h, d] = 1.0
        s = O.score_row(_bf(q), kc, 4 * nb - 1)
        assert np.array_equal(s, O.bf16_to_f64(kc[:, h, d]).astype(np.float32))


def test_score_sums_heads_and_scales_exactly():
    rng = np.random.default_rng(12)
    H, D, nb = 4, 128, 33
    kc = _bf(rng.standard_normal((nb, H, D)))
    q = np.zeros((H, D), dtype=np.float32)
    q[0, 5] = 1.0
    q[3, 9] = 1.0
    s = O.score_row(_bf(q), kc, 4 * nb - 1)
    ref = (O.bf16_to_f64(kc[:, 0, 5]) + O.bf16_to_f64(kc[:, 3, 9])).astype(np.float32)
    assert np.array_equal(s, ref)
    qr = _bf(rng.standard_normal((H, D)))
    q2 = _bf(O.bf16_to_f64(qr) * 2.0)
    assert np.array_equal(O.score_row(q2, kc, 4 * nb - 1), 2 * O.score_row(qr, kc, 4 * nb - 1))


def test_score_matches_exact_sum_and_counts_full_blocks():
    rng = np.random.default_rng(13)
    H, D, nb = 2, 128, 20
    kc = _bf(rng.standard_normal((nb, H, D)))
    q = _bf(rng.standard_normal((H, D)))
    for p in [0, 2, 3, 4, 7, 8, 78, 79]:
        s = O.score_row(q, kc, p)
        assert s.shape == ((p + 1) // 4,)
        assert s.dtype == np.float32
        for b in range(s.shape[0]):
            terms = [O.bf16_to_f64(q[h, d : d + 1])[0] * O.bf16_to_f64(kc[b, h, d : d + 1])[0]
                     for h in range(H) for d in range(D)]
            exact = np.float32(math.fsum(terms))
            assert abs(float(s[b]) - float(exact)) <= abs(float(exact)) * 2 ** -23


# --------------------------------------------------------------------------
# top-k
# --------------------------------------------------------------------------

def _brute_topk(s, k=512):
    """Block b is kept iff fewer than k blocks beat it: a higher score, or an
    equal score (with -0.0 == +0.0) at a lower index; NaN is beaten by any
    number and NaNs order by index."""
    n = len(s)
    keep = []
    for b in range(n):
        beat = 0
        for c in range(n):
            if c == b:
                continue
            sb, sc = s[b], s[c]
            if math.isnan(sb):
                better = (not math.isnan(sc)) or c < b
            elif math.isnan(sc):
                better = False
            else:
                better = sc > sb or (sc == sb and c < b)
            beat += better
        if beat < k:
            keep.append(b)
    out = np.full(k, -1, dtype=np.int32)
    out[: len(keep)] = keep
    return out


@pytest.mark.parametrize("n", [0, 1, 37, 511, 512, 513, 900])
def test_topk_random_vs_brute(n):
    rng = np.random.default_rng(n)
    s = rng.standard_normal(n).astype(np.float32)
    assert np.array_equal(O.topk_blocks(s), _brute_topk(s.tolist()))


def _adversarial_rows():
    rows = {}
    rows["all_equal"] = np.full(1500, 0.75, np.float32)
    rows["two_values"] = np.where(np.arange(1400) % 3 == 0, 1.0, -1.0).astype(np.float32)
    rows["ascending"] = np.arange(1200, dtype=np.float32)
    rows["descending"] = np.arange(1200, dtype=np.float32)[::-1].copy()
    z = np.zeros(1300, np.float32)
    z[::2] = -0.0
    z[5::97] = -1.0
    rows["signed_zeros"] = z
    t = np.full(1000, -5.0, np.float32)
    t[100:612] = 2.0  # exactly 512 tied at the top
    rows["exactly_512_tied"] = t
    u = np.full(1000, -5.0, np.float32)
    u[::3] = 2.0  # 334 above the threshold
    u[1::3] = 1.0  # 333 tied at the threshold, 178 needed
    rows["ties_at_threshold"] = u
    w = np.linspace(-3, 3, 800).astype(np.float32)
    w[::7] = np.nan
    rows["with_nan"] = w
    return rows


@pytest.mark.parametrize("name", list(_adversarial_rows().keys()))
def test_topk_adversarial_vs_brute(name):
    s = _adversarial_rows()[name]
    assert np.array_equal(O.topk_blocks(s), _brute_topk(s.tolist()))


def _partition_topk(s, k=512):
    """Second formulation: threshold = k-th largest value, take all larger,
    then the lowest-index blocks equal to the threshold."""
    n = len(s)
    if n <= k:
        out = np.full(k, -1, np.int32)
        out[:n] = np.arange(n)
        return out
    thr = np.partition(s, n - k)[n - k]
    above = np.nonzero(s > thr)[0]
    ties = np.nonzero(s == thr)[0][: k - above.shape[0]]
    return np.sort(np.concatenate([above, ties])).astype(np.int32)


@pytest.mark.parametrize("n", [513, 12501, 65537])
def test_topk_long_rows_vs_partition(n):
    rng = np.random.default_rng(n)
    s = (rng.standard_normal(n) * 5.7).astype(np.float32)
    s[rng.integers(0, n, 40)] = s[rng.integers(0, n, 40)]  # a few duplicate values
    assert np.array_equal(O.topk_blocks(s), _partition_topk(s))


# --------------------------------------------------------------------------
# selection buffer
# --------------------------------------------------------------------------

def _valid(sp):
    return int(np.sum(sp >= 0))


@pytest.mark.parametrize("p", [0, 1, 2, 3, 4, 2046, 2047, 2048, 2049, 2050, 2051, 4098, 50000, 50001, 50002, 50003])
def test_selection_width_invariant(p):
    rng = np.random.default_rng(p)
    s = rng.standard_normal(O.n_full(p)).astype(np.float32)
    sp = O.select_positions(O.topk_blocks(s), p)
    assert sp.shape == (2051,)
    nv = _valid(sp)
    assert nv == 4 * min(512, O.n_full(p)) + O.n_part(p) <= 2051
    v = sp[:nv]
    assert np.all(sp[nv:] == -1)
    assert np.all(np.diff(v) > 0) and v[-1] <= p
    # the unfilled block's positions are kept whatever the scores
    part = list(range(4 * O.n_full(p), p + 1))
    assert v[nv - len(part):].tolist() == part
    if O.n_full(p) <= 512:
        assert v.tolist() == list(range(p + 1))


def test_selection_counts_of_the_two_verify_workloads():
    # one query at 4,098: 1,024 full blocks + 3 partial tokens -> width filled
    assert 4 * min(512, O.n_full(4098)) + O.n_part(4098) == 2051
    # four verify queries at 50,000..50,003
    got = [4 * min(512, O.n_full(p)) + O.n_part(p) for p in range(50000, 50004)]
    assert got == [2049, 2050, 2051, 2048]


# --------------------------------------------------------------------------
# attention
# --------------------------------------------------------------------------

def _oracle_inputs(spec):
    inp = synth.make_inputs(spec)
    npi = to_numpy_inputs(inp)
    B = spec.batch
    npi["kc"] = np.stack([O.compress_keys(npi["idx_keys"][r], spec.max_blocks()) for r in range(B)])
    return npi


def _dense_for(npi, spec, r, j, allowed):
    T = spec.tokens()[r]
    K = unpage(npi["k_cache"], npi["page_table"][r], T)
    V = unpage(npi["v_cache"], npi["page_table"][r], T)
    if spec.kv_dtype == "fp8":
        K = O.e4m3_to_f64(K) * npi["k_scale"][None, :, None]
        V = O.e4m3_to_f64(V) * npi["v_scale"][None, :, None]
    else:
        K, V = O.bf16_to_f64(K), O.bf16_to_f64(V)
    return O.dense_attn(O.bf16_to_f64(npi["q"][r, j]), K, V, allowed)


@pytest.mark.parametrize("first,kv", [(0, "bf16"), (5, "bf16"), (130, "fp8"), (2044, "bf16"), (2047, "fp8")])
def test_sparse_equals_dense_when_all_blocks_fit(first, kv):
    spec = small_spec([first], n_q=4, kv_dtype=kv, seed=100 + first)
    npi = _oracle_inputs(spec)
    res = O.decode_step(npi, kv)
    for j in range(4):
        p = first + j
        assert O.n_full(p) <= 512
        dense = _dense_for(npi, spec, 0, j, list(range(p + 1)))
        assert np.max(np.abs(res["out"][(0, j)] - dense)) < 1e-12


def test_one_block_dropped_at_513_full_blocks():
    # p = 2051: 2,052 tokens, 513 full blocks, nothing unfilled
    spec = small_spec([2051], n_q=1, seed=41)
    npi = _oracle_inputs(spec)
    res = O.decode_step(npi)
    s = res["scores"][(0, 0)]
    assert s.shape == (513,)
    lowest = min(range(513), key=lambda b: (s[b], -b))  # ties drop the higher index
    allowed = [t for t in range(2052) if t // 4 != lowest]
    dense = _dense_for(npi, spec, 0, 0, allowed)
    assert np.max(np.abs(res["out"][(0, 0)] - dense)) < 1e-12
    assert _valid(res["sel_pos"][(0, 0)]) == 2048


def test_each_verify_query_sees_only_its_prefix():
    spec = small_spec([3001], n_q=4, seed=55)
    npi = _oracle_inputs(spec)
    base = O.decode_step(npi)
    P = spec.page_size
    for j in range(4):
        p = 3001 + j
        pert = {k: v.copy() for k, v in npi.items()}
        # change every token after p: K, V and index keys (hence compressed keys)
        for t in range(p + 1, spec.tokens()[0]):
            page = pert["page_table"][0, t // P]
            pert["k_cache"][page, :, t % P] ^= np.uint16(0x0013)
            pert["v_cache"][page, :, t % P] ^= np.uint16(0x000F)
        pert["idx_keys"][0, p + 1 :] ^= np.uint16(0x0021)  # mantissa bits: stays finite
        pert["kc"] = np.stack([O.compress_keys(pert["idx_keys"][0], spec.max_blocks())])
        res = O.decode_step(pert, rows=[(0, jj) for jj in range(4)])
        changed = set(range(p + 1, spec.tokens()[0]))
        for jj in range(4):
            if jj <= j:
                assert np.array_equal(res["scores"][(0, jj)], base["scores"][(0, jj)])
                assert np.array_equal(res["sel_pos"][(0, jj)], base["sel_pos"][(0, jj)])
                assert np.array_equal(res["out"][(0, jj)], base["out"][(0, jj)])
            else:
                # a later query reads some changed token, so its output moves
                assert changed & set(base["sel_pos"][(0, jj)].tolist())
                assert not np.array_equal(res["out"][(0, jj)], base["out"][(0, jj)])


# --------------------------------------------------------------------------
# MTP draft steps reusing a selection (arex "四类优化", MTP reuse; 10100 第三处)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_draft_equals_dense_when_everything_fits(kv):
    # 1,500 + 4 tokens: the selection of the query at 1,500 holds every position
    # 0..1500, so a draft query at 1,503 reusing it sees exactly 0..1503
    spec = small_spec([1500], n_q=4, kv_dtype=kv, seed=71)
    npi = _oracle_inputs(spec)
    res = O.decode_step(npi, kv, rows=[(0, 0)])
    row = res["sel_pos"][(0, 0)]
    q = npi["q"][0, 3]
    ks = npi["k_scale"] if kv == "fp8" else None
    vs = npi["v_scale"] if kv == "fp8" else None
    out = O.draft_attn(q, npi["k_cache"], npi["v_cache"], npi["page_table"][0], row, 1500, 1503, kv, ks, vs)
    dense = _dense_for(npi, spec, 0, 3, list(range(1504)))
    assert np.max(np.abs(out - dense)) < 1e-12


def test_draft_beyond_512_blocks_is_the_row_plus_the_gap():
    spec = small_spec([3001], n_q=4, seed=72)
    npi = _oracle_inputs(spec)
    res = O.decode_step(npi, rows=[(0, 0)])
    row = res["sel_pos"][(0, 0)]
    assert _valid(row) == 2050  # 512 blocks + the unfilled block: 3,002 tokens = 4 * 750 + 2
    allowed = sorted(set(int(t) for t in row if t >= 0) | {3002, 3003, 3004})
    assert len(allowed) == 2053
    out = O.draft_attn(npi["q"][0, 3], npi["k_cache"], npi["v_cache"], npi["page_table"][0], row, 3001, 3004)
    dense = _dense_for(npi, spec, 0, 3, allowed)
    assert np.max(np.abs(out - dense)) < 1e-12
    # with no gap the draft query attends over the row alone
    out0 = O.draft_attn(npi["q"][0, 3], npi["k_cache"], npi["v_cache"], npi["page_table"][0], row, 3001, 3001)
    dense0 = _dense_for(npi, spec, 0, 3, sorted(int(t) for t in row if t >= 0))
    assert np.max(np.abs(out0 - dense0)) < 1e-12


def test_draft_position_bounds():
    row = np.full(2051, -1, np.int32)
    row[:3] = [0, 1, 2]
    assert O.draft_positions(row, 10, 10).tolist() == [0, 1, 2]
    assert O.draft_positions(row, 10, 13).tolist() == [0, 1, 2, 11, 12, 13]
    assert len(O.draft_positions(row, 10, 10 + O.MAX_DRAFT_GAP)) == 3 + O.MAX_DRAFT_GAP
    with pytest.raises(ValueError):
        O.draft_positions(row, 10, 9)  # before its selection's query
    with pytest.raises(ValueError):
        O.draft_positions(row, 10, 11 + O.MAX_DRAFT_GAP)  # too far after it
    bad = row.copy()
    bad[3] = 11
    with pytest.raises(ValueError):
        O.draft_positions(bad, 10, 12)  # a reused row may not hold a later position


def test_draft_is_causal():
    spec = small_spec([2600], n_q=4, seed=73)
    npi = _oracle_inputs(spec)
    row = O.decode_step(npi, rows=[(0, 0)])["sel_pos"][(0, 0)]
    args = (npi["q"][0, 2], npi["page_table"][0], row, 2600, 2602)
    base = O.draft_attn(args[0], npi["k_cache"], npi["v_cache"], *args[1:])
    P = spec.page_size
    kc, vc = npi["k_cache"].copy(), npi["v_cache"].copy()
    page = npi["page_table"][0, 2603 // P]
    kc[page, :, 2603 % P] ^= np.uint16(0x0013)  # after the draft query: no effect
    vc[page, :, 2603 % P] ^= np.uint16(0x000F)
    assert np.array_equal(O.draft_attn(args[0], kc, vc, *args[1:]), base)
    page = npi["page_table"][0, 2602 // P]
    vc[page, :, 2602 % P] ^= np.uint16(0x000F)  # in the gap: the output moves
    assert not np.array_equal(O.draft_attn(args[0], kc, vc, *args[1:]), base)


def test_attention_softmax_invariants():
    spec = small_spec([700], n_q=1, seed=61)
    npi = _oracle_inputs(spec)
    row = npi["page_table"][0]
    # all V rows equal -> output equals that row for every head
    v = npi["v_cache"].copy()
    vrow = O.f32_to_bf16_bits(np.linspace(-1, 1, 128).astype(np.float32))
    v[:, :, :] = vrow
    sp = O.select_positions(O.topk_blocks(np.zeros(O.n_full(700), np.float32)), 700)
    out = O.sparse_attn(npi["q"][0, 0], npi["k_cache"], v, row, sp)
    assert np.max(np.abs(out - O.bf16_to_f64(vrow)[None, :])) < 1e-14
    # a single valid position -> output equals that position's V
    one = np.full(2051, -1, np.int32)
    one[0] = 333
    out = O.sparse_attn(npi["q"][0, 0], npi["k_cache"], npi["v_cache"], row, one)
    page = row[333 // 64]
    for h in range(16):
        assert np.array_equal(out[h], O.bf16_to_f64(npi["v_cache"][page, h // 8, 333 % 64]))


def test_attention_two_positions_closed_form():
    spec = small_spec([100], n_q=1, seed=62)
    npi = _oracle_inputs(spec)
    row = npi["page_table"][0]
    sel = np.full(2051, -1, np.int32)
    sel[:2] = [10, 90]
    out = O.sparse_attn(npi["q"][0, 0], npi["k_cache"], npi["v_cache"], row, sel)
    q = O.bf16_to_f64(npi["q"][0, 0])
    for h in (0, 9):
        g = h // 8
        k = [O.bf16_to_f64(npi["k_cache"][row[t // 64], g, t % 64]) for t in (10, 90)]
        v = [O.bf16_to_f64(npi["v_cache"][row[t // 64], g, t % 64]) for t in (10, 90)]
        d = (q[h] @ k[1] - q[h] @ k[0]) / math.sqrt(128)
        w1 = 1.0 / (1.0 + math.exp(-d))  # logistic of the logit gap
        assert np.max(np.abs(out[h] - ((1 - w1) * v[0] + w1 * v[1]))) < 1e-12


def test_fp8_cache_decodes_with_scales():
    spec = small_spec([300], n_q=2, kv_dtype="fp8", seed=63)
    npi = _oracle_inputs(spec)
    assert npi["k_cache"].dtype == np.uint8 and npi["k_scale"].shape == (2,)
    res = O.decode_step(npi, "fp8")
    for j in range(2):
        dense = _dense_for(npi, spec, 0, j, list(range(300 + j + 1)))
        assert np.max(np.abs(res["out"][(0, j)] - dense)) < 1e-12


# --------------------------------------------------------------------------
# the input generator
# --------------------------------------------------------------------------

def test_generator_is_splitmix64_and_chunk_independent(monkeypatch):
    assert synth.splitmix64_py(0, 0) == 0xE220A8397B1DCDAF  # first SplitMix64 output of seed 0
    c = torch.arange(1000, dtype=torch.int64)
    got = synth.splitmix64(c, 12345).tolist()
    assert got == [synth._s64(synth.splitmix64_py(i, 12345)) for i in range(1000)]
    a = synth.normal_bf16((3, 1000), 9)
    monkeypatch.setattr(synth, "_CHUNK", 77)
    b = synth.normal_bf16((3, 1000), 9)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    x = synth.normal_f32(1 << 20, 4)
    assert abs(x.mean().item()) < 5e-3 and abs(x.std().item() - 1) < 5e-3


def test_generator_e4m3_storage():
    x = synth.normal_bf16((50, 2, 64, 128), 21)
    codes, scale = synth.quantize_e4m3(x, 1)
    dec = O.e4m3_to_f64(bits(codes)) * scale.numpy()[None, :, None, None]
    xf = x.float().numpy()
    assert np.all(np.abs(bits(codes).astype(np.int64) & 0x7F) <= 0x7E)
    # round to nearest: error at most half a step of 3 mantissa bits
    assert np.all(np.abs(dec - xf) <= np.abs(xf) * 2 ** -4 + scale.numpy().max() * 2 ** -10)
