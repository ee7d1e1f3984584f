"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Tolerances (stated by the step's contract and restated here):
  * compressed keys, top-k block ids and selection buffers: bit-exact;
  * scores: |gpu - ref| <= 1e-4 * max(|ref|, 1);
  * attention outputs: max-abs <= 1e-2 with BF16 KV, <= 3e-2 with FP8 KV
    (the oracle decodes the same E4M3 bytes and scales).
Top-k is bit-exact when both sides start from the same FP32 score buffer, so
its unit tests feed both sides seeded score buffers. End to end, every row is
chained stage by stage: the GPU's scores against the oracle's, the oracle's
selection on the GPU's own scores against the GPU's selection (bit-exact),
and the oracle's attention over the GPU's own selection against the GPU's
output. The pure oracle chain is compared as well; a row whose 512th and
513th oracle scores are closer than the score tolerance can legitimately
select differently there and is counted.
"""

import math

import numpy as np
import pytest
import torch

from block_sparse_attention_qsa_gb300 import synth
from oracle import qsa_oracle as O
from tests._util import bits, small_spec, to_numpy_inputs

pytestmark = pytest.mark.gpu

SCORE_RTOL = 1e-4
ATOL = {"bf16": 1e-2, "fp8": 3e-2}


@pytest.fixture(scope="module")
def qsa():
    import __graft_entry__

    __graft_entry__.build()
    from block_sparse_attention_qsa_gb300 import qsa as q

    return q


def _dev(inp):
    return {k: v.cuda() for k, v in inp.items()}


def _kc_oracle(npi, spec):
    return np.stack([O.compress_keys(npi["idx_keys"][r], spec.max_blocks()) for r in range(spec.batch)])


def _bf16_tensor(bits_u16):
    return torch.from_numpy(np.ascontiguousarray(bits_u16).view(np.int16)).view(torch.bfloat16)


def _check_ok(qsa, ws):
    st, info = qsa.check_errors(ws)
    assert st == qsa.OK, info


SPECS = {
    "b2-h1-bf16": lambda: small_spec([3001, 1498], n_q=4, seed=5),
    "b3-h4-fp8": lambda: small_spec([2600, 4097, 77], n_q=4, n_idx_heads=4, kv_dtype="fp8", seed=6),
    "b1-nq1-h2": lambda: small_spec([5003], n_q=1, n_idx_heads=2, seed=7),
    "b2-nq3-h3": lambda: small_spec([2100, 3333], n_q=3, n_idx_heads=3, seed=8),
    "b2-nq2-h1-fp8": lambda: small_spec([9000, 2050], n_q=2, kv_dtype="fp8", seed=9),
    # other page sizes: 16-token pages (a block of 4 tokens is a quarter page) and 256-token pages
    "b2-p16-fp8": lambda: synth.Spec("small-p16", 2, 4, [2600, 999], 1, "fp8", True, 10, page_size=16),
    "b2-p256-nq2-h2": lambda: synth.Spec("small-p256", 2, 2, [4000, 2301], 2, "bf16", True, 11, page_size=256),
}


# --------------------------------------------------------------------------
# per-stage parity on small specs (several tiles, ragged tails)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", list(SPECS))
def test_compress_keys_bit_exact(qsa, name):
    spec = SPECS[name]()
    inp = synth.make_inputs(spec)
    npi = to_numpy_inputs(inp)
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    g = _dev(inp)
    kc = torch.zeros((spec.batch, spec.max_blocks(), spec.n_idx_heads, 128), dtype=torch.bfloat16, device="cuda")
    qsa.compress_keys(d, g["idx_keys"], g["q_pos"], kc, ws)
    _check_ok(qsa, ws)
    ref = _kc_oracle(npi, spec)
    got = bits(kc)
    for r in range(spec.batch):
        nb = O.n_full(max(spec.q_pos()[r]))
        assert np.array_equal(got[r, :nb], ref[r, :nb])
        assert np.all(got[r, nb:] == 0)  # blocks not yet full are left alone


def test_compress_keys_block_lo_refreshes_only_new_blocks(qsa):
    spec = small_spec([3001, 1498], n_q=4, seed=15)
    inp = synth.make_inputs(spec)
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    g = _dev(inp)
    kc = torch.zeros((2, spec.max_blocks(), 1, 128), dtype=torch.bfloat16, device="cuda")
    lo = torch.tensor([700, 100], dtype=torch.int32, device="cuda")
    qsa.compress_keys(d, g["idx_keys"], g["q_pos"], kc, ws, block_lo=lo)
    _check_ok(qsa, ws)
    ref = _kc_oracle(to_numpy_inputs(inp), spec)
    got = bits(kc)
    assert np.all(got[0, :700] == 0) and np.array_equal(got[0, 700:751], ref[0, 700:751])
    assert np.all(got[1, :100] == 0) and np.array_equal(got[1, 100:375], ref[1, 100:375])


@pytest.mark.parametrize("name", list(SPECS))
def test_score_parity(qsa, name):
    spec = SPECS[name]()
    inp = synth.make_inputs(spec)
    npi = to_numpy_inputs(inp)
    npi["kc"] = _kc_oracle(npi, spec)
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    g = _dev(inp)
    kc = _bf16_tensor(npi["kc"]).cuda()
    scores = torch.full((spec.batch, spec.n_q, spec.max_blocks()), float("nan"), device="cuda")
    qsa.score(d, g["q_idx"], kc, g["q_pos"], scores, ws)
    _check_ok(qsa, ws)
    got = scores.cpu().numpy()
    for r in range(spec.batch):
        for j in range(spec.n_q):
            p = spec.q_pos()[r][j]
            ref = O.score_row(npi["q_idx"][r, j], npi["kc"][r], p)
            nb = ref.shape[0]
            err = np.abs(got[r, j, :nb].astype(np.float64) - ref) / np.maximum(np.abs(ref), 1.0)
            assert err.max() <= SCORE_RTOL, (r, j, err.max())
            assert np.all(np.isnan(got[r, j, nb:]))  # nothing written past the full blocks


@pytest.mark.parametrize("config,batch,ctx", [(2, 32, None), (4, 8, 131072)])
def test_score_full_size_every_row(qsa, config, batch, ctx):
    # every score of every row at a full batch, written once and nowhere else,
    # on repeated calls through one workspace
    spec = synth.spec_for(config, batch=batch, ctx=ctx)
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    H, nb_max = spec.n_idx_heads, spec.max_blocks()
    q_idx = synth.normal_bf16((spec.batch, spec.n_q, H, 128), spec.seed + 11, "cuda")
    kc = synth.normal_bf16((spec.batch, nb_max, H, 128), spec.seed + 12, "cuda")
    q_pos = torch.tensor(spec.q_pos(), dtype=torch.int32, device="cuda")
    scores = torch.full((spec.batch, spec.n_q, nb_max), float("nan"), device="cuda")
    for _ in range(2):
        qsa.score(d, q_idx, kc, q_pos, scores, ws)
    _check_ok(qsa, ws)
    qb, kb, got = bits(q_idx), bits(kc), scores.cpu().numpy()
    for r in range(spec.batch):
        for j in range(spec.n_q):
            ref = O.score_row(qb[r, j], kb[r], spec.q_pos()[r][j])
            nb = ref.shape[0]
            err = np.abs(got[r, j, :nb].astype(np.float64) - ref) / np.maximum(np.abs(ref), 1.0)
            assert err.max() <= SCORE_RTOL, (r, j, err.max())
            assert np.all(np.isnan(got[r, j, nb:]))


def test_score_batch_with_tables_beyond_48kb(qsa):
    # 7,000 short requests: the scoring kernel's per-request tables need more
    # than the default 48 KB of shared memory, raised by the launcher on use
    B, n_q, mb = 7000, 2, 12
    d = qsa.make_dims(B, n_q, mb, 1, 1)
    ws = qsa.make_workspace(d)
    q_idx = synth.normal_bf16((B, n_q, 1, 128), 501, "cuda")
    kc = synth.normal_bf16((B, mb, 1, 128), 502, "cuda")
    pos = [[(7 * r) % 48, (7 * r) % 48 + 1] for r in range(B)]
    q_pos = torch.tensor(pos, dtype=torch.int32, device="cuda")
    scores = torch.full((B, n_q, mb), float("nan"), device="cuda")
    qsa.score(d, q_idx, kc, q_pos, scores, ws)
    _check_ok(qsa, ws)
    qb, kb, got = bits(q_idx), bits(kc), scores.cpu().numpy()
    for r in (0, 1, 2, 3999, 6997, 6998, 6999):
        for j in range(n_q):
            ref = O.score_row(qb[r, j], kb[r], pos[r][j])
            nb = ref.shape[0]
            err = np.abs(got[r, j, :nb].astype(np.float64) - ref) / np.maximum(np.abs(ref), 1.0)
            assert nb == 0 or err.max() <= SCORE_RTOL, (r, j)
            assert np.all(np.isnan(got[r, j, nb:]))


def _score_rows(kind, n, seed):
    rng = np.random.default_rng(seed)
    if kind == "normal":
        return (rng.standard_normal(n) * 5.7).astype(np.float32)
    if kind == "all_equal":
        return np.full(n, 1.5, np.float32)
    if kind == "two_values":
        return np.where(rng.random(n) < 0.3, 2.0, -1.0).astype(np.float32)
    if kind == "ascending":
        return np.arange(n, dtype=np.float32)
    if kind == "descending":
        return np.arange(n, dtype=np.float32)[::-1].copy()
    if kind == "signed_zeros":
        z = np.zeros(n, np.float32)
        z[::2] = -0.0
        z[3::11] = -2.0
        z[5::13] = 1.0
        return z
    if kind == "exact_512_top":
        z = np.full(n, -3.0, np.float32)
        z[rng.choice(n, 512, replace=False)] = 7.0
        return z
    if kind == "ties_at_threshold":
        z = (rng.standard_normal(n) - 10).astype(np.float32)
        z[rng.choice(n, 300, replace=False)] = 50.0
        idx = rng.choice(np.nonzero(z < 0)[0], 600, replace=False)
        z[idx] = 1.25  # 600 tied, 212 taken
        return z
    if kind == "few_bits":
        # values that agree in their top 22 key bits: exercises the last pass
        base = np.float32(3.0).view(np.uint32)
        return (base + rng.integers(0, 1024, n).astype(np.uint32)).view(np.float32)
    if kind == "with_nan":
        z = rng.standard_normal(n).astype(np.float32)
        z[::5] = np.nan
        return z
    raise ValueError(kind)


TOPK_CASES = [
    ("normal", 0), ("normal", 1), ("normal", 511), ("normal", 512), ("normal", 513),
    ("normal", 12501), ("normal", 15301), ("normal", 65537),
    ("all_equal", 2000), ("all_equal", 65537), ("two_values", 9000), ("ascending", 5000),
    ("descending", 5000), ("signed_zeros", 4000), ("exact_512_top", 7000),
    ("ties_at_threshold", 6000), ("few_bits", 3000), ("few_bits", 60000), ("with_nan", 3000),
    # longer than the register path: the cluster path at 4 rows
    ("normal", 32769), ("ties_at_threshold", 40000), ("two_values", 30000), ("with_nan", 26000),
    ("exact_512_top", 131073),
]


def _topk_case(qsa, kind, n, batch):
    # requests of 2 queries: rows of n and shorter ragged rows. 160 rows take
    # one CTA per row; 2 or 4 rows longer than the register path take the
    # cluster path (several CTAs per row).
    n_q = 2
    mb = max(n, 1)
    lens = ([[n, max(0, n - 37)], [max(0, n // 3), n]] * ((batch + 1) // 2))[:batch]
    # query k of a row with L full blocks sits at 4L + k - 1 (k partial tokens)
    q_pos = [[max(0, 4 * L + k - 1) for k, L in enumerate(row)] for row in lens]
    for row in q_pos:
        for p in row:
            assert O.n_full(p) <= mb
    scores = np.stack([np.stack([_score_rows(kind, mb, 100 * (r % 2) + j + 7 * (r // 2)) for j in range(n_q)])
                       for r in range(batch)])
    d = qsa.make_dims(batch, n_q, mb, 1, 1)
    ws = qsa.make_workspace(d)
    sc = torch.from_numpy(scores).cuda()
    qp = torch.tensor(q_pos, dtype=torch.int32, device="cuda")
    sb = torch.full((batch, n_q, 512), 7, dtype=torch.int32, device="cuda")
    sp = torch.full((batch, n_q, 2051), 7, dtype=torch.int32, device="cuda")
    qsa.topk(d, sc, qp, sb, sp, ws)
    _check_ok(qsa, ws)
    gb, gp = sb.cpu().numpy(), sp.cpu().numpy()
    for r in (range(batch) if batch <= 2 else (0, 1, 2, 3, batch // 2, batch - 2, batch - 1)):
        for j in range(n_q):
            p = q_pos[r][j]
            ref_b = O.topk_blocks(scores[r, j, : O.n_full(p)])
            assert np.array_equal(gb[r, j], ref_b), (r, j)
            assert np.array_equal(gp[r, j], O.select_positions(ref_b, p)), (r, j)


@pytest.mark.parametrize("batch", [2, 80])
@pytest.mark.parametrize("kind,n", TOPK_CASES)
def test_topk_bit_exact_on_shared_scores(qsa, kind, n, batch):
    _topk_case(qsa, kind, n, batch)


@pytest.mark.parametrize("batch", [1, 2])
@pytest.mark.parametrize("n", [98305, 131073, 262144, 262145])
@pytest.mark.parametrize("kind", ["all_equal", "two_values", "ties_at_threshold"])
def test_topk_long_rows_with_many_ties_at_small_batches(qsa, kind, n, batch):
    # 2 or 4 rows of up to 262,144 blocks take the cluster path with eight
    # CTAs per row and up to 32 keys per thread; all-equal and two-valued rows
    # put more than 65,535 tied blocks in the CTAs before the last ones, so the
    # slots of the ties taken depend on the counts of every lower-ranked CTA.
    # One block more (262,145) leaves the cluster path for the long-row path
    # (radix passes over the whole row, listed 65,536 blocks at a time).
    _topk_case(qsa, kind, n, batch)


def test_topk_is_deterministic_across_runs(qsa):
    n = 20000
    scores = np.stack([_score_rows("two_values", n, 3)])[None]
    d = qsa.make_dims(1, 1, n, 1, 1)
    ws = qsa.make_workspace(d)
    sc = torch.from_numpy(scores).cuda()
    qp = torch.tensor([[4 * n - 1]], dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(3):
        sb = torch.empty((1, 1, 512), dtype=torch.int32, device="cuda")
        sp = torch.empty((1, 1, 2051), dtype=torch.int32, device="cuda")
        qsa.topk(d, sc, qp, sb, sp, ws)
        outs.append((sb.cpu(), sp.cpu()))
    assert all(torch.equal(outs[0][0], o[0]) and torch.equal(outs[0][1], o[1]) for o in outs)


@pytest.mark.parametrize("name", list(SPECS))
def test_sparse_attn_parity_on_oracle_selection(qsa, name):
    spec = SPECS[name]()
    inp = synth.make_inputs(spec)
    npi = to_numpy_inputs(inp)
    npi["kc"] = _kc_oracle(npi, spec)
    res = O.decode_step(npi, spec.kv_dtype)
    sel = np.stack([np.stack([res["sel_pos"][(r, j)] for j in range(spec.n_q)]) for r in range(spec.batch)])
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    g = _dev(inp)
    out = torch.full((spec.batch, spec.n_q, 16, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    qsa.sparse_attn(d, g["q"], g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"], g["page_table"],
                    torch.from_numpy(sel).cuda(), g["q_pos"], out, ws)
    _check_ok(qsa, ws)
    got = out.float().cpu().numpy()
    for r in range(spec.batch):
        for j in range(spec.n_q):
            err = np.max(np.abs(got[r, j] - res["out"][(r, j)]))
            assert err <= ATOL[spec.kv_dtype], (r, j, err)


@pytest.mark.parametrize("name", ["b2-h1-bf16", "b2-p16-fp8"])
def test_resolve_then_rows_attention_equals_sparse_attn(qsa, name):
    # qsa_sparse_attn's two launches called one by one: the same rows and the
    # same output bit for bit; rows outside the cache are skipped like -1
    spec = SPECS[name]()
    inp = synth.make_inputs(spec)
    npi = to_numpy_inputs(inp)
    npi["kc"] = _kc_oracle(npi, spec)
    res = O.decode_step(npi, spec.kv_dtype)
    sel = torch.from_numpy(np.stack([np.stack([res["sel_pos"][(r, j)] for j in range(spec.n_q)])
                                     for r in range(spec.batch)])).cuda()
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    g = _dev(inp)
    ref = torch.empty((spec.batch, spec.n_q, 16, 128), dtype=torch.bfloat16, device="cuda")
    qsa.sparse_attn(d, g["q"], g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"], g["page_table"], sel,
                    g["q_pos"], ref, ws)
    rows = torch.full_like(sel, -7)
    qsa.resolve(d, sel, g["q_pos"], g["page_table"], rows, ws)
    out = torch.empty_like(ref)
    qsa.sparse_attn_rows(d, g["q"], g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"], rows, out, ws)
    _check_ok(qsa, ws)
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    # the rows follow the documented formula
    P, H = spec.page_size, spec.n_kv_heads
    s_h, r_h, pt = sel.cpu().numpy(), rows.cpu().numpy(), inp["page_table"].numpy()
    for r in range(spec.batch):
        for j in range(spec.n_q):
            t = s_h[r, j]
            want = np.where(t >= 0, pt[r, np.maximum(t, 0) // P] * H * P + np.maximum(t, 0) % P, -1)
            assert np.array_equal(r_h[r, j], want), (r, j)
    # out-of-range rows planted where -1 was: skipped, the output is unchanged
    bad = rows.clone()
    lim = d.num_pages * H * P - (H - 1) * P
    holes = bad < 0
    bad[holes] = torch.tensor([lim, lim + 5, 2 ** 31 - 1, -2], dtype=torch.int32, device="cuda").repeat(
        int(holes.sum().item()) // 4 + 1)[: int(holes.sum().item())]
    out2 = torch.empty_like(ref)
    qsa.sparse_attn_rows(d, g["q"], g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"], bad, out2, ws)
    _check_ok(qsa, ws)
    assert torch.equal(out2.view(torch.int16), ref.view(torch.int16))


def test_sparse_attn_with_holes_and_single_positions(qsa):
    spec = small_spec([4000, 130], n_q=2, seed=21)
    inp = synth.make_inputs(spec)
    npi = to_numpy_inputs(inp)
    rng = np.random.default_rng(4)
    sel = np.full((2, 2, 2051), -1, np.int32)
    sel[0, 0, :1500] = np.sort(rng.choice(4001, 1500, replace=False))
    sel[0, 0, rng.choice(1500, 300, replace=False)] = -1  # holes anywhere
    sel[0, 1, 0] = 4001  # a single position
    sel[1, 0, 1000] = 17  # a single position late in the buffer
    sel[1, 1, :131] = np.arange(131)[::-1]  # any order
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    g = _dev(inp)
    out = torch.empty((2, 2, 16, 128), dtype=torch.bfloat16, device="cuda")
    qsa.sparse_attn(d, g["q"], g["k_cache"], g["v_cache"], None, None, g["page_table"],
                    torch.from_numpy(sel).cuda(), g["q_pos"], out, ws)
    _check_ok(qsa, ws)
    got = out.float().cpu().numpy()
    for r in range(2):
        for j in range(2):
            ref = O.sparse_attn(npi["q"][r, j], npi["k_cache"], npi["v_cache"], npi["page_table"][r], sel[r, j])
            assert np.max(np.abs(got[r, j] - ref)) <= 1e-2


# --------------------------------------------------------------------------
# the fused step, chained stage by stage
# --------------------------------------------------------------------------

def _flip_is_near_tie(gpu_blk, ref_blk, ref_scores, k=512, tol=SCORE_RTOL):
    """True when two selections differ only in blocks whose oracle scores sit
    within the score tolerance of the oracle's k-th largest score: a boundary
    that FP32 rounding may legitimately move."""
    g = set(int(b) for b in gpu_blk if b >= 0)
    o = set(int(b) for b in ref_blk if b >= 0)
    if len(g) != len(o):
        return False
    thr = np.sort(ref_scores.astype(np.float64))[::-1][k - 1]
    band = 2 * tol * max(abs(thr), 1.0)
    return all(abs(float(ref_scores[b]) - thr) <= band for b in g ^ o)


def _oracle_request(spec, g, r):
    """The oracle's own view of request r, copied from the generator's
    tensors (its pages renumbered 0..n-1), with its compressed keys."""
    npg = spec.pages_per_request()[r]
    pages = g["page_table"][r, :npg].long()
    npi = {
        "q_idx": bits(g["q_idx"][r : r + 1]),
        "q": bits(g["q"][r : r + 1]),
        "k_cache": bits(g["k_cache"][pages]),
        "v_cache": bits(g["v_cache"][pages]),
        "k_scale": g["k_scale"].cpu().numpy(),
        "v_scale": g["v_scale"].cpu().numpy(),
        "page_table": np.arange(npg, dtype=np.int32)[None],
        "q_pos": bits(g["q_pos"][r : r + 1]),
    }
    npi["kc"] = O.compress_keys(bits(g["idx_keys"][r]), spec.max_blocks())[None]
    return npi


def _check_row_chain(spec, npi, j, got_scores, got_blk, got_pos, got_out):
    """Stage-by-stage parity of one (request, query) row of a fused step:

      1. the GPU's FP32 scores against the oracle's scores (1e-4 relative);
      2. the oracle's top-k and selection run on the GPU's own FP32 scores
         against the GPU's block ids and selection buffer, bit-exact;
      3. the oracle's attention over the GPU's own selection buffer against
         the GPU's output (1e-2 BF16 KV, 3e-2 FP8 KV);
      4. the pure oracle chain (oracle scores -> oracle selection -> oracle
         attention): the same selection and output, unless the two selections
         differ only in blocks within the score tolerance of the oracle's 512th
         score (FP32 rounding may move that boundary).

    Returns True when the pure oracle chain took another boundary block."""
    p = int(npi["q_pos"][0, j])
    fp8 = spec.kv_dtype == "fp8"
    ks, vs = (npi["k_scale"], npi["v_scale"]) if fp8 else (None, None)
    res = O.decode_step(npi, spec.kv_dtype, rows=[(0, j)])
    ref_s = res["scores"][(0, j)]
    nb = ref_s.shape[0]
    err = np.abs(got_scores[:nb].astype(np.float64) - ref_s) / np.maximum(np.abs(ref_s), 1.0)
    assert np.max(err, initial=0.0) <= SCORE_RTOL, (j, "scores")
    own_blk = O.topk_blocks(got_scores[:nb])
    assert np.array_equal(got_blk, own_blk), (j, "selection on the GPU's scores")
    assert np.array_equal(got_pos, O.select_positions(own_blk, p)), (j, "selection buffer")
    own_out = O.sparse_attn(npi["q"][0, j], npi["k_cache"], npi["v_cache"], npi["page_table"][0], got_pos,
                            spec.kv_dtype, ks, vs)
    err = np.max(np.abs(got_out - own_out))
    assert err <= ATOL[spec.kv_dtype], (j, "attention over the GPU's selection", err)
    if not np.array_equal(got_blk, res["sel_blk"][(0, j)]):
        assert _flip_is_near_tie(got_blk, res["sel_blk"][(0, j)], ref_s), (j, "pure chain")
        return True
    assert np.array_equal(got_pos, res["sel_pos"][(0, j)]), (j, "pure chain")
    err = np.max(np.abs(got_out - res["out"][(0, j)]))
    assert err <= ATOL[spec.kv_dtype], (j, "pure chain", err)
    return False


def _decode_and_compare(qsa, spec, rows=None, gpu_inputs=None):
    """Run qsa_decode on the GPU and check the requested (r, j) rows against
    the oracle stage by stage (_check_row_chain). Every row passes the chained
    stages; returns (rows whose pure oracle chain took another boundary block,
    rows checked)."""
    g = gpu_inputs if gpu_inputs is not None else _dev(synth.make_inputs(spec))
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    kc = torch.zeros((spec.batch, spec.max_blocks(), spec.n_idx_heads, 128), dtype=torch.bfloat16, device="cuda")
    qsa.compress_keys(d, g["idx_keys"], g["q_pos"], kc, ws)
    scores = torch.empty((spec.batch, spec.n_q, spec.max_blocks()), device="cuda")
    sb = torch.empty((spec.batch, spec.n_q, 512), dtype=torch.int32, device="cuda")
    sp = torch.empty((spec.batch, spec.n_q, 2051), dtype=torch.int32, device="cuda")
    out = torch.empty((spec.batch, spec.n_q, 16, 128), dtype=torch.bfloat16, device="cuda")
    qsa.decode(d, g["q_idx"], kc, g["q"], g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"],
               g["page_table"], g["q_pos"], out, ws, scores=scores, sel_blk=sb, sel_pos=sp)
    _check_ok(qsa, ws)
    if rows is None:
        rows = [(r, j) for r in range(spec.batch) for j in range(spec.n_q)]
    skipped = 0
    sc_h, sb_h, sp_h, out_h = scores.cpu().numpy(), sb.cpu().numpy(), sp.cpu().numpy(), out.float().cpu().numpy()
    for r in sorted(set(r for r, _ in rows)):
        npi = _oracle_request(spec, g, r)
        nb_r = O.n_full(max(spec.q_pos()[r]))
        assert np.array_equal(bits(kc[r, :nb_r]), npi["kc"][0, :nb_r])
        for rr, j in rows:
            if rr == r:
                skipped += _check_row_chain(spec, npi, j, sc_h[r, j], sb_h[r, j], sp_h[r, j], out_h[r, j])
    print(f"{spec.name}: {len(rows)} rows checked stage by stage; the pure oracle chain took another "
          f"boundary block in {skipped}")
    return skipped, len(rows)


@pytest.mark.parametrize("name", list(SPECS))
def test_decode_small_specs(qsa, name):
    skipped, n = _decode_and_compare(qsa, SPECS[name]())
    assert skipped <= max(1, n // 10)


@pytest.mark.parametrize("config", [0, 1])
def test_decode_full_size_batch1_configs(qsa, config):
    spec = synth.spec_for(config)
    skipped, n = _decode_and_compare(qsa, spec)
    assert skipped <= 1


@pytest.mark.parametrize("config", [2, 3])
def test_decode_full_size_batch32_every_row(qsa, config):
    # all 128 (request, query) rows of the 50K-token verify batch
    spec = synth.spec_for(config)
    skipped, n = _decode_and_compare(qsa, spec)
    assert n == 128 and skipped <= 2


@pytest.mark.parametrize("config,batch", [(2, 8), (2, 16), (2, 24), (3, 8)])
def test_decode_full_size_every_row_mid_batches(qsa, config, batch):
    # batches whose attention runs in the cluster form with 5, 3 and 2 CTAs per
    # unit (units of the verify batch split over one thread-block cluster each),
    # every row checked stage by stage like batch 32
    spec = synth.spec_for(config, batch=batch)
    skipped, n = _decode_and_compare(qsa, spec)
    assert n == 4 * batch and skipped <= 2


def test_decode_long_context_batch1_sampled(qsa):
    spec = synth.spec_for(4, batch=1, ctx=131072)
    skipped, n = _decode_and_compare(qsa, spec, rows=[(0, 0), (0, 3)])
    assert skipped <= 1


def test_decode_long_context_262k_row_over_shared_memory(qsa):
    # 65,537 full blocks: the selector's keys no longer fit in shared memory
    spec = synth.spec_for(4, batch=1, ctx=262144)
    skipped, n = _decode_and_compare(qsa, spec, rows=[(0, 3)])
    assert skipped <= 1


def test_decode_long_context_batch8_cluster_rows_sampled(qsa):
    # 8 requests x 4 queries of 32,769 blocks: rows longer than the register
    # path, few enough for a cluster of four CTAs per row (inputs drawn on the
    # device; the oracle sees the same tensors)
    spec = synth.spec_for(4, batch=8, ctx=131072)
    g = synth.make_inputs(spec, device="cuda")
    skipped, n = _decode_and_compare(qsa, spec, rows=[(0, 0), (3, 2), (7, 3)], gpu_inputs=g)
    assert skipped <= 1


@pytest.mark.parametrize("batch", [32, 1, 8])
def test_decode_replayed_as_a_cuda_graph_matches_direct_calls(qsa, batch):
    # the launch the benchmark times: the fused step captured once as a CUDA
    # graph (kernels and programmatic dependencies) and replayed, at full size;
    # its outputs must equal those of direct calls bit for bit, replay after
    # replay (batch 32: stream-K attention; 1 and 8: its cluster form)
    spec = synth.spec_for(2, batch=batch)
    g = synth.make_inputs(spec, device="cuda")
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    kc = torch.zeros((spec.batch, spec.max_blocks(), 1, 128), dtype=torch.bfloat16, device="cuda")
    qsa.compress_keys(d, g["idx_keys"], g["q_pos"], kc, ws)
    out = torch.empty((spec.batch, spec.n_q, 16, 128), dtype=torch.bfloat16, device="cuda")

    def step():
        qsa.decode(d, g["q_idx"], kc, g["q"], g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"],
                   g["page_table"], g["q_pos"], out, ws)

    step()
    torch.cuda.synchronize()
    direct = out.view(torch.int16).clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(3):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), direct)
    _check_ok(qsa, ws)


# --------------------------------------------------------------------------
# invariances and errors
# --------------------------------------------------------------------------

def _run_decode(qsa, spec, g):
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    kc = torch.zeros((spec.batch, spec.max_blocks(), spec.n_idx_heads, 128), dtype=torch.bfloat16, device="cuda")
    qsa.compress_keys(d, g["idx_keys"], g["q_pos"], kc, ws)
    out = torch.empty((spec.batch, spec.n_q, 16, 128), dtype=torch.bfloat16, device="cuda")
    sp = torch.empty((spec.batch, spec.n_q, 2051), dtype=torch.int32, device="cuda")
    qsa.decode(d, g["q_idx"], kc, g["q"], g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"],
               g["page_table"], g["q_pos"], out, ws, sel_pos=sp)
    _check_ok(qsa, ws)
    return out, sp


# --------------------------------------------------------------------------
# chunked (prefill) scoring: many queries per request (qsa_score_chunk)
# --------------------------------------------------------------------------

def _chunk_case(qsa, spec, n_chunk, q_pos, seed, pad_to=1):
    """Chunked scoring of n_chunk queries per request; the buffers' block
    capacity is the spec's max_blocks rounded up to a multiple of pad_to."""
    inp = synth.make_inputs(spec)
    g = _dev(inp)
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    mb = spec.max_blocks()
    kc = torch.zeros((spec.batch, mb, spec.n_idx_heads, 128), dtype=torch.bfloat16, device="cuda")
    qsa.compress_keys(d, g["idx_keys"], g["q_pos"], kc, ws)
    mb_pad = (mb + pad_to - 1) // pad_to * pad_to
    if mb_pad != mb:
        kcp = torch.zeros((spec.batch, mb_pad, spec.n_idx_heads, 128), dtype=torch.bfloat16, device="cuda")
        kcp[:, :mb] = kc
        kc = kcp
        d.max_blocks = mb_pad
        ws = qsa.make_workspace(d)
    qi = synth.normal_bf16((spec.batch, n_chunk, spec.n_idx_heads, 128), seed, device="cuda")
    qp = torch.tensor(q_pos, dtype=torch.int32, device="cuda")
    sc = torch.full((spec.batch, n_chunk, mb_pad), float("nan"), device="cuda")
    qsa.score_chunk(d, qi, kc, qp, sc, ws)
    return sc.cpu().numpy(), bits(qi), bits(kc), ws


@pytest.mark.parametrize("h,pad_to", [(1, 1), (2, 1), (4, 1), (1, 32), (3, 32)])
def test_score_chunk_parity(qsa, h, pad_to):
    # two requests, 150 queries each: two 128-query tiles, the second ragged;
    # block capacity as drawn (misaligned rows) or padded to 32 blocks
    spec = small_spec([5003, 2900], n_q=1, n_idx_heads=h, seed=31 + h)
    n_chunk = 150
    q_pos = [[max(0, spec.first_pos[r] - 3 * (n_chunk - 1 - i)) for i in range(n_chunk)] for r in range(2)]
    q_pos[1][0] = 5  # a query with no full block yet... and one with 1
    q_pos[1][1] = 4
    sc, qi, kcb, ws = _chunk_case(qsa, spec, n_chunk, q_pos, 9001 + h, pad_to)
    _check_ok(qsa, ws)
    for r in range(2):
        for i in range(n_chunk):
            p = q_pos[r][i]
            n = O.n_full(p)
            ref = O.score_row(qi[r, i], kcb[r], p)
            got = sc[r, i, :n]
            assert np.all(np.abs(got - ref) <= SCORE_RTOL * np.maximum(np.abs(ref), 1.0)), (r, i)
            assert np.all(np.isnan(sc[r, i, n:])), (r, i)  # nothing written past the causal blocks


@pytest.mark.parametrize("pad_to", [1, 32])
def test_score_chunk_full_size_sampled(qsa, pad_to):
    # the benchmark's launch: one request of 50,000 tokens, 1,024 queries, block
    # capacity padded to 32 blocks (aligned score rows); and unpadded
    spec = synth.spec_for(1)
    n_chunk = 1024
    L = spec.first_pos[0]
    q_pos = [[L - (n_chunk - 1 - i) for i in range(n_chunk)]]
    sc, qi, kcb, ws = _chunk_case(qsa, spec, n_chunk, q_pos, 9100, pad_to)
    _check_ok(qsa, ws)
    for i in (0, 1, 63, 64, 127, 128, 511, 777, 1000, 1023):
        p = q_pos[0][i]
        n = O.n_full(p)
        ref = O.score_row(qi[0, i], kcb[0], p)
        assert np.all(np.abs(sc[0, i, :n] - ref) <= SCORE_RTOL * np.maximum(np.abs(ref), 1.0)), i
        assert np.all(np.isnan(sc[0, i, n:])), i


@pytest.mark.parametrize("case", ["no_full_block", "tiny_capacity", "one_query", "ragged_by_one", "three_requests"])
def test_score_chunk_edge_cases(qsa, case):
    # shapes at the tensor-memory kernel's edges: every tile of a chunk whose
    # queries see no full block (a CTA's first tile is still copied and
    # multiplied, and must store nothing), a block capacity below one 128-block
    # tile, a single query, 129 queries (a second query tile of one), and three
    # requests of different lengths with three index heads
    if case == "no_full_block":
        spec, n_chunk = small_spec([2000], n_q=1, seed=41), 40
        q_pos = [[i % 3 for i in range(n_chunk)]]  # positions 0..2: no full block yet
    elif case == "tiny_capacity":
        spec, n_chunk = small_spec([19], n_q=1, seed=42), 20
        q_pos = [[i for i in range(n_chunk)]]  # at most 5 full blocks
    elif case == "one_query":
        spec, n_chunk = small_spec([3333], n_q=1, n_idx_heads=2, seed=43), 1
        q_pos = [[3333]]
    elif case == "ragged_by_one":
        spec, n_chunk = small_spec([4100], n_q=1, seed=44), 129
        q_pos = [[4100 - 2 * (n_chunk - 1 - i) for i in range(n_chunk)]]
    else:
        spec, n_chunk = small_spec([5000, 700, 2600], n_q=1, n_idx_heads=3, seed=45), 70
        q_pos = [[max(0, spec.first_pos[r] - 5 * (n_chunk - 1 - i)) for i in range(n_chunk)] for r in range(3)]
    sc, qi, kcb, ws = _chunk_case(qsa, spec, n_chunk, q_pos, 9300)
    _check_ok(qsa, ws)
    for r in range(spec.batch):
        for i in range(n_chunk):
            p = q_pos[r][i]
            n = O.n_full(p)
            ref = O.score_row(qi[r, i], kcb[r], p)
            assert np.all(np.abs(sc[r, i, :n] - ref) <= SCORE_RTOL * np.maximum(np.abs(ref), 1.0)), (r, i)
            assert np.all(np.isnan(sc[r, i, n:])), (r, i)


def test_score_chunk_more_tiles_per_cta_than_its_table(qsa):
    # 16,384 queries against a 100,000-token request: 128 query tiles x 196
    # block tiles = 25,088 tiles, about 165 per CTA, more than the 128 whose
    # causal extents a CTA keeps in its table (the rest are computed on the
    # fly); sampled rows against the oracle, the scores stay on the device
    B, n_chunk, L = 1, 16384, 100000
    mb = (L + 3) // 4
    d = qsa.make_dims(B, 1, mb, 1, 1)
    ws = qsa.make_workspace(d)
    kc = synth.normal_bf16((B, mb, 1, 128), 9401, "cuda")
    qi = synth.normal_bf16((B, n_chunk, 1, 128), 9402, "cuda")
    pos = [L - 1 - 6 * (n_chunk - 1 - i) for i in range(n_chunk)]
    qp = torch.tensor([pos], dtype=torch.int32, device="cuda")
    sc = torch.full((B, n_chunk, mb), float("nan"), device="cuda")
    qsa.score_chunk(d, qi, kc, qp, sc, ws)
    _check_ok(qsa, ws)
    kb, qb = bits(kc), bits(qi)
    for i in (0, 1, 127, 128, 5000, 8191, 12345, 16255, 16256, 16383):
        p = pos[i]
        n = O.n_full(p)
        ref = O.score_row(qb[0, i], kb[0], p)
        got = sc[0, i].cpu().numpy()
        assert np.all(np.abs(got[:n] - ref) <= SCORE_RTOL * np.maximum(np.abs(ref), 1.0)), i
        assert np.all(np.isnan(got[n:])), i


def test_chunk_kernel_wait_runs_out_and_reports_a_timeout(qsa):
    # Failure detection without a fault: the test hook withholds one TMA copy
    # of the chunked-scoring kernel's first CTA, whose MMA warp then waits for
    # it until its clock limit (about a second), records a timeout, stops every
    # role and frees its tensor memory; the other CTAs finish. The timeout is
    # reported, and the next call on the same context is complete and correct.
    import time

    spec = small_spec([5003, 2900], n_q=1, seed=51)
    n_chunk = 150
    q_pos = [[max(0, spec.first_pos[r] - 3 * (n_chunk - 1 - i)) for i in range(n_chunk)] for r in range(2)]
    inp = synth.make_inputs(spec)
    g = _dev(inp)
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    kc = torch.zeros((2, spec.max_blocks(), 1, 128), dtype=torch.bfloat16, device="cuda")
    qsa.compress_keys(d, g["idx_keys"], g["q_pos"], kc, ws)
    _check_ok(qsa, ws)
    qi = synth.normal_bf16((2, n_chunk, 1, 128), 9501, device="cuda")
    qp = torch.tensor(q_pos, dtype=torch.int32, device="cuda")
    sc = torch.full((2, n_chunk, spec.max_blocks()), float("nan"), device="cuda")
    torch.cuda.synchronize()
    t0 = time.time()
    qsa.test_chunk_timeout(d, qi, kc, qp, sc, ws)
    torch.cuda.synchronize()
    waited = time.time() - t0
    st, info = qsa.check_errors(ws)
    assert st == qsa.ERR_TIMEOUT and info[0] == 5, info
    assert 0.2 < waited < 30, waited
    # the first CTA's tile (request 0, queries 0..127, blocks 0..127) was not written
    assert torch.isnan(sc[0, :128, :128]).all()
    sc.fill_(float("nan"))
    qsa.score_chunk(d, qi, kc, qp, sc, ws)
    _check_ok(qsa, ws)
    got, qb, kb = sc.cpu().numpy(), bits(qi), bits(kc)
    for r in range(2):
        for i in (0, 1, 77, 127, 128, 149):
            p = q_pos[r][i]
            n = O.n_full(p)
            ref = O.score_row(qb[r, i], kb[r], p)
            assert np.all(np.abs(got[r, i, :n] - ref) <= SCORE_RTOL * np.maximum(np.abs(ref), 1.0)), (r, i)
            assert np.all(np.isnan(got[r, i, n:])), (r, i)


def test_score_chunk_reports_a_bad_position(qsa):
    spec = small_spec([3001], n_q=1, seed=33)
    q_pos = [[-1] + [3001 - 40 + i for i in range(39)]]
    sc, qi, kcb, ws = _chunk_case(qsa, spec, 40, q_pos, 9200)
    st, info = qsa.check_errors(ws)
    assert st == qsa.ERR_BAD_INDEX and info[0] == 1 and info[2] == 0, info
    assert np.all(np.isnan(sc[0, 0]))
    p = q_pos[0][5]
    ref = O.score_row(qi[0, 5], kcb[0], p)
    assert np.all(np.abs(sc[0, 5, :O.n_full(p)] - ref) <= SCORE_RTOL * np.maximum(np.abs(ref), 1.0))


# --------------------------------------------------------------------------
# compressed keys in the KV cache's pages (qsa_*_paged)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("page_size,h,kv", [(64, 1, "bf16"), (16, 4, "fp8"), (128, 2, "bf16")])
def test_paged_compressed_keys_match_the_contiguous_path_and_the_oracle(qsa, page_size, h, kv):
    spec = synth.Spec(f"paged-kc-{page_size}", 3, 4, [3001, 1498, 5000], h, kv, True, 91 + page_size,
                      page_size=page_size)
    inp = synth.make_inputs(spec)
    g = _dev(inp)
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    B, mb, bpp = spec.batch, spec.max_blocks(), page_size // 4
    kc = torch.zeros((B, mb, h, 128), dtype=torch.bfloat16, device="cuda")
    qsa.compress_keys(d, g["idx_keys"], g["q_pos"], kc, ws)
    kcp = torch.zeros((spec.num_pages(), bpp, h, 128), dtype=torch.bfloat16, device="cuda")
    qsa.compress_keys_paged(d, g["idx_keys"], g["q_pos"], g["page_table"], kcp, ws)
    _check_ok(qsa, ws)
    kc_h, kcp_h, pt = bits(kc), bits(kcp), inp["page_table"].numpy()
    for r in range(B):
        nb = O.n_full(max(spec.q_pos()[r]))
        b = np.arange(nb)
        assert np.array_equal(kcp_h[pt[r, b // bpp], b % bpp], kc_h[r, :nb]), r
    # scores: bit for bit
    sc = torch.full((B, 4, mb), float("nan"), device="cuda")
    scp = torch.full((B, 4, mb), float("nan"), device="cuda")
    qsa.score(d, g["q_idx"], kc, g["q_pos"], sc, ws)
    qsa.score_paged(d, g["q_idx"], kcp, g["page_table"], g["q_pos"], scp, ws)
    _check_ok(qsa, ws)
    sc_h, scp_h = sc.cpu().numpy(), scp.cpu().numpy()
    for r in range(B):
        for j in range(4):
            n = O.n_full(spec.q_pos()[r][j])
            assert np.array_equal(sc_h[r, j, :n].view(np.uint32), scp_h[r, j, :n].view(np.uint32)), (r, j)
    # the fused step: the same scores, selection and output, bit for bit
    outs = []
    for paged in (False, True):
        out = torch.empty((B, 4, 16, 128), dtype=torch.bfloat16, device="cuda")
        scs = torch.empty((B, 4, mb), device="cuda")
        sb = torch.empty((B, 4, 512), dtype=torch.int32, device="cuda")
        sp = torch.empty((B, 4, 2051), dtype=torch.int32, device="cuda")
        fn = qsa.decode_paged if paged else qsa.decode
        fn(d, g["q_idx"], kcp if paged else kc, g["q"], g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"],
           g["page_table"], g["q_pos"], out, ws, scores=scs, sel_blk=sb, sel_pos=sp)
        _check_ok(qsa, ws)
        outs.append((bits(out), sp.cpu().numpy(), scs.cpu().numpy(), sb.cpu().numpy(), out.float().cpu().numpy()))
    assert np.array_equal(outs[0][1], outs[1][1])
    assert np.array_equal(outs[0][0], outs[1][0])
    # and the paged path against the oracle: compressed keys bit-exact, then
    # every row chained stage by stage (scores, selection, attention)
    _, _, sc_p, sb_p, out_p = outs[1]
    skipped = 0
    for r in range(B):
        npi = _oracle_request(spec, g, r)
        nb = O.n_full(max(spec.q_pos()[r]))
        b = np.arange(nb)
        assert np.array_equal(kcp_h[pt[r, b // bpp], b % bpp], npi["kc"][0, :nb]), r
        for j in range(4):
            skipped += _check_row_chain(spec, npi, j, sc_p[r, j], sb_p[r, j], outs[1][1][r, j], out_p[r, j])
    assert skipped <= 1


# --------------------------------------------------------------------------
# MTP draft steps reusing an earlier selection (qsa_draft_attn)
# --------------------------------------------------------------------------

def _draft_case(qsa, spec, g, q_sel, src, p_draft):
    """Selections of verify queries at q_sel (through qsa_decode), then draft
    queries at p_draft reusing rows src of them. Returns (out, sel_pos)."""
    gs = dict(g)
    gs["q_pos"] = torch.tensor(q_sel, dtype=torch.int32, device="cuda")
    _, sp = _run_decode(qsa, spec, gs)
    n_d = len(src[0])
    d = qsa.dims_for_spec(spec)
    d.n_q = n_d
    ws = qsa.make_workspace(d)
    qd = g["q"][:, :n_d].contiguous()
    out = torch.full((spec.batch, n_d, 16, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    qsa.draft_attn(d, qd, g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"], g["page_table"], sp,
                   gs["q_pos"], torch.tensor(src, dtype=torch.int32, device="cuda"),
                   torch.tensor(p_draft, dtype=torch.int32, device="cuda"), out, ws)
    return out, sp, ws


def _draft_ref(npi, spec, sp, q_sel, src, p_draft, r, jd):
    s = src[r][jd]
    ks = npi["k_scale"] if spec.kv_dtype == "fp8" else None
    vs = npi["v_scale"] if spec.kv_dtype == "fp8" else None
    return O.draft_attn(npi["q"][r, jd], npi["k_cache"], npi["v_cache"], npi["page_table"][r], sp[r, s],
                        q_sel[r][s], p_draft[r][jd], spec.kv_dtype, ks, vs)


@pytest.mark.parametrize("name", ["b2-h1-bf16", "b2-nq2-h1-fp8", "b2-nq3-h3"])
def test_draft_attn_parity(qsa, name):
    spec = SPECS[name]()
    inp = synth.make_inputs(spec)
    npi = to_numpy_inputs(inp)
    g = _dev(inp)
    # verify queries 70 positions before the cache's end leave room for drafts
    q_sel = [[p - 70 for p in row] for row in spec.q_pos()]
    last = spec.n_q - 1
    src = [[last, 0] for _ in range(spec.batch)]
    p_draft = [[row[last] + 60, row[0] + 5] for row in q_sel]  # gaps of 60 and 5
    out, sp, ws = _draft_case(qsa, spec, g, q_sel, src, p_draft)
    _check_ok(qsa, ws)
    got = out.float().cpu().numpy()
    spn = sp.cpu().numpy()
    for r in range(spec.batch):
        for jd in range(2):
            ref = _draft_ref(npi, spec, spn, q_sel, src, p_draft, r, jd)
            err = np.max(np.abs(got[r, jd] - ref))
            assert err <= ATOL[spec.kv_dtype], (r, jd, err)


def test_draft_attn_full_size_sampled(qsa):
    spec = synth.spec_for(2)
    inp = synth.make_inputs(spec)
    g = _dev(inp)
    q_sel = spec.q_pos()
    src = [[0] for _ in range(spec.batch)]
    p_draft = [[row[0] + 3] for row in q_sel]  # the step's last verify position, from the first one's selection
    out, sp, ws = _draft_case(qsa, spec, g, q_sel, src, p_draft)
    _check_ok(qsa, ws)
    got = out.float().cpu().numpy()
    spn = sp.cpu().numpy()
    npi = to_numpy_inputs({k: inp[k] for k in ("q", "k_cache", "v_cache", "k_scale", "v_scale", "page_table")})
    for r in (0, 13, 31):
        ref = _draft_ref(npi, spec, spn, q_sel, src, p_draft, r, 0)
        err = np.max(np.abs(got[r, 0] - ref))
        assert err <= ATOL["bf16"], (r, err)


def test_draft_attn_reports_a_draft_before_its_selection(qsa):
    spec = SPECS["b2-h1-bf16"]()
    inp = synth.make_inputs(spec)
    npi = to_numpy_inputs(inp)
    g = _dev(inp)
    q_sel = [[p - 70 for p in row] for row in spec.q_pos()]
    src = [[1], [0]]
    p_draft = [[q_sel[0][1] - 1], [q_sel[1][0] + 2]]  # request 0's draft lies before its selection's query
    out, sp, ws = _draft_case(qsa, spec, g, q_sel, src, p_draft)
    st, info = qsa.check_errors(ws)
    assert st == qsa.ERR_BAD_INDEX and info[0] == 4 and info[1] == 0, info
    got = out.float().cpu().numpy()
    assert np.all(got[0, 0] == 0.0)  # the bad row attends over nothing
    ref = _draft_ref(npi, spec, sp.cpu().numpy(), q_sel, src, p_draft, 1, 0)
    assert np.max(np.abs(got[1, 0] - ref)) <= ATOL["bf16"]


def test_decode_repeats_bit_exactly_on_one_workspace(qsa):
    # the workspace's counters and histograms must be left clean by every call
    spec = small_spec([9000, 3001, 5000], n_q=4, seed=36)
    g = _dev(synth.make_inputs(spec))
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    kc = torch.zeros((spec.batch, spec.max_blocks(), 1, 128), dtype=torch.bfloat16, device="cuda")
    qsa.compress_keys(d, g["idx_keys"], g["q_pos"], kc, ws)
    outs = []
    for _ in range(3):
        out = torch.empty((spec.batch, 4, 16, 128), dtype=torch.bfloat16, device="cuda")
        sp = torch.empty((spec.batch, 4, 2051), dtype=torch.int32, device="cuda")
        qsa.decode(d, g["q_idx"], kc, g["q"], g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"],
                   g["page_table"], g["q_pos"], out, ws, sel_pos=sp)
        outs.append((out.view(torch.int16).clone(), sp.clone()))
    _check_ok(qsa, ws)
    for o, s in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(s, outs[0][1])


def test_page_permutation_invariance(qsa):
    spec = small_spec([6000, 3000], n_q=4, seed=31)
    g = _dev(synth.make_inputs(spec))
    out0, sp0 = _run_decode(qsa, spec, g)
    perm = torch.randperm(spec.num_pages(), generator=torch.Generator().manual_seed(3)).cuda()
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(perm.numel(), device="cuda")
    g2 = dict(g)
    g2["k_cache"] = g["k_cache"][perm].contiguous()  # new slot i holds old page perm[i]
    g2["v_cache"] = g["v_cache"][perm].contiguous()
    pt = g["page_table"].clone()
    valid = pt >= 0
    pt[valid] = inv[pt[valid].long()].to(torch.int32)
    g2["page_table"] = pt
    out1, sp1 = _run_decode(qsa, spec, g2)
    assert torch.equal(sp0, sp1)
    assert torch.equal(out0.view(torch.int16), out1.view(torch.int16))


def test_causality_tokens_after_query_do_not_matter(qsa):
    spec = small_spec([5000], n_q=4, seed=32)
    g = _dev(synth.make_inputs(spec))
    out0, sp0 = _run_decode(qsa, spec, g)
    P = spec.page_size
    p0 = spec.q_pos()[0][0]
    g2 = {k: v.clone() for k, v in g.items()}
    for t in range(p0 + 1, spec.tokens()[0]):
        page = int(g["page_table"][0, t // P])
        g2["k_cache"][page, :, t % P] = 3.0
        g2["v_cache"][page, :, t % P] = -3.0
    g2["idx_keys"][0, p0 + 1 :] = 5.0
    out1, sp1 = _run_decode(qsa, spec, g2)
    assert torch.equal(sp0[0, 0], sp1[0, 0])
    assert torch.equal(out0[0, 0].view(torch.int16), out1[0, 0].view(torch.int16))
    assert not torch.equal(out0[0, 3].view(torch.int16), out1[0, 3].view(torch.int16))


def test_uniform_v_gives_v(qsa):
    spec = small_spec([4500], n_q=4, seed=33)
    g = _dev(synth.make_inputs(spec))
    row = torch.linspace(-2, 2, 128, device="cuda").to(torch.bfloat16)
    g["v_cache"][:] = row
    out, _ = _run_decode(qsa, spec, g)
    assert torch.max(torch.abs(out.float() - row.float())).item() <= 1e-2


def test_fp8_every_code_through_attention(qsa):
    # Attention over one selected position returns that position's V row. With
    # V rows holding every finite E4M3 code (the two NaN codes set to 0), the
    # kernel's packed FP8 -> FP16 widening must reproduce the OCP decode of each
    # code exactly (every E4M3 value is exact in FP16 and in BF16).
    spec = synth.Spec("fp8-codes", 1, 2, [40], 1, "fp8", True, 61)
    g = _dev(synth.make_inputs(spec))
    codes = np.arange(256, dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0
    pt = g["page_table"][0].long()
    page0 = int(pt[0].item())
    v = g["v_cache"]
    for h in range(spec.n_kv_heads):
        # token 0: codes 0..127; token 1: codes 128..255 (both KV heads, rolled so heads differ)
        v[page0, h, 0] = torch.from_numpy(np.roll(codes[:128], 17 * h).copy()).cuda()
        v[page0, h, 1] = torch.from_numpy(np.roll(codes[128:], 17 * h).copy()).cuda()
    g["k_scale"][:] = 1.0
    g["v_scale"][:] = 1.0
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    sel = torch.full((1, 2, 2051), -1, dtype=torch.int32, device="cuda")
    sel[0, 0, 0] = 0  # query 0 attends to token 0 only
    sel[0, 1, 0] = 1  # query 1 to token 1 only
    out = torch.empty((1, 2, 16, 128), dtype=torch.bfloat16, device="cuda")
    qsa.sparse_attn(d, g["q"], g["k_cache"], v, g["k_scale"], g["v_scale"], g["page_table"], sel, g["q_pos"], out,
                    ws)
    _check_ok(qsa, ws)
    got = out.float().cpu().numpy()
    vh = v.cpu().numpy()
    for j, tok in ((0, 0), (1, 1)):
        for hq in range(16):
            want = O.e4m3_to_f64(vh[page0, hq // 8, tok])
            assert np.array_equal(got[0, j, hq], want), (j, hq)


@pytest.mark.parametrize("kv", ["fp8", "bf16"])
@pytest.mark.parametrize("magnitude", [1e5, 1e-7])
def test_queries_outside_fp16_range(qsa, kv, magnitude):
    # The query is BF16 for either cache type. The FP8 path contracts in FP16,
    # whose range BF16 exceeds (65,504 at the top, normal down to 6.1e-5), so
    # queries near 1e5 (past FP16's largest value) and near 1e-7 (FP16
    # subnormals) must still match the oracle. Tiny queries get a large
    # softmax scale, so that their logits are of order one and every bit of
    # the query matters; large ones make each head's softmax nearly one-hot.
    spec = small_spec([4000, 2600], n_q=2, kv_dtype=kv, seed=71)
    inp = synth.make_inputs(spec)
    q = (inp["q"].float() * magnitude).to(torch.bfloat16)
    q[1, 1, 8:] = inp["q"][1, 1, 8:]  # heads of another magnitude in the same call (KV group 1)
    inp["q"] = q
    npi = to_numpy_inputs(inp)
    sm_scale = (1.0 / magnitude) / math.sqrt(128) if magnitude < 1 else 1.0 / math.sqrt(128)
    d = qsa.dims_for_spec(spec)
    d.sm_scale = sm_scale
    ws = qsa.make_workspace(d)
    g = _dev(inp)
    rng = np.random.default_rng(72)
    sel = np.full((2, 2, 2051), -1, np.int32)
    for r in range(2):
        for j in range(2):
            p = spec.q_pos()[r][j]
            sel[r, j] = np.sort(rng.choice(p + 1, 2051, replace=False))
    out = torch.full((2, 2, 16, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    qsa.sparse_attn(d, g["q"], g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"], g["page_table"],
                    torch.from_numpy(sel).cuda(), g["q_pos"], out, ws)
    _check_ok(qsa, ws)
    got = out.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    fp8 = kv == "fp8"
    for r in range(2):
        for j in range(2):
            ref = O.sparse_attn(npi["q"][r, j], npi["k_cache"], npi["v_cache"], npi["page_table"][r], sel[r, j],
                                kv, npi["k_scale"] if fp8 else None, npi["v_scale"] if fp8 else None,
                                sm_scale=float(np.float32(sm_scale)))
            err = np.max(np.abs(got[r, j] - ref))
            assert err <= ATOL[kv], (r, j, err)


def test_bf16_single_position_returns_its_v_row_exactly(qsa):
    # softmax over one position has weight 1: the output is the V row itself
    spec = synth.Spec("bf16-one", 1, 2, [40], 1, "bf16", True, 62)
    g = _dev(synth.make_inputs(spec))
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    sel = torch.full((1, 2, 2051), -1, dtype=torch.int32, device="cuda")
    sel[0, 0, 0] = 5
    sel[0, 1, 0] = 41  # the query's own token
    out = torch.empty((1, 2, 16, 128), dtype=torch.bfloat16, device="cuda")
    qsa.sparse_attn(d, g["q"], g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"], g["page_table"], sel,
                    g["q_pos"], out, ws)
    _check_ok(qsa, ws)
    pt = g["page_table"][0]
    for j, tok in ((0, 5), (1, 41)):
        page = int(pt[tok // spec.page_size].item())
        for hq in range(16):
            row = g["v_cache"][page, hq // 8, tok % spec.page_size]
            assert torch.equal(out[0, j, hq].view(torch.int16), row.view(torch.int16)), (j, hq)


@pytest.mark.parametrize("h", [1, 2])
def test_one_hot_query_reads_one_key_dimension(qsa, h):
    # closed form: a query equal to 1 at (head hh, dim dd) and 0 elsewhere
    # scores each block with exactly its compressed key's (hh, dd) component
    spec = small_spec([3001, 1498], n_q=4, n_idx_heads=h, seed=63)
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    mb = spec.max_blocks()
    kc = synth.normal_bf16((spec.batch, mb, h, 128), 64, "cuda")
    picks = [(j % h, (37 * j + 5) % 128) for j in range(4)]
    q_idx = torch.zeros((spec.batch, 4, h, 128), dtype=torch.bfloat16, device="cuda")
    for j, (hh, dd) in enumerate(picks):
        q_idx[:, j, hh, dd] = 1.0
    q_pos = torch.tensor(spec.q_pos(), dtype=torch.int32, device="cuda")
    scores = torch.full((spec.batch, 4, mb), float("nan"), device="cuda")
    qsa.score(d, q_idx, kc, q_pos, scores, ws)
    _check_ok(qsa, ws)
    for r in range(spec.batch):
        for j, (hh, dd) in enumerate(picks):
            nb = O.n_full(spec.q_pos()[r][j])
            assert torch.equal(scores[r, j, :nb], kc[r, :nb, hh, dd].float()), (r, j)


def test_compressed_key_of_identical_tokens_is_the_token_key(qsa):
    # closed form: the FP32 mean of four equal BF16 values is that value exactly
    spec = small_spec([2001, 777], n_q=2, n_idx_heads=2, seed=65)
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    mb = spec.max_blocks()
    base = synth.normal_bf16((spec.batch, mb, 2, 128), 66, "cuda")
    idx_keys = base.repeat_interleave(4, dim=1).contiguous()  # [B][4 mb][2][128]: 4 equal tokens per block
    q_pos = torch.tensor(spec.q_pos(), dtype=torch.int32, device="cuda")
    kc = torch.zeros_like(base)
    qsa.compress_keys(d, idx_keys, q_pos, kc, ws)
    _check_ok(qsa, ws)
    for r in range(spec.batch):
        nb = O.n_full(max(spec.q_pos()[r]))
        assert torch.equal(kc[r, :nb].view(torch.int16), base[r, :nb].view(torch.int16)), r


def test_chunk_one_hot_queries_read_one_key_dimension(qsa):
    spec = small_spec([3001], n_q=1, n_idx_heads=2, seed=67)
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    mb = spec.max_blocks()
    n_chunk = 70  # two query tiles, the second ragged
    kc = synth.normal_bf16((1, mb, 2, 128), 68, "cuda")
    q_idx = torch.zeros((1, n_chunk, 2, 128), dtype=torch.bfloat16, device="cuda")
    picks = [(i % 2, (29 * i + 3) % 128) for i in range(n_chunk)]
    for i, (hh, dd) in enumerate(picks):
        q_idx[0, i, hh, dd] = 1.0
    pos = [2999 - 7 * i for i in range(n_chunk)]
    q_pos = torch.tensor([pos], dtype=torch.int32, device="cuda")
    scores = torch.full((1, n_chunk, mb), float("nan"), device="cuda")
    qsa.score_chunk(d, q_idx, kc, q_pos, scores, ws)
    _check_ok(qsa, ws)
    for i, (hh, dd) in enumerate(picks):
        nb = O.n_full(pos[i])
        assert torch.equal(scores[0, i, :nb], kc[0, :nb, hh, dd].float()), i
        assert torch.all(torch.isnan(scores[0, i, nb:]))


@pytest.mark.parametrize("config,kv", [(1, "bf16"), (3, "fp8")])
def test_zero_keys_give_the_mean_of_v_over_the_selection(qsa, config, kv):
    # closed form: with every key zero all scores tie, so each output is the
    # plain mean of V over the query's selected positions; at batch 1 a unit is
    # cut into about 17 pieces, so this checks the merge of pieces as well
    spec = synth.spec_for(config, batch=1) if config == 3 else synth.spec_for(config)
    g = synth.make_inputs(spec, device="cuda")
    g["k_cache"].zero_()
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    rng = np.random.default_rng(69)
    sel = torch.full((1, 4, 2051), -1, dtype=torch.int32)
    for j in range(4):
        p = spec.q_pos()[0][j]
        pick = np.sort(rng.choice(p + 1, size=2051, replace=False))
        sel[0, j] = torch.from_numpy(pick.astype(np.int32))
    sel = sel.cuda()
    out = torch.empty((1, 4, 16, 128), dtype=torch.bfloat16, device="cuda")
    qsa.sparse_attn(d, g["q"], g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"], g["page_table"], sel,
                    g["q_pos"], out, ws)
    _check_ok(qsa, ws)
    P = spec.page_size
    pt = g["page_table"][0].long()
    for j in range(4):
        t = sel[0, j].long()
        pages, slots = pt[t // P], t % P
        for kvh in range(2):
            rows = g["v_cache"][pages, kvh, slots]
            if kv == "fp8":
                vals = torch.from_numpy(O.e4m3_to_f64(rows.cpu().numpy())) * float(g["v_scale"][kvh].item())
            else:
                vals = rows.double().cpu()
            mean = vals.mean(dim=0)
            for hq in range(8 * kvh, 8 * kvh + 8):
                err = (out[0, j, hq].double().cpu() - mean).abs().max().item()
                assert err <= ATOL[kv], (j, hq, err)


def test_device_errors_are_reported_not_fatal(qsa):
    spec = small_spec([3000, 2000], n_q=2, seed=34)
    g = _dev(synth.make_inputs(spec))
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    # a query position past the buffers
    bad = g["q_pos"].clone()
    bad[1, 1] = 4 * spec.max_blocks() + 100
    kc = torch.zeros((2, spec.max_blocks(), 1, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((2, 2, 16, 128), dtype=torch.bfloat16, device="cuda")
    qsa.decode(d, g["q_idx"], kc, g["q"], g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"],
               g["page_table"], bad, out, ws)
    st, info = qsa.check_errors(ws)
    assert st == qsa.ERR_BAD_INDEX and info[0] == 1 and info[1] == 1 and info[2] == 1
    assert torch.all(out[1, 1] == 0)
    assert qsa.check_errors(ws)[0] == qsa.OK  # cleared
    # a page id outside the cache
    pt = g["page_table"].clone()
    pt[0, 3] = spec.num_pages() + 5
    sel = torch.full((2, 2, 2051), -1, dtype=torch.int32, device="cuda")
    sel[0, 0, :10] = torch.arange(190, 200, dtype=torch.int32)
    sel[1, :, 0] = 5
    qsa.sparse_attn(d, g["q"], g["k_cache"], g["v_cache"], None, None, pt, sel, g["q_pos"], out, ws)
    st, info = qsa.check_errors(ws)
    assert st == qsa.ERR_BAD_INDEX and info[0] == 2
    # a selected position after its query (causality violation)
    sel2 = sel.clone()
    sel2[0, 0, :10] = 2999 + 5
    qsa.sparse_attn(d, g["q"], g["k_cache"], g["v_cache"], None, None, g["page_table"], sel2, g["q_pos"], out, ws)
    st, info = qsa.check_errors(ws)
    assert st == qsa.ERR_BAD_INDEX and info[0] == 3 and info[3] == 3004
    # the context still works afterwards
    out2, _ = _run_decode(qsa, spec, g)
    assert torch.isfinite(out2.float()).all()


def test_synchronous_argument_errors(qsa):
    spec = small_spec([3000], n_q=1, seed=35)
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    small = torch.zeros(256, dtype=torch.uint8, device="cuda")
    f = torch.zeros((1, 1, spec.max_blocks()), device="cuda")
    qp = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    sb = torch.zeros((1, 1, 512), dtype=torch.int32, device="cuda")
    sp = torch.zeros((1, 1, 2051), dtype=torch.int32, device="cuda")
    import ctypes

    st = qsa.lib.qsa_topk(ctypes.byref(d), ctypes.c_void_p(f.data_ptr()), ctypes.c_void_p(qp.data_ptr()),
                          ctypes.c_void_p(sb.data_ptr()), ctypes.c_void_p(sp.data_ptr()),
                          ctypes.c_void_p(small.data_ptr()), 256, None)
    assert st == qsa.ERR_WORKSPACE
    st = qsa.lib.qsa_topk(ctypes.byref(d), None, ctypes.c_void_p(qp.data_ptr()), ctypes.c_void_p(sb.data_ptr()),
                          ctypes.c_void_p(sp.data_ptr()), ctypes.c_void_p(ws.data_ptr()), ws.numel(), None)
    assert st == qsa.ERR_INVALID_ARG
    d2 = qsa.dims_for_spec(spec)
    d2.head_dim = 64
    st = qsa.lib.qsa_topk(ctypes.byref(d2), ctypes.c_void_p(f.data_ptr()), ctypes.c_void_p(qp.data_ptr()),
                          ctypes.c_void_p(sb.data_ptr()), ctypes.c_void_p(sp.data_ptr()),
                          ctypes.c_void_p(ws.data_ptr()), ws.numel(), None)
    assert st == qsa.ERR_UNSUPPORTED
    with pytest.raises(ValueError):
        qsa.topk(d, f.cpu(), qp, sb, sp, ws)  # host tensors are refused: no CPU path
