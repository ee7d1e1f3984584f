"""qsa_sparse_attn_noalloc: sparse attention for callers that cannot allocate
device memory (no cudaMalloc allowed where they run, a fixed memory pool, a
plugin handed tensors but no allocator). It keeps its scratch in the
library's own static device array instead of a workspace, so the test checks
that it gives the same output as qsa_sparse_attn, and keeps giving it when
called again on the array the previous call left behind.

This file is collected last on purpose: a failure here should not stop a run
before every other test has run.
"""

import pytest
import torch

from block_sparse_attention_qsa_gb300 import synth
from tests._util import small_spec

pytestmark = pytest.mark.gpu

ATOL = {"bf16": 1e-2, "fp8": 3e-2}  # the tolerances of the attention parity tests


@pytest.fixture(scope="module")
def qsa():
    import __graft_entry__

    __graft_entry__.build()
    from block_sparse_attention_qsa_gb300 import qsa as q

    return q


def _selection(qsa, spec, g, d, ws):
    kc = torch.zeros((spec.batch, spec.max_blocks(), spec.n_idx_heads, 128), dtype=torch.bfloat16, device="cuda")
    qsa.compress_keys(d, g["idx_keys"], g["q_pos"], kc, ws)
    out = torch.empty((spec.batch, spec.n_q, 16, 128), dtype=torch.bfloat16, device="cuda")
    sel = torch.empty((spec.batch, spec.n_q, 2051), dtype=torch.int32, device="cuda")
    qsa.decode(d, g["q_idx"], kc, g["q"], g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"],
               g["page_table"], g["q_pos"], out, ws, sel_pos=sel)
    return sel


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_noalloc_matches_workspace_entry_point_on_two_calls(qsa, kv):
    spec = small_spec([9000, 3001, 2050], n_q=4, kv_dtype=kv, seed=91)
    g = {k: v.cuda() for k, v in synth.make_inputs(spec).items()}
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    sel = _selection(qsa, spec, g, d, ws)
    ref = torch.empty((spec.batch, spec.n_q, 16, 128), dtype=torch.bfloat16, device="cuda")
    qsa.sparse_attn(d, g["q"], g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"], g["page_table"], sel,
                    g["q_pos"], ref, ws)
    st, info = qsa.check_errors(ws)
    assert st == qsa.OK, info
    for call in range(2):  # the second call starts from what the first left in the scratch
        out = torch.full_like(ref, float("nan"))
        qsa.sparse_attn_noalloc(d, g["q"], g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"],
                                g["page_table"], sel, g["q_pos"], out)
        torch.cuda.synchronize()
        err = (out.float() - ref.float()).abs().max().item()
        assert err <= ATOL[kv], (call, err)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_noalloc_with_fewer_ctas_to_fit_the_array(qsa, kv):
    # 480 requests x 4 queries = 1,920 rows: their resolved cache rows (8 KB
    # each) fill most of the 16 MiB array, so the call lowers the CTA count
    # (456 CTAs -> about 120) to fit the softmax partials into what is left,
    # which cuts the rows' attention into pieces at other places. Sampled rows
    # against the oracle, every row against qsa_sparse_attn, on two calls.
    import math

    import numpy as np

    from oracle import qsa_oracle as O
    from tests._util import bits

    B = 480
    spec = synth.Spec("noalloc-b480", B, 4, [2200 + 97 * (r % 7) for r in range(B)], 1, kv, True, 93)
    g = synth.make_inputs(spec, device="cuda", with_index_keys=False)
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    # per row, 2,051 distinct causal positions drawn at random, ascending
    gen = torch.Generator(device="cuda").manual_seed(94)
    pos = g["q_pos"].view(-1, 1).long()
    keys = torch.rand((B * 4, 3000), generator=gen, device="cuda")
    keys[torch.arange(3000, device="cuda").view(1, -1) > pos] = 2.0  # past the query: never picked
    sel = torch.sort(torch.argsort(keys, dim=1)[:, :2051], dim=1).values.to(torch.int32).view(B, 4, 2051)
    assert int(sel.max()) <= max(max(p) for p in spec.q_pos())
    ref = torch.empty((B, 4, 16, 128), dtype=torch.bfloat16, device="cuda")
    qsa.sparse_attn(d, g["q"], g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"], g["page_table"], sel,
                    g["q_pos"], ref, ws)
    st, info = qsa.check_errors(ws)
    assert st == qsa.OK, info
    for call in range(2):
        out = torch.full_like(ref, float("nan"))
        qsa.sparse_attn_noalloc(d, g["q"], g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"],
                                g["page_table"], sel, g["q_pos"], out)
        torch.cuda.synchronize()
        err = (out.float() - ref.float()).abs().max().item()
        assert err <= ATOL[kv], (call, err)
    got = out.float().cpu().numpy()
    fp8 = kv == "fp8"
    ks, vs = g["k_scale"].cpu().numpy(), g["v_scale"].cpu().numpy()
    for r, j in ((0, 0), (1, 3), (239, 2), (478, 1), (479, 3)):
        npg = spec.pages_per_request()[r]
        pages = g["page_table"][r, :npg].long()
        want = O.sparse_attn(bits(g["q"][r, j]), bits(g["k_cache"][pages]), bits(g["v_cache"][pages]),
                             np.arange(npg), sel[r, j].cpu().numpy(), kv, ks if fp8 else None,
                             vs if fp8 else None, 1.0 / math.sqrt(128))
        err = np.max(np.abs(got[r, j] - want))
        assert err <= ATOL[kv], (r, j, err)
