"""The phase-timeline tool (block_sparse_attention_qsa_gb300/timeline.py) and
the tracing entry point qsa_trace_read.

CPU: the summary of per-CTA stamps (hand-offs between the chained kernels,
per-SM spread of the attention CTAs) on synthetic stamps, and the ordering
check catching a dependent released before its producer ended. The product
library answers qsa_trace_read with QSA_ERR_UNSUPPORTED and rejects bad
arguments without touching a device.

GPU: the tracing build of the library runs the fused step; in every step each
kernel's CTAs start, are released, finish and end in that order, and each
dependent kernel is released only after the last CTA of the kernel before it
ended (the programmatic-dependent-launch chain keeps its promise).
"""

import json
import os
import subprocess
import sys

import numpy as np
import pytest

from block_sparse_attention_qsa_gb300 import timeline as T

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _table(n, t0, released, work, end, sm_of=lambda i: i % 152):
    a = np.zeros((4096, 8), np.uint64)
    for i in range(n):
        a[i, T.SLOT_START] = t0 + 10 * i
        a[i, T.SLOT_RELEASED] = released + 10 * i
        a[i, T.SLOT_WORK] = work + 100 * i
        a[i, T.SLOT_END] = end + 100 * i
        a[i, T.SLOT_SM] = sm_of(i) + 1
    return a


def _steps():
    score = _table(152, 1_000_000, 1_000_000, 1_020_000, 1_020_100)  # ends by 1,035,200 ns
    topk = _table(128, 1_030_000, 1_036_000, 1_045_000, 1_045_100)   # ends by 1,057,800 ns
    attn = _table(456, 1_040_000, 1_059_000, 1_090_000, 1_091_000, sm_of=lambda i: i // 3)
    attn[5, T.SLOT_PUBLISHED] = 1_095_000
    attn[7, T.SLOT_MERGED] = 1_097_000
    return {"score": score, "topk": topk, "attn": attn}


def test_summary_of_synthetic_stamps():
    s = T.summarize_step(_steps())
    assert s["ctas"] == {"score": 152, "topk": 128, "attn": 456}
    assert s["score"]["start"][0] == 0.0
    assert s["handoff_us"]["score->topk"] == pytest.approx(1036.0 - 1035.2)
    assert s["handoff_us"]["topk->attn"] == pytest.approx(1059.0 - 1057.8)
    a = s["attn_sm"]
    assert a["sms"] == 152 and a["ctas_per_sm_max"] == 3
    # CTAs 3k, 3k+1, 3k+2 share SM k; their work ends are 100 ns apart
    assert a["within_sm_spread_p50_p90_max"] == pytest.approx([0.2, 0.2, 0.2])
    assert a["cta_work_done_max"] == pytest.approx((1_090_000 + 45_500 - 1_000_000) / 1e3)
    assert s["attn_pieces"]["published"] == 1 and s["attn_pieces"]["merges"] == 1
    assert T.check_order(s) == []
    m = T.median_summary([s, s, s])
    assert m["handoff_us"]["topk->attn"] == pytest.approx(s["handoff_us"]["topk->attn"])
    assert "attention, per SM" in T.markdown(m, "synthetic")


def test_order_check_catches_an_early_release():
    st = _steps()
    st["attn"][:456, T.SLOT_RELEASED] = 1_050_000  # before the selector's last CTA ended
    bad = T.check_order(T.summarize_step(st))
    assert any("topk->attn" in b for b in bad)
    st = _steps()
    st["score"][3, T.SLOT_END] = 1_000_001  # a CTA ending before its work was done
    bad = T.check_order(T.summarize_step(st))
    assert any(b.startswith("score: phases out of order") for b in bad)


def test_product_library_has_no_trace():
    import __graft_entry__

    __graft_entry__.build()
    from block_sparse_attention_qsa_gb300 import qsa

    if os.path.basename(qsa.LIB_PATH) != "libqsa.so":
        pytest.skip("another build is loaded")
    lib = qsa.lib
    assert lib.qsa_trace_read(qsa.TRACE_ATTN, None, 0, 1) == qsa.ERR_UNSUPPORTED
    assert lib.qsa_trace_read(7, None, 0, 0) == qsa.ERR_INVALID_ARG
    assert lib.qsa_trace_read(qsa.TRACE_SCORE, None, 1, 0) == qsa.ERR_INVALID_ARG
    assert lib.qsa_trace_read(qsa.TRACE_SCORE, None, qsa.TRACE_CTAS + 1, 0) == qsa.ERR_INVALID_ARG
    with pytest.raises(qsa.QSAError):
        qsa.trace_read(qsa.TRACE_TOPK, 4)


@pytest.mark.gpu
@pytest.mark.parametrize("args", [["--config", "0"], ["--config", "2", "--batch", "4"], ["--config", "3", "--batch", "32"]])
def test_traced_step_keeps_the_chain_order(args):
    cmd = [sys.executable, "-m", "block_sparse_attention_qsa_gb300.timeline", *args, "--steps", "3", "--warmup", "1",
           "--json"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert len(res["steps"]) == 3
    for step, bad in zip(res["steps"], res["violations"]):
        assert bad == [], bad
        assert all(step["ctas"][k] > 0 for k in T.KERNELS)
        assert set(step["handoff_us"]) == {"score->topk", "topk->attn"}
        assert step["attn_sm"]["ctas_per_sm_max"] >= 1
