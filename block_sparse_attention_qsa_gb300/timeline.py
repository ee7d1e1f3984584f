"""Phase timeline of the fused QSA step (score -> select -> attention).

    python -m block_sparse_attention_qsa_gb300.timeline [--config 2] [--batch 32] [--ctx N]
        [--steps 8] [--warmup 2] [--json]

Builds the tracing library (libqsa_trace.so: the product sources compiled
with -DQSA_TRACE, whose score, selector and attention kernels stamp
%globaltimer per CTA at their start, the release of their wait on the
previous kernel, the end of their main work and their end), runs qsa_decode
on a seeded synthetic workload with L2 flushed before every step, reads the
stamps back with qsa_trace_read and prints, per kernel, when its CTAs start,
are released, finish their work and end (µs from the first score CTA's
start; medians over the measured steps of each step's min / p50 / max), the
hand-offs between the kernels and, for attention, how the CTAs that share an
SM finish relative to each other. Run it in its own process: the binding
loads one library per process.

The stamps cost a few instructions per CTA; the product library has none.
"""

from __future__ import annotations

import argparse
import json
import os
import sys

import numpy as np

SLOT_START, SLOT_RELEASED, SLOT_WORK, SLOT_END, SLOT_SM, SLOT_PUBLISHED, SLOT_MERGED = range(7)
KERNELS = ("score", "topk", "attn")


def live_records(table: np.ndarray) -> np.ndarray:
    """Rows of a trace table that belong to a CTA of the launch (start stamped)."""
    return table[table[:, SLOT_START] > 0]


def _stats(v: np.ndarray):
    v = v[np.isfinite(v)]
    if v.size == 0:
        return None
    return [float(v.min()), float(np.median(v)), float(v.max())]


def summarize_step(tables: dict) -> dict:
    """One step's stamps (kernel name -> [CTAs][slots] uint64) -> µs relative
    to the first score CTA's start: per kernel and slot [min, p50, max], the
    hand-offs (last CTA end of one kernel -> first release of the next) and
    the attention CTAs' spread of main-work ends within and across SMs."""
    recs = {k: live_records(t) for k, t in tables.items()}
    t0 = min(int(r[:, SLOT_START].min()) for r in recs.values() if len(r))
    out = {"ctas": {k: int(len(r)) for k, r in recs.items()}}

    def rel(r, slot):
        v = r[:, slot].astype(np.float64)
        v[v == 0] = np.nan
        return (v - t0) / 1e3

    for k, r in recs.items():
        out[k] = {name: _stats(rel(r, s)) for name, s in
                  (("start", SLOT_START), ("released", SLOT_RELEASED), ("work_done", SLOT_WORK), ("end", SLOT_END))}
    hand = {}
    for a, b in (("score", "topk"), ("topk", "attn")):
        if len(recs[a]) and len(recs[b]):
            hand[f"{a}->{b}"] = float(np.nanmin(rel(recs[b], SLOT_RELEASED)) - np.nanmax(rel(recs[a], SLOT_END)))
    out["handoff_us"] = hand
    ra = recs["attn"]
    if len(ra):
        work = rel(ra, SLOT_WORK)
        sm = ra[:, SLOT_SM].astype(np.int64) - 1
        per_sm = {}
        for s, w in zip(sm, work):
            if s >= 0 and np.isfinite(w):
                per_sm.setdefault(int(s), []).append(float(w))
        within = [max(v) - min(v) for v in per_sm.values() if len(v) > 1]
        means = [float(np.mean(v)) for v in per_sm.values()]
        out["attn_sm"] = {
            "sms": len(per_sm),
            "ctas_per_sm_max": max((len(v) for v in per_sm.values()), default=0),
            "within_sm_spread_p50_p90_max": ([float(np.median(within)), float(np.percentile(within, 90)),
                                              float(np.max(within))] if within else None),
            "sm_mean_min_max": [min(means), max(means)] if means else None,
            "cta_work_done_max": float(np.nanmax(work)),
        }
        pub = rel(ra, SLOT_PUBLISHED)
        mer = rel(ra, SLOT_MERGED)
        both = np.isfinite(pub) & np.isfinite(mer)
        lag = pub - work  # a CTA whose last segment was a whole unit published before it: not counted
        lag[lag < 0] = np.nan
        out["attn_pieces"] = {"published": int(np.isfinite(pub).sum()), "merges": int(np.isfinite(mer).sum()),
                              "publish_time": _stats(lag),
                              "merge_time": _stats(mer[both] - pub[both]),
                              "last_merge_end": _stats(mer)}
    return out


def check_order(step: dict, tol_us: float = 0.05) -> list:
    """Ordering the chain guarantees, as a list of violations (empty: none):
    within every kernel start <= released <= work done <= end, and each
    dependent kernel's first release after the previous kernel's last end."""
    bad = []
    for k in KERNELS:
        s = step.get(k)
        if not s or not s["start"]:
            continue
        seq = [s[n] for n in ("start", "released", "work_done", "end") if s[n]]
        for a, b in zip(seq, seq[1:]):
            if b[0] < a[0] - tol_us or b[2] < a[2] - tol_us:
                bad.append(f"{k}: phases out of order {a} -> {b}")
    for h, v in step["handoff_us"].items():
        if v < -tol_us:
            bad.append(f"{h}: released {-v:.3f} us before the previous kernel ended")
    return bad


def median_summary(steps: list) -> dict:
    """Element-wise median over steps of the numeric leaves of summarize_step."""
    def med(vals):
        if all(isinstance(v, (int, float)) for v in vals):
            return float(np.median(vals))
        if all(isinstance(v, list) for v in vals) and len({len(v) for v in vals}) == 1:
            return [med([v[i] for v in vals]) for i in range(len(vals[0]))]
        if all(isinstance(v, dict) for v in vals):
            return {k: med([v[k] for v in vals]) for k in vals[0]}
        return vals[0]
    return med(steps)


def markdown(summary: dict, title: str) -> str:
    f = lambda v: "—" if v is None else " / ".join(f"{x:.2f}" for x in v)  # noqa: E731
    lines = [f"### {title}", "",
             "µs from the first score CTA's start; each cell min / p50 / max over the kernel's CTAs (median over steps)",
             "", "| kernel | CTAs | start | released | work done | end |", "|---|---|---|---|---|---|"]
    for k in KERNELS:
        s = summary[k]
        lines.append(f"| {k} | {summary['ctas'][k]:.0f} | {f(s['start'])} | {f(s['released'])} | "
                     f"{f(s['work_done'])} | {f(s['end'])} |")
    lines.append("")
    lines.append("hand-offs (first release minus the previous kernel's last end): " +
                 ", ".join(f"{k} {v:.2f} µs" for k, v in summary["handoff_us"].items()))
    if "attn_sm" in summary:
        a = summary["attn_sm"]
        lines.append(f"attention, per SM ({a['sms']:.0f} SMs, up to {a['ctas_per_sm_max']:.0f} CTAs each): spread of "
                     f"the CTAs' work ends within an SM p50 / p90 / max {f(a['within_sm_spread_p50_p90_max'])} µs; "
                     f"SM means {f(a['sm_mean_min_max'])} µs; last CTA {a['cta_work_done_max']:.2f} µs")
        p = summary["attn_pieces"]
        lines.append(f"attention pieces: {p['published']:.0f} published ({f(p['publish_time'])} µs from the "
                     f"CTA's work end to its ticket), {p['merges']:.0f} merges ({f(p['merge_time'])} µs from the "
                     f"ticket to the merged output), last merge ends {f(p['last_merge_end'])} µs")
    return "\n".join(lines)


def collect(config: int, batch, ctx, steps: int, warmup: int):
    """Runs the traced step; returns (per-step summaries, workload name)."""
    from block_sparse_attention_qsa_gb300 import _build

    os.environ["QSA_LIBRARY"] = _build.build(trace=True)
    if "block_sparse_attention_qsa_gb300.qsa" in sys.modules:
        raise RuntimeError("the binding is already loaded with another library: run the timeline in its own process")
    import torch

    from block_sparse_attention_qsa_gb300 import qsa, synth

    spec = synth.spec_for(config, batch=batch, ctx=ctx)
    g = synth.make_inputs(spec, device="cuda")
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    kc = torch.zeros((spec.batch, spec.max_blocks(), spec.n_idx_heads, spec.head_dim), dtype=torch.bfloat16,
                     device="cuda")
    qsa.compress_keys(d, g["idx_keys"], g["q_pos"], kc, ws)
    out = torch.empty((spec.batch, spec.n_q, d.n_q_heads, spec.head_dim), dtype=torch.bfloat16, device="cuda")
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    wbuf = torch.empty(2 * l2 // 4, dtype=torch.float32, device="cuda")
    rbuf = torch.zeros(2 * l2 // 4, dtype=torch.float32, device="cuda")
    sink = torch.empty((), device="cuda")
    ids = (qsa.TRACE_SCORE, qsa.TRACE_TOPK, qsa.TRACE_ATTN)
    res = []
    for it in range(warmup + steps):
        for k in ids:
            qsa.trace_read(k, 0, clear=True)
        wbuf.zero_()
        torch.sum(rbuf, dim=0, out=sink)
        torch.cuda.synchronize()
        qsa.decode(d, g["q_idx"], kc, g["q"], g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"],
                   g["page_table"], g["q_pos"], out, ws)
        torch.cuda.synchronize()
        st, info = qsa.check_errors(ws)
        if st != qsa.OK:
            raise RuntimeError(f"step reported {info}")
        if it >= warmup:
            res.append(summarize_step({n: qsa.trace_read(k) for n, k in zip(KERNELS, ids)}))
    return res, spec.name


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--config", type=int, default=2)
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--ctx", type=int, default=None)
    ap.add_argument("--steps", type=int, default=8)
    ap.add_argument("--warmup", type=int, default=2)
    ap.add_argument("--json", action="store_true", help="print the per-step summaries as one JSON line")
    a = ap.parse_args(argv)
    steps, name = collect(a.config, a.batch, a.ctx, a.steps, a.warmup)
    if a.json:
        print(json.dumps({"workload": name, "steps": steps, "violations": [check_order(s) for s in steps]}))
        return
    print(markdown(median_summary(steps), f"{name}, {a.steps} steps"))
    bad = [v for s in steps for v in check_order(s)]
    print("\nordering checks: " + ("all hold" if not bad else "; ".join(bad)))


if __name__ == "__main__":
    ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    main()
