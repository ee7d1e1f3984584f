"""Benchmark of the QSA decode / MTP-verify step on GB300.

Default workload: MTP verify at batch 32, 4 verify queries per request,
contexts 50,000 + 800*t tokens (t uniform in 0..14, seeded), 1 index head of
128, 16/2 attention heads of 128, paged BF16 KV (pages of 64, seeded random
page permutation). One step = qsa_decode: FP32 block scores -> top-512
selection + unfilled block (width 2,051) -> sparse attention, PDL-chained.

Prints one JSON line. `value` is HBM GB/s of algorithmic bytes (compressed
keys read once per request + K/V of the union of each request's selected
positions) over the device time of the step; `latency_us` is the step time.
L2 is flushed before every timed step (a write of twice its size, then a read
of another buffer that size, so the lines the write leaves dirty are written
back before the timed region); the flush is outside the timed events.

The same run also times a sweep (batches 1-32 of the 50K-token verify step
with BF16 KV, batches 1 and 32 with FP8 KV, and the long-context workload at
131,072 tokens) and the CPU oracle, on one core and on all of the host's
cores.

    python bench.py [--steps K] [--warmup W] [--config {0,1,2,3,4}] [--impl reference]
"""

import os

# the oracle baseline runs single-threaded (numpy's BLAS included)
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import re  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_sparse_attention_qsa_gb300 import synth  # noqa: E402

METRIC = "QSA step latency (µs) and HBM GB/s, batch 1–32, 50K ctx, 4 verify queries"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0  # the HBM3e figure the target is also quoted against (nominal, not measured)

# the sweep of the metric: (config, batch, context) beside the headline
SWEEP = [(2, 1, None), (2, 2, None), (2, 4, None), (2, 8, None), (2, 16, None), (2, 32, None),
         (3, 1, None), (3, 32, None), (4, 1, 131072), (4, 8, 131072)]


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=2)
    ap.add_argument("--batch", type=int, default=None)
    ap.add_argument("--ctx", type=int, default=None)
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="seconds of oracle work in the CPU baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-flush", action="store_true", help="warm-L2 numbers (reported as such)")
    ap.add_argument("--step-only", action="store_true",
                    help="only the warm-up and timed fused steps (for profiler captures)")
    ap.add_argument("--no-graph", action="store_true",
                    help="time direct calls instead of replaying the step captured as a CUDA graph")
    ap.add_argument("--paged-kc", action="store_true",
                    help="the compressed keys in the KV cache's pages (qsa_decode_paged)")
    ap.add_argument("--chunk", type=int, default=0,
                    help="time chunked scoring instead: one request (config 1's 50K context), this many queries")
    ap.add_argument("--draft", action="store_true",
                    help="time an MTP draft step instead: one draft query per request attending over the "
                         "selection of the request's first verify query plus the 3 positions after it")
    ap.add_argument("--no-sweep", action="store_true", help="skip the batch / cache-type sweep")
    ap.add_argument("--sweep-steps", type=int, default=100, help="timed steps per sweep entry")
    ap.add_argument("--cpu-requests", type=int, default=8,
                    help="requests of the batch saved for the all-core oracle timing (cycled)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (replicas: every rank runs its own independent batch)
# ---------------------------------------------------------------------------

def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# algorithmic bytes
# ---------------------------------------------------------------------------

def kv_row_bytes(spec):
    return spec.n_kv_heads * spec.head_dim * (1 if spec.kv_dtype == "fp8" else 2)


def kc_bytes(spec):
    return sum(max(1, (max(qp) + 1) // 4) * spec.n_idx_heads * spec.head_dim * 2 for qp in spec.q_pos())


def kv_bytes(spec, sel_pos_host):
    """(union over each request's queries, plain sum) of selected K+V bytes."""
    union = 0
    total = 0
    for r in range(spec.batch):
        s = sel_pos_host[r]
        valid = s[s >= 0]
        total += valid.size
        union += np.unique(valid).size
    row = 2 * kv_row_bytes(spec)  # K and V
    return union * row, total * row


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

_CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, device_index=0):
        self.proc = None
        self.t0 = self.t1 = None
        cmd = ["nvidia-smi", f"--query-gpu={_CLOCK_FIELDS}", "--format=csv,noheader,nounits", "-lms", "20"]
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            cmd += ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            pass
        self.cmd = cmd

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.15)
        except Exception:
            self.proc = None

    def mark(self, which):
        if which == "start":
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            return None
        rows = [ln.split(",") for ln in out.strip().splitlines() if ln.count(",") >= 8]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip().lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------

def build_lib():
    import __graft_entry__

    __graft_entry__.build()
    from block_sparse_attention_qsa_gb300 import qsa

    return qsa


def make_gpu_state(qsa, spec):
    g = synth.make_inputs(spec, device="cuda")
    d = qsa.dims_for_spec(spec)
    ws = qsa.make_workspace(d)
    kc = torch.zeros((spec.batch, spec.max_blocks(), spec.n_idx_heads, spec.head_dim), dtype=torch.bfloat16,
                     device="cuda")
    qsa.compress_keys(d, g["idx_keys"], g["q_pos"], kc, ws)
    del g["idx_keys"]
    st = {
        "g": g, "d": d, "ws": ws, "kc": kc,
        "scores": torch.empty((spec.batch, spec.n_q, spec.max_blocks()), device="cuda"),
        "sel_blk": torch.empty((spec.batch, spec.n_q, 512), dtype=torch.int32, device="cuda"),
        "sel_pos": torch.empty((spec.batch, spec.n_q, 2051), dtype=torch.int32, device="cuda"),
        "out": torch.empty((spec.batch, spec.n_q, spec.n_q_heads, spec.head_dim), dtype=torch.bfloat16,
                           device="cuda"),
    }
    return st


def decode_call(qsa, st, inputs=None, out=None):
    g = st["g"] if inputs is None else inputs
    fn = qsa.decode_paged if st.get("paged_kc") else qsa.decode
    fn(st["d"], g["q_idx"], st["kc"], g["q"], st["g"]["k_cache"], st["g"]["v_cache"], st["g"]["k_scale"],
       st["g"]["v_scale"], g["page_table"], g["q_pos"], st["out"] if out is None else out, st["ws"])


class L2Flush:
    """Evicts the step's data from L2 between timed iterations: a write of a
    buffer twice the size of L2, then a read of another one, so the lines the
    write leaves dirty are written back here and not inside the timed region."""

    def __init__(self, l2_bytes):
        n = 2 * l2_bytes // 4 + 1024
        self.w = torch.empty(n, dtype=torch.float32, device="cuda")
        self.r = torch.zeros(n, dtype=torch.float32, device="cuda")
        self.sink = torch.empty((), dtype=torch.float32, device="cuda")

    def __call__(self):
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)


def timed(fn, steps, flush, stream):
    """Per-step device times (ms) of fn, with the L2 flush outside the events."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in evs:
        if flush is not None:
            flush()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def ncu_traffic(kernel_tag):
    """Per-launch DRAM bytes from the committed ncu summary of `kernel_tag`, or
    None if absent or if the kernel source changed since the capture."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m = re.search(r"source_sha256:\s*([0-9a-f]{64})", txt)
    t = re.search(r"dram_bytes_per_launch_full_size:\s*([0-9.eE+]+)", txt)
    src = re.search(r"source_file:\s*(\S+)", txt)
    if not (m and t and src):
        return None
    cur = hashlib.sha256(open(os.path.join(ROOT, src.group(1)), "rb").read()).hexdigest()
    return float(t.group(1)) if cur == m.group(1) else None


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def _bits(t):
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def host_request(spec, src, r, idx_keys=None):
    """The oracle's inputs for request r as numpy (pages renumbered 0..n-1)."""
    npg = spec.pages_per_request()[r]
    pages = src["page_table"][r, :npg].long()
    npi = {
        "q_idx": _bits(src["q_idx"][r:r + 1]),
        "q": _bits(src["q"][r:r + 1]),
        "k_cache": _bits(src["k_cache"][pages]),
        "v_cache": _bits(src["v_cache"][pages]),
        "k_scale": _bits(src["k_scale"]),
        "v_scale": _bits(src["v_scale"]),
        "page_table": np.arange(npg, dtype=np.int32)[None],
        "q_pos": _bits(src["q_pos"][r:r + 1]),
    }
    return npi


def oracle_steps(spec, src, idx_keys_fn, n_steps=None, seconds=None):
    """Time the oracle's decode step one request at a time (inputs copied to
    host and compressed keys prepared outside the timing). Returns (bytes,
    seconds, requests)."""
    from oracle import qsa_oracle as O

    tot_b = 0
    tot_s = 0.0
    done = 0
    r = 0
    while True:
        if n_steps is not None and done >= n_steps:
            break
        if seconds is not None and tot_s >= seconds and done > 0:
            break
        rr = r % spec.batch
        npi = host_request(spec, src, rr)
        npi["kc"] = O.compress_keys(idx_keys_fn(rr), spec.max_blocks())[None]
        t0 = time.perf_counter()
        res = O.decode_step(npi, spec.kv_dtype, rows=[(0, j) for j in range(spec.n_q)])
        tot_s += time.perf_counter() - t0
        nb = (max(spec.q_pos()[rr]) + 1) // 4
        sel = np.stack([res["sel_pos"][(0, j)] for j in range(spec.n_q)])
        valid = sel[sel >= 0]
        tot_b += nb * spec.n_idx_heads * spec.head_dim * 2 + np.unique(valid).size * 2 * kv_row_bytes(spec)
        done += 1
        r += 1
    return tot_b, tot_s, done


def run_draft(qsa, args, spec, st, sel_host, flush, stream, world, rank):
    """MTP draft step reusing the step's selection (no scoring, no top-k):
    per request one draft query at the last verify position, attending over
    the first verify query's selection row plus the 3 positions after it."""
    g = st["g"]
    d = qsa.dims_for_spec(spec)
    d.n_q = 1
    ws = qsa.make_workspace(d)
    qd = g["q"][:, :1].contiguous()
    src = torch.zeros((spec.batch, 1), dtype=torch.int32, device="cuda")
    p_draft = (g["q_pos"][:, :1] + 3).contiguous()
    out = torch.empty((spec.batch, 1, spec.n_q_heads, spec.head_dim), dtype=torch.bfloat16, device="cuda")

    def call():
        qsa.draft_attn(d, qd, g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"], g["page_table"],
                       st["sel_pos"], g["q_pos"], src, p_draft, out, ws)

    call()
    status, info = qsa.check_errors(ws)
    if status != qsa.OK:
        raise RuntimeError(f"device error during the draft step: {info}")
    for _ in range(args.warmup):
        if flush is not None:
            flush()
        call()
    torch.cuda.synchronize()
    barrier(world)
    ms_list = timed(call, args.steps, flush, stream)
    barrier(world)
    ms = max_over_ranks(sum(ms_list) / len(ms_list), world)
    n_pos = sum(int((sel_host[r, 0] >= 0).sum()) + 3 for r in range(spec.batch))
    b = n_pos * kv_row_bytes(spec) * 2  # K and V of each attended position, both KV heads
    if rank == 0:
        print(json.dumps({"metric": "QSA MTP draft-step attention over a reused selection", "workload": spec.name,
                          "latency_us": round(ms * 1e3, 2),
                          "latency_us_p10_p50_p90": [round(float(np.percentile(ms_list, q)) * 1e3, 2)
                                                     for q in (10, 50, 90)],
                          "value": round(b * world / (ms * 1e-3) / 1e9, 1), "unit": UNIT,
                          "bytes_per_step": int(b), "draft_queries_per_request": 1, "gap": 3,
                          "l2": "no flush (warm)" if flush is None else "flushed before every step",
                          "note": "entry-point time: positions resolved to cache rows, then attention"}))


def run_chunk(qsa, args, world, rank):
    """Chunked (prefill) scoring: args.chunk queries of one 50K-token request
    at the chunk's last positions, against all of the request's blocks. The
    block capacity of the buffers (max_blocks) is the request's 12,501 blocks
    rounded up to a multiple of 32, so every score row starts on a 128-byte
    boundary (the capacity is the caller's choice; unaligned rows cost the
    stores partial sectors)."""
    spec = synth.spec_for(1)
    g = synth.make_inputs(spec, device="cuda")
    d0 = qsa.dims_for_spec(spec)
    ws0 = qsa.make_workspace(d0)
    mb = spec.max_blocks()
    kc0 = torch.zeros((1, mb, spec.n_idx_heads, spec.head_dim), dtype=torch.bfloat16, device="cuda")
    qsa.compress_keys(d0, g["idx_keys"], g["q_pos"], kc0, ws0)
    mb_pad = (mb + 31) // 32 * 32
    d = qsa.dims_for_spec(spec)
    d.max_blocks = mb_pad
    ws = qsa.make_workspace(d)
    kc = torch.zeros((1, mb_pad, spec.n_idx_heads, spec.head_dim), dtype=torch.bfloat16, device="cuda")
    kc[:, :mb] = kc0
    del kc0, ws0
    n = args.chunk
    L = spec.first_pos[0]
    qi = synth.normal_bf16((1, n, spec.n_idx_heads, spec.head_dim), spec.seed + 77, device="cuda")
    qp = torch.tensor([[L - (n - 1 - i) for i in range(n)]], dtype=torch.int32, device="cuda")
    sc = torch.empty((1, n, mb_pad), dtype=torch.float32, device="cuda")
    call = lambda: qsa.score_chunk(d, qi, kc, qp, sc, ws)
    call()
    status, info = qsa.check_errors(ws)
    if status != qsa.OK:
        raise RuntimeError(f"device error in chunked scoring: {info}")
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush = None if args.no_flush else L2Flush(l2)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    ms_list = timed(call, args.steps, flush, torch.cuda.current_stream())
    ms = max_over_ranks(sum(ms_list) / len(ms_list), world)
    nf = [(int(p) + 1) // 4 for p in qp[0].tolist()]
    b_out = sum(nf) * 4
    b_kc = max(nf) * spec.n_idx_heads * spec.head_dim * 2
    flops = 2 * sum(nf) * spec.n_idx_heads * spec.head_dim
    if rank == 0:
        print(json.dumps({"metric": "QSA chunked (prefill) scoring", "workload": f"b1-ctx{L}-chunk{n}",
                          "max_blocks": mb_pad, "kernel": "tcgen05 (TMA, TMEM accumulators), persistent",
                          "latency_us": round(ms * 1e3, 2),
                          "latency_us_p10_p50_p90": [round(float(np.percentile(ms_list, q)) * 1e3, 2)
                                                     for q in (10, 50, 90)],
                          "value": round((b_out + b_kc) * world / (ms * 1e-3) / 1e9, 1), "unit": UNIT,
                          "bytes": {"scores_written": b_out, "keys_read_once": b_kc},
                          "tflops": round(flops * world / (ms * 1e-3) / 1e12, 2),
                          "l2": "no flush (warm)" if flush is None else "flushed before every call"}))


def workload_config(spec, args, world):
    """The workload the line measures (the same dict in both arms)."""
    return {"workload": spec.name, "batch": spec.batch, "n_q": spec.n_q,
            "contexts": "50000+800*t, t~U{0..14}" if args.config in (2, 3) else str(spec.first_pos[0]),
            "n_idx_heads": spec.n_idx_heads, "kv": spec.kv_dtype, "page_size": spec.page_size,
            "compressed_keys": "in the KV pages" if args.paged_kc else "contiguous per request",
            "parallelism": f"replicas x{world}"}


def prepare_step(qsa, spec, paged_kc=False):
    """Device state of one workload and one checked step, whose selection
    gives the algorithmic byte count. Returns (state, sel_pos on the host,
    compressed-key bytes, K/V bytes of the union per request, K/V bytes
    summed over queries)."""
    st = make_gpu_state(qsa, spec)
    if paged_kc:
        g = st["g"]
        kcp = torch.zeros((spec.num_pages(), spec.page_size // 4, spec.n_idx_heads, spec.head_dim),
                          dtype=torch.bfloat16, device="cuda")
        idx_keys = synth.normal_bf16((spec.batch, 4 * spec.max_blocks(), spec.n_idx_heads, spec.head_dim),
                                     spec.seed + synth.T_IDXKEYS, device="cuda")
        qsa.compress_keys_paged(st["d"], idx_keys, g["q_pos"], g["page_table"], kcp, st["ws"])
        del idx_keys
        st["kc"], st["paged_kc"] = kcp, True
    g = st["g"]
    (qsa.decode_paged if paged_kc else qsa.decode)(
        st["d"], g["q_idx"], st["kc"], g["q"], g["k_cache"], g["v_cache"], g["k_scale"], g["v_scale"],
        g["page_table"], g["q_pos"], st["out"], st["ws"], scores=st["scores"], sel_blk=st["sel_blk"],
        sel_pos=st["sel_pos"])
    status, info = qsa.check_errors(st["ws"])
    if status != qsa.OK:
        raise RuntimeError(f"device error during the step: {info}")
    sel_host = st["sel_pos"].cpu().numpy()
    b_kv_union, b_kv_sum = kv_bytes(spec, sel_host)
    return st, sel_host, kc_bytes(spec), b_kv_union, b_kv_sum


def step_launcher(qsa, st, graph):
    """The timed step: qsa_decode captured once as a CUDA graph (its three
    kernels and their programmatic dependencies) and replayed, as a serving
    loop would run it, or direct calls."""
    if not graph:
        return lambda: decode_call(qsa, st)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(3):
            decode_call(qsa, st)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        decode_call(qsa, st)
    st["graph"] = g
    return g.replay


def warm(fn, n, flush):
    for _ in range(n):
        if flush is not None:
            flush()
        fn()
    torch.cuda.synchronize()


def sweep(qsa, args, flush, stream, peak, headline):
    """Step latency and algorithmic GB/s over the metric's batches and cache
    types, each entry its own workload (inputs drawn for that batch)."""
    out = []
    for config, batch, ctx in SWEEP:
        if headline is not None and (config, batch, ctx) == headline[0]:
            out.append(dict(headline[1], reused="the headline measurement"))
            continue
        spec = synth.spec_for(config, batch=batch, ctx=ctx)
        st, _, b_kc, b_kv, _ = prepare_step(qsa, spec)
        fn = step_launcher(qsa, st, not args.no_graph)
        warm(fn, max(3, args.warmup), flush)
        ms = timed(fn, args.sweep_steps, flush, stream)
        out.append(sweep_entry(spec, config, ms, b_kc + b_kv, peak))
        del st, fn
        torch.cuda.empty_cache()
    return out


def sweep_entry(spec, config, ms_list, bytes_step, peak):
    ms = sum(ms_list) / len(ms_list)
    gbs = bytes_step / (ms * 1e-3) / 1e9
    return {"workload": spec.name, "config": config, "batch": spec.batch, "kv": spec.kv_dtype,
            "context": "50000+800*t, t~U{0..14}" if config in (2, 3) else spec.first_pos[0],
            "us_mean": round(ms * 1e3, 2), "us_p50": round(float(np.percentile(ms_list, 50)) * 1e3, 2),
            "steps": len(ms_list), "alg_bytes": int(bytes_step), "gbs": round(gbs, 1),
            "frac_of_measured_peak": round(gbs / peak, 4), "frac_of_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4)}


def oracle_all_cores(spec, src, idx_keys_fn, n_saved, seconds, t_req_single):
    """The oracle on every host core: whole requests of the workload (the
    first n_saved of the batch, cycled) run one per process on a spawn-context
    pool, inputs memory-mapped from files written before the timing. Returns
    (bytes, seconds, requests, workers)."""
    import shutil
    import tempfile

    from oracle import parallel as OP
    from oracle import qsa_oracle as O

    workers = OP.host_cores()
    tmp = tempfile.mkdtemp(prefix="qsa_oracle_")
    try:
        n_saved = max(1, min(n_saved, spec.batch))
        for r in range(n_saved):
            npi = host_request(spec, src, r)
            npi["kc"] = O.compress_keys(idx_keys_fn(r), spec.max_blocks())[None]
            OP.save_request(tmp, r, npi)
        pool = OP.OraclePool(workers)
        try:
            pool.timed(tmp, range(min(workers, n_saved)), spec.kv_dtype, kv_row_bytes(spec))  # page the files in
            n = max(workers, int(seconds * workers / max(t_req_single, 1e-3)))
            b, s, done = pool.timed(tmp, [i % n_saved for i in range(n)], spec.kv_dtype, kv_row_bytes(spec))
        finally:
            pool.close()
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
    return b, s, done, workers


def run_ours(args, world, rank):
    qsa = build_lib()
    if args.chunk:
        return run_chunk(qsa, args, world, rank)
    spec = synth.spec_for(args.config, batch=args.batch, ctx=args.ctx, replica=rank)
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush = None if args.no_flush else L2Flush(l2)

    # one checked step: its selection gives the byte count
    st, sel_host, b_kc, b_kv_union, b_kv_sum = prepare_step(qsa, spec, args.paged_kc)
    d = st["d"]
    bytes_step = b_kc + b_kv_union
    if args.draft:
        return run_draft(qsa, args, spec, st, sel_host, flush, stream, world, rank)

    # warm-up, then exactly K timed steps
    step_fn = step_launcher(qsa, st, not args.no_graph)
    warm(step_fn, args.warmup, flush)
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("start")
    step_ms = timed(step_fn, args.steps, flush, stream)
    torch.cuda.synchronize()
    barrier(world)
    if sampler:
        sampler.mark("stop")
    clocks = sampler.stop() if sampler else None
    ms_local = sum(step_ms) / len(step_ms)
    ms = max_over_ranks(ms_local, world)
    value = bytes_step * world / (ms * 1e-3) / 1e9

    if args.step_only:
        if rank == 0:
            print(json.dumps({"workload": spec.name, "latency_us": round(ms * 1e3, 2), "value": round(value, 1),
                              "unit": UNIT, "steps": args.steps, "note": "step-only run"}))
        return

    # per-kernel device times through each kernel's own entry point (same inputs, same flush);
    # the attention kernel alone runs on cache rows resolved once beforehand, as the
    # selector writes them inside the fused step
    g = st["g"]
    reps = max(20, min(args.steps, 200))
    rows = torch.empty_like(st["sel_pos"])
    qsa.resolve(d, st["sel_pos"], g["q_pos"], g["page_table"], rows, st["ws"])
    k_ms = {
        "score": statistics.mean(timed(
            (lambda: qsa.score_paged(d, g["q_idx"], st["kc"], g["page_table"], g["q_pos"], st["scores"], st["ws"]))
            if args.paged_kc else (lambda: qsa.score(d, g["q_idx"], st["kc"], g["q_pos"], st["scores"], st["ws"])),
            reps, flush, stream)),
        "topk": statistics.mean(timed(lambda: qsa.topk(d, st["scores"], g["q_pos"], st["sel_blk"], st["sel_pos"],
                                                       st["ws"]), reps, flush, stream)),
        "attn": statistics.mean(timed(lambda: qsa.sparse_attn_rows(d, g["q"], g["k_cache"], g["v_cache"],
                                                                   g["k_scale"], g["v_scale"], rows, st["out"],
                                                                   st["ws"]), reps, flush, stream)),
    }
    k_bytes = {
        "score": b_kc + sum((p + 1) // 4 for qp in spec.q_pos() for p in qp) * 4,
        "topk": sum((p + 1) // 4 for qp in spec.q_pos() for p in qp) * 4 + spec.batch * spec.n_q * (512 + 2051) * 4,
        "attn": b_kv_union,
    }
    kernels = {k: {"us": round(v * 1e3, 2), "alg_bytes": int(k_bytes[k]),
                   "gbs": round(k_bytes[k] / (v * 1e-3) / 1e9, 1)} for k, v in k_ms.items()}
    dom = max(k_ms, key=lambda k: k_ms[k])
    peak, peak_kind = peaks()
    tags = {"score": "score_kernel_verify_b32_ctx50k", "topk": "topk_kernel_verify_b32_ctx50k",
            "attn": "attn_kernel_verify_b32_ctx50k_bf16"}
    traffic = ncu_traffic(tags[dom]) if args.config == 2 and args.batch in (None, 32) else None
    achieved = k_bytes[dom] / (k_ms[dom] * 1e-3) / 1e9
    roofline = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} hbm_gbs (copy, burst)",
                "traffic": traffic, "alg_bytes_per_launch": int(k_bytes[dom]),
                "step_frac": round(value / world / peak, 4),
                "step_frac_of_nominal_8tbs": round(value / world / NOMINAL_HBM_GBS, 4)}

    # end to end through the public API with host buffers: the step's inputs
    # (index queries, queries, positions, page table) live in one pinned host
    # staging buffer, as an engine would keep them, and go over in one copy;
    # the output comes back in one copy
    per_step = ["q_idx", "q", "q_pos", "page_table"]
    offs, total = {}, 0
    for k in per_step:
        offs[k] = total
        total += (g[k].numel() * g[k].element_size() + 255) // 256 * 256
    host_buf = torch.empty(total, dtype=torch.uint8).pin_memory()
    dev_buf = torch.empty(total, dtype=torch.uint8, device="cuda")

    def view(buf, k):
        nb = g[k].numel() * g[k].element_size()
        return buf[offs[k]:offs[k] + nb].view(g[k].dtype).view(g[k].shape)

    for k in per_step:
        view(host_buf, k).copy_(g[k].cpu())
    dev_in = {k: view(dev_buf, k) for k in per_step}
    out_host = torch.empty(st["out"].shape, dtype=st["out"].dtype).pin_memory()
    h2d = total
    d2h = out_host.numel() * out_host.element_size()

    def e2e_step():
        dev_buf.copy_(host_buf, non_blocking=True)
        decode_call(qsa, st, inputs=dev_in)
        out_host.copy_(st["out"], non_blocking=True)

    # launched like the timed step: the copies and the call captured once as a
    # CUDA graph (copy nodes from and to the pinned host buffers), or direct calls
    e2e_fn = e2e_step
    if not args.no_graph:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(3):
                e2e_step()
        torch.cuda.current_stream().wait_stream(side)
        e2e_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(e2e_graph):
            e2e_step()
        e2e_fn = e2e_graph.replay
    for _ in range(3):
        e2e_fn()
    e2e_ms = statistics.mean(timed(e2e_fn, reps, flush, stream))
    e2e_ms = max_over_ranks(e2e_ms, world)
    e2e = {"value": round(bytes_step * world / (e2e_ms * 1e-3) / 1e9, 1), "unit": UNIT,
           "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
           "launch": "direct calls" if args.no_graph else "copies and step captured once as a CUDA graph, replayed"}

    cpu, cpu1 = None, None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        idx_keys = synth.normal_bf16((spec.batch, 4 * spec.max_blocks(), spec.n_idx_heads, spec.head_dim),
                                     spec.seed + synth.T_IDXKEYS, device="cuda")
        kfn = lambda r: _bits(idx_keys[r])  # noqa: E731
        b1, s1, n1 = oracle_steps(spec, g, kfn, seconds=args.cpu_seconds)
        cpu1 = {"value": round(b1 / s1 / 1e9, 6), "unit": UNIT, "cores": 1, "kind": "oracle",
                "sample": f"{n1} requests of the {spec.batch}-request batch (cycling), all {spec.n_q} queries each, "
                          f"one at a time, numpy FP64, one thread", "seconds": round(s1, 2)}
        bn, sn, nn, workers = oracle_all_cores(spec, g, kfn, args.cpu_requests, args.cpu_seconds, s1 / n1)
        del idx_keys
        cpu = {"value": round(bn / sn / 1e9, 6), "unit": UNIT, "cores": workers, "kind": "oracle",
               "sample": f"{nn} requests (the first {min(args.cpu_requests, spec.batch)} of the "
                         f"{spec.batch}-request batch, cycled), all {spec.n_q} queries each, one request per "
                         f"process on {workers} processes (spawn), numpy FP64",
               "seconds": round(sn, 2), "host_cpu_count": os.cpu_count()}

    sweep_out = None
    if not args.no_sweep and world == 1 and args.config in (2, 3) and not args.paged_kc:
        headline_entry = sweep_entry(spec, args.config, step_ms, bytes_step, peak)
        key = (args.config, spec.batch, None)
        del st, step_fn, rows, host_buf, dev_buf, dev_in, out_host, e2e_fn
        torch.cuda.empty_cache()
        sweep_out = sweep(qsa, args, flush, stream, peak, (key, headline_entry))

    if rank == 0:
        res = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 5), "latency_us": round(ms * 1e3, 2),
            "latency_us_p10_p50_p90": [round(float(np.percentile(step_ms, q)) * 1e3, 2) for q in (10, 50, 90)],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp8" if spec.kv_dtype == "fp8" else "bf16", "data": "synthetic",
            "config": workload_config(spec, args, world),
            "protocol": {"l2": "no flush (warm)" if flush is None else "flushed before every step (a write of 2x L2, then a read of 2x L2)",
                         "launch": "direct calls" if args.no_graph else "the step captured once as a CUDA graph, replayed"},
            "bytes_per_step": {"kc": int(b_kc), "kv_union": int(b_kv_union), "kv_sum": int(b_kv_sum)},
            "kernels": kernels, "roofline": roofline, "e2e": e2e, "cpu_baseline": cpu,
            "cpu_baseline_single_core": cpu1, "sweep": sweep_out,
            "gpu_launches": 3 * args.steps, "clocks": clocks,
        }
        print(json.dumps(res))


def run_reference(args, world, rank):
    """The oracle as it stands, timed on the host's cores: each step runs as
    many whole requests of the workload as there are cores, one per process."""
    if rank != 0:
        return
    import shutil
    import tempfile

    from oracle import parallel as OP
    from oracle import qsa_oracle as O

    spec = synth.spec_for(args.config, batch=args.batch, ctx=args.ctx)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    g = synth.make_inputs(spec, device=dev, with_index_keys=False)
    idx_keys = synth.normal_bf16((spec.batch, 4 * spec.max_blocks(), spec.n_idx_heads, spec.head_dim),
                                 spec.seed + synth.T_IDXKEYS, device=dev)
    workers = OP.host_cores()
    per_step = workers  # one whole request per process each step, cycling over the batch
    n_saved = max(1, min(spec.batch, args.cpu_requests))
    tmp = tempfile.mkdtemp(prefix="qsa_oracle_")
    try:
        for r in range(n_saved):
            npi = host_request(spec, g, r)
            npi["kc"] = O.compress_keys(_bits(idx_keys[r]), spec.max_blocks())[None]
            OP.save_request(tmp, r, npi)
        del idx_keys, g
        pool = OP.OraclePool(workers)
        try:
            nxt = 0
            for _ in range(args.warmup):
                pool.timed(tmp, [(nxt + i) % n_saved for i in range(per_step)], spec.kv_dtype, kv_row_bytes(spec))
                nxt += per_step
            b = s = n = 0
            for _ in range(args.steps):
                bb, ss, nn = pool.timed(tmp, [(nxt + i) % n_saved for i in range(per_step)], spec.kv_dtype,
                                        kv_row_bytes(spec))
                nxt += per_step
                b, s, n = b + bb, s + ss, n + nn
        finally:
            pool.close()
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
    value = b / s / 1e9
    res = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(s / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": workload_config(spec, args, world),
        "protocol": {"step": f"{per_step} whole requests of the batch (cycling over its first {n_saved}), "
                             f"one per process"},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": workers, "kind": "oracle",
                         "sample": f"{n} requests of {spec.name}, {per_step} per step on {workers} processes "
                                   f"(spawn), numpy FP64"},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(res))


def main():
    args = parse_args()
    world, rank, _ = dist_init()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
