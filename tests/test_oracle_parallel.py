"""The all-core oracle runner (oracle/parallel.py) against plain oracle calls.

bench.py times the oracle on every host core by running whole requests in a
spawn-context process pool that reads each request's inputs from memory-mapped
files. These tests check, on the CPU, that the pool computes what the oracle
computes in process: the same selections, so the same algorithmic bytes, and
that its byte count agrees with bench.py's own accounting of a step.
"""

import numpy as np

import bench
from block_sparse_attention_qsa_gb300 import synth
from oracle import parallel as OP
from oracle import qsa_oracle as O
from tests._util import small_spec


def _request_inputs(spec, inp, r):
    npi = bench.host_request(spec, inp, r)
    npi["kc"] = O.compress_keys(bench._bits(inp["idx_keys"][r]), spec.max_blocks())[None]
    return npi


def test_pool_runs_the_oracle_like_a_plain_call(tmp_path):
    spec = small_spec([2300, 800, 1500], n_q=3, seed=17)
    inp = synth.make_inputs(spec)
    reqs = [_request_inputs(spec, inp, r) for r in range(spec.batch)]
    for r, npi in enumerate(reqs):
        OP.save_request(str(tmp_path), r, npi)
    order = [0, 2, 1, 0]
    pool = OP.OraclePool(2)
    try:
        b, s, n = pool.timed(str(tmp_path), order, spec.kv_dtype, bench.kv_row_bytes(spec))
    finally:
        pool.close()
    assert n == len(order) and s > 0
    want = 0
    for r in order:
        res = O.decode_step(reqs[r], spec.kv_dtype, rows=[(0, j) for j in range(spec.n_q)])
        want += OP.request_bytes(reqs[r], [res["sel_pos"][(0, j)] for j in range(spec.n_q)],
                                 bench.kv_row_bytes(spec))
    assert b == want


def test_request_bytes_agree_with_the_bench_accounting():
    spec = small_spec([3100, 2900], n_q=4, seed=18)
    inp = synth.make_inputs(spec)
    sel = np.zeros((spec.batch, spec.n_q, O.WIDTH), np.int32)
    total = 0
    for r in range(spec.batch):
        npi = _request_inputs(spec, inp, r)
        res = O.decode_step(npi, spec.kv_dtype, rows=[(0, j) for j in range(spec.n_q)])
        rows = [res["sel_pos"][(0, j)] for j in range(spec.n_q)]
        sel[r] = np.stack(rows)
        total += OP.request_bytes(npi, rows, bench.kv_row_bytes(spec))
    union, _ = bench.kv_bytes(spec, sel)
    assert total == bench.kc_bytes(spec) + union


def test_host_cores_is_positive():
    assert OP.host_cores() >= 1
