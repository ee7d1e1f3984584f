"""The oracle's decode step on several host cores.

TEST AND BENCHMARK INFRASTRUCTURE ONLY, like ``qsa_oracle``: nothing in the
library path imports it. ``bench.py`` uses it to time the oracle on all of the
host's cores; it changes nothing in what the oracle computes, it only runs
whole requests of a batch in separate processes.

Each request's inputs are written once as ``.npy`` files and memory-mapped by
the workers, so the processes share one copy through the page cache and no
array is pickled per task. The pool uses the ``spawn`` start method: a process
forked from a parent that has touched the GPU can hang.
"""

from __future__ import annotations

import multiprocessing as mp
import os
import time
from concurrent.futures import ProcessPoolExecutor
from typing import Dict, Iterable, Tuple

import numpy as np

from oracle import qsa_oracle as O

KEYS = ("q_idx", "kc", "q", "k_cache", "v_cache", "k_scale", "v_scale", "page_table", "q_pos")


def host_cores() -> int:
    """Cores this process may run on (its affinity mask), else the CPU count."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def save_request(dirpath: str, r: int, npi: Dict[str, np.ndarray]) -> None:
    """Writes request r's oracle inputs (one request, pages renumbered)."""
    for k in KEYS:
        np.save(os.path.join(dirpath, f"r{r}_{k}.npy"), np.ascontiguousarray(npi[k]))


def load_request(dirpath: str, r: int) -> Dict[str, np.ndarray]:
    # plain ndarray views of the mapped files: indexing a np.memmap builds a
    # new memmap object per lookup, which the oracle's per-row gathers would pay
    return {k: np.asarray(np.load(os.path.join(dirpath, f"r{r}_{k}.npy"), mmap_mode="r")) for k in KEYS}


def request_bytes(npi: Dict[str, np.ndarray], sel_rows: Iterable[np.ndarray], kv_row_bytes: int) -> int:
    """Algorithmic bytes of one request's step: its compressed keys read once
    (the full blocks of its last query) plus K and V of the union of its
    queries' selected positions."""
    kc = npi["kc"]
    nb = max(1, O.n_full(int(np.max(npi["q_pos"]))))
    kc_b = nb * kc.shape[2] * kc.shape[3] * 2
    sel = np.concatenate([np.asarray(s) for s in sel_rows])
    return kc_b + np.unique(sel[sel >= 0]).size * 2 * kv_row_bytes


def run_request(dirpath: str, r: int, kv_dtype: str, kv_row_bytes: int) -> int:
    """The oracle's whole step for every query of saved request r; returns
    its algorithmic bytes."""
    npi = load_request(dirpath, r)
    nq = npi["q_pos"].shape[1]
    res = O.decode_step(npi, kv_dtype, rows=[(0, j) for j in range(nq)])
    return request_bytes(npi, [res["sel_pos"][(0, j)] for j in range(nq)], kv_row_bytes)


def _ready(_=None) -> int:
    return os.getpid()


class OraclePool:
    """A spawn-context process pool whose workers are started (and have
    imported numpy and the oracle) before any timing."""

    def __init__(self, workers: int):
        self.workers = workers
        self.ex = ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn"))
        list(self.ex.map(_ready, range(4 * workers)))

    def timed(self, dirpath: str, requests: Iterable[int], kv_dtype: str, kv_row_bytes: int) -> Tuple[int, float, int]:
        """Runs the saved requests (one task each, any order) across the
        workers; returns (bytes, wall seconds, requests done)."""
        reqs = list(requests)
        t0 = time.perf_counter()
        futs = [self.ex.submit(run_request, dirpath, r, kv_dtype, kv_row_bytes) for r in reqs]
        total = sum(f.result() for f in futs)
        return total, time.perf_counter() - t0, len(reqs)

    def close(self):
        self.ex.shutdown(wait=True)
