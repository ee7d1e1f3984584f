"""Multi-process paths on CPU (gloo, world size 2): the replica plumbing of
bench.py (each rank runs its own shard of the batch; barrier and the max of
the ranks' times) and the reference arm under torchrun. No GPU involved."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

from block_sparse_attention_qsa_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "WORLD_SIZE": str(world),
                       "RANK": str(rank), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist

    w, r, _ = bench.dist_init()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    m = bench.max_over_ranks(float(10 * (rank + 1)), w)  # each rank's "time"
    spec = synth.spec_for(2, batch=4, replica=rank)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max": m, "first_pos": spec.first_pos, "seed": spec.seed}, f)
    dist.destroy_process_group()


def test_replica_plumbing_two_ranks(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_worker, args=(world, port, str(tmp_path)), nprocs=world, start_method="spawn")
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    assert all(x["max"] == 20.0 for x in res)  # the slowest rank's time, on every rank
    assert res[0]["seed"] != res[1]["seed"]  # each replica draws its own shard of requests
    assert len(res[0]["first_pos"]) == len(res[1]["first_pos"]) == 4


def test_replica_shards_have_the_workload_shape():
    a, b = synth.spec_for(2, replica=0), synth.spec_for(2, replica=1)
    assert (a.batch, a.n_q, a.n_idx_heads, a.kv_dtype) == (b.batch, b.n_q, b.n_idx_heads, b.kv_dtype)
    for spec in (a, b):  # contexts 50,000 + 800 t, t in 0..14
        assert all((p - 50_000) % 800 == 0 and 0 <= (p - 50_000) // 800 <= 14 for p in spec.first_pos)
    assert synth.spec_for(2).seed == a.seed  # replica 0 is the single-GPU workload


@pytest.mark.timeout(600)
def test_reference_arm_under_torchrun_two_ranks():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--config", "0", "--steps", "1", "--warmup", "1"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1  # rank 0 alone prints
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
