"""The benchmark's multi-rank plumbing on CPU (gloo, world size 2): replicas
draw independent batches, ranks meet at barriers, and the reported time is
the slowest rank's while the work is summed.  Also the reference arm (the
oracle on the host cores) and its one-line JSON contract."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    from paged_kv_cache_230_gb300 import workloads as W
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(dist)
    mx = bench.max_over_ranks(dist, 1.5 + rank)
    sm = bench.sum_over_ranks(dist, 10.0 * (rank + 1))
    lens = W.config_lengths(2, 2 + 1000 * rank)
    out.put((rank, mx, sm, lens.tolist()))
    bench.barrier(dist)
    dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_bench():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.5, 2.5]      # time = slowest rank
    assert [r[2] for r in res] == [30.0, 30.0]    # work = sum over ranks
    assert res[0][3] != res[1][3]                  # replicas draw different batches


def _json_lines(text):
    return [json.loads(l) for l in text.splitlines() if l.strip().startswith("{")]


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "0",
                        "--steps", "2", "--warmup", "1", "--ref-budget", "0.2"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["config"]["workload"] == "tiny" and d["steps"] == 2


def test_reference_arm_under_torchrun_prints_from_rank0_only():
    port = _free_port()
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                        "--gpus", "2", "--impl", "reference", "--config", "0", "--steps", "1", "--warmup", "0",
                        "--ref-budget", "0.2"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2
