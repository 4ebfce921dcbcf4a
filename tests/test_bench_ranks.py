"""Multi-rank host logic of bench.py on the CPU (gloo, world size 2).

The decode shards with no exchange: every rank runs its own input replicas on its own
GPU, the ranks meet at barriers around the timed region and the step time is the maximum
over ranks. These checks run that plumbing with two CPU processes: the rendezvous, the
barrier, the max-over-ranks reduction, disjoint replica seeds per rank, and a torchrun
launch of the reference arm in which only rank 0 prints.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench

    ws, r, local = bench.dist_info()
    bench.init_dist(ws, "gloo")
    bench.barrier(ws)
    worst = bench.max_over_ranks(10.0 + 5.0 * r, ws, "cpu")
    seeds = bench.shard_replicas(4, ws, r)
    bench.barrier(ws)
    torch.distributed.destroy_process_group()
    q.put((r, ws, local, worst, seeds))


def test_two_rank_barrier_max_and_sharding():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == 2 for g in got)
    assert all(g[3] == 15.0 for g in got)            # the slower rank's time on every rank
    s0, s1 = set(got[0][4]), set(got[1][4])
    assert len(s0) == len(s1) == 4 and not (s0 & s1)  # same per-rank count, own inputs


def test_torchrun_reference_arm_prints_on_rank0_only():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--workload", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    res = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["cpu_baseline"]["kind"] == "oracle"
    assert line["higher_is_better"] is False and line["value"] > 0
