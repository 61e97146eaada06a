"""The bench's multi-process path on CPU (gloo, world size 2).

The verify path shards into independent replicas (one per GPU, no exchange),
so the only cross-rank steps are the bench's own: the rendezvous, the barrier
around the timed region, the maximum of the ranks' times and rank 0 alone
printing.  These run here with the gloo backend on 127.0.0.1.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), LBX_BENCH_GLOO="1")
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    r, w, local = bench.dist_setup(world)
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    # each rank's "time": the slowest must win on every rank
    got = bench.max_over_ranks(10.0 + 5.0 * rank, w, "cpu")
    out.put((rank, got))
    bench.barrier(w)
    dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = dict(q.get(timeout=10) for _ in range(world))
    assert res == {0: 15.0, 1: 15.0}


def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` under torchrun (2 ranks, gloo): rank 0 times
    the oracle and prints one JSON line, the other rank exits 0 silently."""
    port = free_port()
    env = dict(os.environ, LBX_BENCH_GLOO="1", OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--workload", "tiny"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["n_gpus"] == 2 and j["value"] > 0
    assert j["cpu_baseline"]["kind"] == "oracle"
