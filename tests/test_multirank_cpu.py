"""The benchmark's multi-rank logic on CPU ranks (gloo, world size 2): every
rank scans its own problem (no collective on the data path); timing is the
maximum over ranks and throughput counts the units of all ranks."""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    import workloads as W
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cpu = torch.device("cpu")
        secs = 1.0 + rank  # rank 1 is the slow one
        mx = bench.max_over_ranks(secs, world, cpu)
        bench.barrier(world)
        shape = W.ScanShape("t", 1, 4, 4, 16, torch.float32)
        u = W.scan_inputs(shape, seed=bench.rank_seed(rank))["u"]
        gathered = [torch.empty_like(u) for _ in range(world)]
        dist.all_gather(gathered, u)  # test-only check that ranks hold different problems
        q.put((rank, mx, bool(torch.equal(gathered[0], gathered[1]))))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, same in res:
        assert mx == 2.0          # max over ranks
        assert not same           # each rank has its own problem


def test_aggregate_throughput():
    import bench
    assert bench.aggregate_throughput(1000, 4, 10, 2.0) == 4 * 1000 * 10 / 2.0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
