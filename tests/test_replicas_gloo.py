"""The N > 1 host path of bench.py: independent replicas (no collective on the
data path), the job's time taken from the slowest rank, throughput summed
over ranks.  Two gloo ranks on CPU; no GPU.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sys.path.insert(0, ROOT)
        import bench
        ms = bench.slowest_rank(10.0 + 5.0 * rank, world)          # rank 1 is the slow one
        alone = bench.slowest_rank(3.0, 1)
        q.put((rank, ms, bench.job_rate(world, 100, ms), alone, bench.replica_seed(1, rank)))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1]
    for rank, ms, rate, alone, seed in got:
        assert ms == 15.0                      # both ranks report the slowest rank's time
        assert rate == pytest.approx(2 * 100 / 0.015)
        assert alone == 3.0
    assert got[0][4] != got[1][4]              # each replica draws its own inputs


def test_reference_arm_runs_on_rank_zero_only():
    # under torchrun the other ranks of the reference arm exit 0 without work or output
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    for wl in ("decode_70b", "snapkv"):
        r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", wl,
                            "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True, timeout=120)
        assert r.returncode == 0, r.stderr
        assert r.stdout.strip() == ""
