"""bench.py's N > 1 host logic on CPU: two gloo ranks on 127.0.0.1.

Each rank reports the slowest rank's step time, and the whole-job value
counts every rank's tokens over that time (replicas, weak scaling). The
reference arm runs on rank 0 alone and the other ranks exit without output."""
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


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    step_s = bench.max_over_ranks(0.001 * (1 + rank), world, torch.device("cpu"))
    value = bench.job_throughput(world, 8, step_s)
    dist.barrier()
    q.put((rank, step_s, value))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step_and_count_every_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1]
    for _, step_s, value in got:
        assert step_s == pytest.approx(0.002)          # the slower rank
        assert value == pytest.approx(2 * 8 / 0.002)   # both ranks' tokens


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_prints_on_rank0_only(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr[-500:]
    if rank == 0:
        import json
        line = json.loads(r.stdout.strip().splitlines()[-1])
        assert line["impl"] == "reference" and line["n_gpus"] == 2
    else:
        assert r.stdout.strip() == ""
